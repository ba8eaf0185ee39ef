// Warp-level tf32 tensor-core helpers for the chunk kernels that run on
// mma.sync (16 x 8 x 8, fp32 accumulate) out of shared-memory tiles: operand
// accessors, float32 tile layouts whose 16-byte row groups are XOR-permuted by
// row (conflict-free fragment reads by rows and by columns), and 16-byte
// asynchronous tile copies.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "la_wy.cuh"

namespace la {
namespace wm {

using wy::mma_16x8x8_tf32;
using wy::to_tf32;
using sm100::smem_u32;

constexpr int kCh = 64;        // chunk length
constexpr int kCW = 16;        // value columns per block
// float32 tiles are dense (64 or 16 floats a row) with the 16-byte groups of a
// row permuted by an XOR of the row index, so that the tf32 fragment reads of
// the warp MMAs -- by rows or by columns, as A or as B -- hit 32 distinct banks.
constexpr int kPf = kCh;       // floats per row of C x C tiles
constexpr int kPw = kCW;       // floats per row of x 16 tiles
__host__ __device__ __forceinline__ int swz64(int r) { return ((r & 3) << 3) | (((r >> 2) & 1) << 2); }
__host__ __device__ __forceinline__ int swz16(int r) { return (((r >> 1) & 1) << 3) | (((r >> 2) & 1) << 2); }
__device__ __forceinline__ float &cc(float *p, int r, int c) { return p[r * kPf + (c ^ swz64(r))]; }
__device__ __forceinline__ float &w16(float *p, int r, int c) { return p[r * kPw + (c ^ swz16(r))]; }
template <int DK>
struct Pitch {
  static constexpr int h = DK + 8;  // row pitch (bf16) of q / k tiles: 16-byte rows
};

__device__ __forceinline__ uint32_t bfbits(const __nv_bfloat16 *p) {
  return static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(p)) << 16;
}
__device__ __forceinline__ uint32_t tf(float x) { return to_tf32(x); }

// acc[j] (the 16 x 8 tile at rows m0.., columns n0 + 8 j) += A[m0.., 0..K) B[0..K), ..]:
// ga(m, k) and gb(k, n) return the tf32 bits of one element.
// With one or two tiles the k steps alternate between two accumulator sets, so
// consecutive MMAs do not wait on each other's results.
template <int NT, class GA, class GB>
__device__ __forceinline__ void wmma(float (&acc)[NT][4], int m0, int n0, int K, GA ga, GB gb, int lane) {
  const int g = lane >> 2, t = lane & 3;
  constexpr bool split = NT <= 2;
  float alt[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) alt[j][0] = alt[j][1] = alt[j][2] = alt[j][3] = 0.f;
#pragma unroll
  for (int k0 = 0; k0 < K; k0 += 8) {
    uint32_t a[4] = {ga(m0 + g, k0 + t), ga(m0 + g + 8, k0 + t), ga(m0 + g, k0 + t + 4),
                     ga(m0 + g + 8, k0 + t + 4)};
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      uint32_t b[2] = {gb(k0 + t, n0 + 8 * j + g), gb(k0 + t + 4, n0 + 8 * j + g)};
      mma_16x8x8_tf32(split && (k0 & 8) ? alt[j] : acc[j], a, b);
    }
  }
  if (split) {
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      acc[j][0] += alt[j][0];
      acc[j][1] += alt[j][1];
      acc[j][2] += alt[j][2];
      acc[j][3] += alt[j][3];
    }
  }
}
// wmma with the k loop kept rolled (four steps per iteration): for kernels whose
// fully unrolled body would not stay in the instruction cache
template <int NT, class GA, class GB>
__device__ __forceinline__ void wmma_r(float (&acc)[NT][4], int m0, int n0, int K, GA ga, GB gb, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll 4
  for (int k0 = 0; k0 < K; k0 += 8) {
    uint32_t a[4] = {ga(m0 + g, k0 + t), ga(m0 + g + 8, k0 + t), ga(m0 + g, k0 + t + 4),
                     ga(m0 + g + 8, k0 + t + 4)};
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      uint32_t b[2] = {gb(k0 + t, n0 + 8 * j + g), gb(k0 + t + 4, n0 + 8 * j + g)};
      mma_16x8x8_tf32(acc[j], a, b);
    }
  }
}
// ---- bf16 operands: mma.sync m16n8k16 (fp32 accumulate). A is row-major with k
// contiguous (element (m, k) at pa[m * lda + k]); B is given by columns with k
// contiguous (element (k, n) at pb[n * ldb + k]); both row pitches in bf16 units,
// even, with (pitch / 2) % 32 == 4 or 12 or 20 or 28 for conflict-free fragment reads.
__device__ __forceinline__ void mma_16x8x16_bf16(float *d, const uint32_t *a, const uint32_t *b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
__device__ __forceinline__ uint32_t ld32(const __nv_bfloat16 *p) { return *reinterpret_cast<const uint32_t *>(p); }
// acc[j] (16 x 8 tiles at rows m0.., columns n0 + 8 j) += A B over k in [0, K), K % 16 == 0;
// neg flips the sign of A
template <int NT, bool NEG = false>
__device__ __forceinline__ void wmma16(float (&acc)[NT][4], int m0, int n0, int K, const __nv_bfloat16 *pa,
                                       int lda, const __nv_bfloat16 *pb, int ldb, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const __nv_bfloat16 *a0 = pa + (m0 + g) * lda + 2 * t, *a1 = a0 + 8 * lda;
#pragma unroll
  for (int k0 = 0; k0 < K; k0 += 16) {
    uint32_t a[4] = {ld32(a0 + k0), ld32(a1 + k0), ld32(a0 + k0 + 8), ld32(a1 + k0 + 8)};
    if (NEG) {
#pragma unroll
      for (int e = 0; e < 4; ++e) a[e] ^= 0x80008000u;
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const __nv_bfloat16 *b0 = pb + (n0 + 8 * j + g) * ldb + k0 + 2 * t;
      uint32_t b[2] = {ld32(b0), ld32(b0 + 8)};
      mma_16x8x16_bf16(acc[j], a, b);
    }
  }
}
// The same with B given row-major (element (k, n) at pb[k * ldb + n], 16-byte rows):
// each B fragment comes from one ldmatrix.trans of two 8 x 8 blocks.
template <int NT>
__device__ __forceinline__ void wmma16_bt(float (&acc)[NT][4], int m0, int n0, int K, const __nv_bfloat16 *pa,
                                          int lda, const __nv_bfloat16 *pb, int ldb, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const __nv_bfloat16 *a0 = pa + (m0 + g) * lda + 2 * t, *a1 = a0 + 8 * lda;
  const int lr = (lane & 7) + 8 * ((lane >> 3) & 1);  // the row lanes 0..15 address
#pragma unroll
  for (int k0 = 0; k0 < K; k0 += 16) {
    uint32_t a[4] = {ld32(a0 + k0), ld32(a1 + k0), ld32(a0 + k0 + 8), ld32(a1 + k0 + 8)};
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      uint32_t b[2];
      asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                   : "=r"(b[0]), "=r"(b[1])
                   : "r"(smem_u32(pb + (k0 + lr) * ldb + n0 + 8 * j)));
      mma_16x8x16_bf16(acc[j], a, b);
    }
  }
}
// The same with A given transposed (element (m, k) at pa[k * lda + m], 16-byte rows):
// each A fragment comes from one ldmatrix.trans of four 8 x 8 blocks.
template <int NT, bool NEG = false>
__device__ __forceinline__ void wmma16_at(float (&acc)[NT][4], int m0, int n0, int K, const __nv_bfloat16 *pa,
                                          int lda, const __nv_bfloat16 *pb, int ldb, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const int blk = lane >> 3, lr = lane & 7;  // lanes 8i .. 8i + 7 address block i's rows
  const __nv_bfloat16 *arow = pa + (lr + 8 * (blk >> 1)) * lda + m0 + 8 * (blk & 1);
#pragma unroll
  for (int k0 = 0; k0 < K; k0 += 16) {
    uint32_t a[4];
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                 : "r"(smem_u32(arow + k0 * lda)));
    if (NEG) {
#pragma unroll
      for (int e = 0; e < 4; ++e) a[e] ^= 0x80008000u;
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const __nv_bfloat16 *b0 = pb + (n0 + 8 * j + g) * ldb + k0 + 2 * t;
      uint32_t b[2] = {ld32(b0), ld32(b0 + 8)};
      mma_16x8x16_bf16(acc[j], a, b);
    }
  }
}
// The same with both operands through ldmatrix.trans: A given transposed (element
// (m, k) at pa[k * lda + m]) and B given row-major (element (k, n) at pb[k * ldb + n]).
template <int NT>
__device__ __forceinline__ void wmma16_atbt(float (&acc)[NT][4], int m0, int n0, int K, const __nv_bfloat16 *pa,
                                            int lda, const __nv_bfloat16 *pb, int ldb, int lane) {
  const int blk = lane >> 3, lr = lane & 7;
  const __nv_bfloat16 *arow = pa + (lr + 8 * (blk >> 1)) * lda + m0 + 8 * (blk & 1);
  const int br = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
  for (int k0 = 0; k0 < K; k0 += 16) {
    uint32_t a[4];
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                 : "r"(smem_u32(arow + k0 * lda)));
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      uint32_t b[2];
      asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                   : "=r"(b[0]), "=r"(b[1])
                   : "r"(smem_u32(pb + (k0 + br) * ldb + n0 + 8 * j)));
      mma_16x8x16_bf16(acc[j], a, b);
    }
  }
}
// a float as the high half of a bf16 pair etc.
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// f(row, col, value) over the elements of an accumulator set (values may be changed)
template <int NT, class F>
__device__ __forceinline__ void each(float (&acc)[NT][4], int m0, int n0, int lane, F f) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    f(m0 + g, n0 + 8 * j + 2 * t, acc[j][0]);
    f(m0 + g, n0 + 8 * j + 2 * t + 1, acc[j][1]);
    f(m0 + g + 8, n0 + 8 * j + 2 * t, acc[j][2]);
    f(m0 + g + 8, n0 + 8 * j + 2 * t + 1, acc[j][3]);
  }
}
template <int NT>
__device__ __forceinline__ void zero(float (&acc)[NT][4]) {
#pragma unroll
  for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
}
// element (r, c) of a float32 tile whose rows are W floats long (W a multiple of 32)
template <int W>
__device__ __forceinline__ float &fw(float *p, int r, int c) { return p[r * W + (c ^ swz64(r))]; }

// ---- asynchronous tile copies (16 bytes each; a copy of 0 source bytes fills zeros)
constexpr int kPh = kCW + 8;  // row pitch (bf16) of x 16 bf16 tiles: 48-byte rows

__device__ __forceinline__ void cpa16(void *dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16u : 0u)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// rows [0, 64) of a [T][D] bf16 tensor from the chunk's first token (n valid, zero beyond), pitch P
template <int D, int P>
__device__ __forceinline__ void rows_async(__nv_bfloat16 *dst, const __nv_bfloat16 *src, int n, int tid, int nthr) {
  for (int i = tid; i < kCh * (D / 8); i += nthr) {
    const int r = i / (D / 8), c = (i % (D / 8)) * 8;
    const bool ok = r < n;
    cpa16(dst + r * P + c, src + (ok ? (size_t)r * D + c : 0), ok);
  }
}
// the 64 x 16 columns [c0, c0 + 16) of a [T][D] bf16 tensor, pitch kPh
template <int D>
__device__ __forceinline__ void cols_async(__nv_bfloat16 *dst, const __nv_bfloat16 *src, int c0, int n, int tid,
                                           int nthr) {
  for (int i = tid; i < kCh * 2; i += nthr) {
    const int r = i >> 1, c = (i & 1) * 8;
    const bool ok = r < n;
    cpa16(dst + r * kPh + c, src + (ok ? (size_t)r * D + c0 + c : 0), ok);
  }
}
// a 64 x 64 float32 matrix (row-major, contiguous), pitch kPf
__device__ __forceinline__ void cc_async(float *dst, const float *src, int tid, int nthr) {
  for (int i = tid; i < kCh * kCh / 4; i += nthr) {
    const int r = i >> 4, c = (i & 15) * 4;
    cpa16(dst + r * kPf + (c ^ swz64(r)), src + 4 * i, true);
  }
}
// the D x 16 columns [c0, c0 + 16) of a [D][DV] float32 matrix, pitch kPw
template <int D, int DV>
__device__ __forceinline__ void state_async(float *dst, const float *src, int c0, int tid, int nthr) {
  for (int i = tid; i < D * 4; i += nthr) {
    const int r = i >> 2, c = (i & 3) * 4;
    cpa16(dst + r * kPw + (c ^ swz16(r)), src + (size_t)r * DV + c0 + c, true);
  }
}
// a 64 x DK float32 matrix (row-major, contiguous) into the permuted layout fw<DK>
template <int DK>
__device__ __forceinline__ void wide_async(float *dst, const float *src, int tid, int nthr) {
  for (int i = tid; i < kCh * DK / 4; i += nthr) {
    const int r = i / (DK / 4), c = (i % (DK / 4)) * 4;
    cpa16(dst + r * DK + (c ^ swz64(r)), src + 4 * i, true);
  }
}
__device__ __forceinline__ float bf(const __nv_bfloat16 *p) { return __uint_as_float(bfbits(p)); }

}  // namespace wm
}  // namespace la
