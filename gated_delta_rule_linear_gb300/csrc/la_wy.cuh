// Helpers of the delta rule's triangular solve T = (I + A)^-1 on 16x16 blocks
// (shared by the delta-rule kernels): tf32 rounding and warp-level tf32 MMAs
// on blocks held in shared memory with row pitch kAp.
#pragma once

#include "la_tc_common.cuh"

namespace la {
namespace wy {

constexpr int kAp = tc::kC + 4;  // pitch of A and T: 16-byte rows, conflict-free A fragments

// Round to the nearest tf32 value, ties away from zero (finite inputs): add
// half of the 13 dropped mantissa bits, then clear them; a mantissa carry
// moves into the exponent as it should. Two integer operations.
__device__ __forceinline__ uint32_t to_tf32(float x) { return (__float_as_uint(x) + 0x1000u) & 0xffffe000u; }
__device__ __forceinline__ float round_tf32(float x) { return __uint_as_float(to_tf32(x)); }
// Warp-level 16x8x8 tf32 MMA (register fragments), fp32 accumulate.
__device__ __forceinline__ void mma_16x8x8_tf32(float *d, const uint32_t *a, const uint32_t *b) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// acc (16x16, two 16x8 fragments) += Ab (16x16) * Bb (16x16): blocks of pitch
// kAp in shared memory holding values already rounded to tf32; one warp.
__device__ __forceinline__ void block_mma_16(float (&acc)[2][4], const float *Ab, const float *Bb, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    uint32_t a[4];
    a[0] = __float_as_uint(Ab[g * kAp + 8 * ks + t]);
    a[1] = __float_as_uint(Ab[(g + 8) * kAp + 8 * ks + t]);
    a[2] = __float_as_uint(Ab[g * kAp + 8 * ks + t + 4]);
    a[3] = __float_as_uint(Ab[(g + 8) * kAp + 8 * ks + t + 4]);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      uint32_t b[2];
      b[0] = __float_as_uint(Bb[(8 * ks + t) * kAp + 8 * nt + g]);
      b[1] = __float_as_uint(Bb[(8 * ks + t + 4) * kAp + 8 * nt + g]);
      mma_16x8x8_tf32(acc[nt], a, b);
    }
  }
}
// Column jc of the inverse of the unit lower-triangular 16x16 block I + A_bb
// (blk = b, strictly lower part of A in shared memory with pitch kAp, zeros
// elsewhere) by forward substitution in column (saxpy) order: once x_m is
// final it updates every later row at once, so the dependent chain is 16
// FMAs long instead of 120, and A is read as 16-byte row pieces. The FMAs
// per row run in the same order as in the row-by-row form (rows before jc
// contribute exact zeros). Writes the column, rounded to tf32, into T.
__device__ __forceinline__ void diag_inverse_16(const float *Af, float *Tf, int blk, int jc) {
  const int base = blk * 16;
  float acc[16];
#pragma unroll
  for (int r = 0; r < 16; ++r) acc[r] = (r == jc) ? 1.f : 0.f;
#pragma unroll
  for (int g4 = 0; g4 < 4; ++g4) {
    float4 a4[16];
#pragma unroll
    for (int r = 4 * g4 + 1; r < 16; ++r)
      a4[r] = *reinterpret_cast<const float4 *>(Af + (base + r) * kAp + base + 4 * g4);
#pragma unroll
    for (int mm = 0; mm < 4; ++mm) {
      const int m = 4 * g4 + mm;
      const float xm = acc[m];  // final: rows above m are done
#pragma unroll
      for (int r = m + 1; r < 16; ++r) {
        const float am = mm == 0 ? a4[r].x : mm == 1 ? a4[r].y : mm == 2 ? a4[r].z : a4[r].w;
        acc[r] = fmaf(-am, xm, acc[r]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 16; ++r) Tf[(base + r) * kAp + base + jc] = round_tf32(acc[r]);
}
// Store a 16x16 accumulator (scaled by sgn, rounded to tf32) into a block of pitch kAp.
__device__ __forceinline__ void block_store_16(float *Cb, const float (&acc)[2][4], float sgn, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    *reinterpret_cast<float2 *>(Cb + g * kAp + 8 * nt + 2 * t) =
        make_float2(round_tf32(sgn * acc[nt][0]), round_tf32(sgn * acc[nt][1]));
    *reinterpret_cast<float2 *>(Cb + (g + 8) * kAp + 8 * nt + 2 * t) =
        make_float2(round_tf32(sgn * acc[nt][2]), round_tf32(sgn * acc[nt][3]));
  }
}

}  // namespace wy
}  // namespace la
