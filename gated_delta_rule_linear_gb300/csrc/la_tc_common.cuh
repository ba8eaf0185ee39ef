// Helpers shared by the tensor-core chunk kernels: bf16 packing, swizzled
// operand stores and TMA tensor-map creation on the host.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "la_internal.h"
#include "la_sm100.cuh"

namespace la {
namespace tc {

using namespace sm100;

constexpr int kC = 64;  // chunk length of the tensor-core kernels

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float *f) {
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ uint4 f32_to_bf16x8(const float *f) {
  uint4 u;
  __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}

// Write 16 consecutive fp32 values (columns c0..c0+15 of row `row`) as bf16
// into a K-major 128B-swizzled operand whose atoms are `atom_bytes` apart.
__device__ __forceinline__ void store_row16_bf16(uint8_t *base, uint32_t atom_bytes, int row, int c0,
                                                 const float *v) {
  uint8_t *a = base + (uint32_t)(c0 >> 6) * atom_bytes;
  const int cc = c0 & 63;
  *reinterpret_cast<uint4 *>(a + sw128_off(row, cc)) = f32_to_bf16x8(v);
  *reinterpret_cast<uint4 *>(a + sw128_off(row, cc + 8)) = f32_to_bf16x8(v + 8);
}

__device__ __forceinline__ float bf16_at(const uint8_t *base, uint32_t off) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(base + off));
}


// ---------------------------------------------------------- pipeline helpers

__device__ __forceinline__ void group_sync(int id) {
  asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}
// All-reduce of a predicate over one 128-thread group (also a barrier).
__device__ __forceinline__ bool group_all(bool v, int id) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id)
      : "memory");
  return r != 0;
}

// Bounded wait that also gives up as soon as another role has aborted.
constexpr uint32_t kSpinLimit = 1u << 24;  // polls before a wait gives up (well over 100 ms)
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              unsigned *status) {
  // rolled: every inlined copy of an unrolled spin loop costs kilobytes of
  // instruction cache, and instruction fetch limits these kernels when many SMs are busy
#pragma unroll 1
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  atomicOr(status, kStatusTimeout);
  return false;
}

// wait_or_abort for an mbarrier that another CTA of the cluster arrives on.
__device__ __forceinline__ bool wait_or_abort_cluster(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                                      unsigned *status) {
#pragma unroll 1
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  atomicOr(status, kStatusTimeout);
  return false;
}

// Group-wide wait: one elected thread polls the mbarrier while the rest of
// the 128-thread group sleeps on the group's named barrier (no issue slots
// used); the outcome is shared by the barrier reduction, which also orders
// memory for the whole group.
__device__ __forceinline__ bool group_wait(uint64_t *bar, uint32_t parity, int gtid, int bar_id,
                                           volatile int *abort_flag, unsigned *status) {
  bool ok = true;
  if (gtid == 0) ok = wait_or_abort(bar, parity, abort_flag, status);
  return group_all(ok, bar_id);
}

// 32 consecutive floats (16-byte aligned) into registers with 128-bit loads,
// before a loop that also stores to shared memory (so the loads are not
// serialised behind those stores).
__device__ __forceinline__ void load32(const float *p, float *out) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 t = reinterpret_cast<const float4 *>(p)[q];
    out[4 * q] = t.x;
    out[4 * q + 1] = t.y;
    out[4 * q + 2] = t.z;
    out[4 * q + 3] = t.w;
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

// 32 consecutive fp32 values (columns c0..c0+31 of `row`, c0 % 32 == 0) as
// bf16 into a K-major 128B-swizzled operand with atoms `atom_bytes` apart.
__device__ __forceinline__ void store_row32_bf16(uint8_t *base, uint32_t atom_bytes, int row, int c0,
                                                 const float *v) {
  uint8_t *a = base + (uint32_t)(c0 >> 6) * atom_bytes;
  const int cc = c0 & 63;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint4 u;
    u.x = pack_bf16(v[8 * g + 0], v[8 * g + 1]);
    u.y = pack_bf16(v[8 * g + 2], v[8 * g + 3]);
    u.z = pack_bf16(v[8 * g + 4], v[8 * g + 5]);
    u.w = pack_bf16(v[8 * g + 6], v[8 * g + 7]);
    *reinterpret_cast<uint4 *>(a + sw128_off(row, cc + 8 * g)) = u;
  }
}

__device__ __forceinline__ void unpack8(const uint4 &u, float *f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ uint4 pack8(const float *f) {
  uint4 u;
  u.x = pack_bf16(f[0], f[1]);
  u.y = pack_bf16(f[2], f[3]);
  u.z = pack_bf16(f[4], f[5]);
  u.w = pack_bf16(f[6], f[7]);
  return u;
}


// ---------------------------------------------------------------- host side

inline PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
inline std::once_flag g_encode_once;

inline bool encode_fn() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 3-D map over a [BH][T][d] row-major tensor, box {box_x, 64, 1}.
inline bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, int d, int T,
              int BH, int box_x, CUtensorMapSwizzle sw) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * esize, (cuuint64_t)d * esize * T};
  cuuint32_t box[3] = {(cuuint32_t)box_x, (cuuint32_t)kC, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, dt, 3, const_cast<void *>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


}  // namespace tc
}  // namespace la
