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
