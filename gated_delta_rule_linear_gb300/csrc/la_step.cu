// One decode step of the recurrence for every (b, h): the recurrent form of
// linear attention ("Talk Linear Attention" section 2.1: constant-size state,
// o_t = S_t^T q_t; kernel-attention notes section 14 for the normalised
// variant) with the mode's decay and write rule.
//
// One CTA per (b, h); thread j owns state column j (the elu+1 normaliser z is
// column dv, updated as a value column whose input is 1). The column lives in
// registers for the step, so S is read once and written once -- the step is
// bound by those 2 * dk * W * 4 bytes of HBM traffic per head.
#include <cuda_bf16.h>

#include "la_internal.h"

namespace la {
namespace {

template <typename T> __device__ __forceinline__ float ldv(const T *p, size_t i);
template <> __device__ __forceinline__ float ldv<float>(const float *p, size_t i) { return __ldg(p + i); }
template <> __device__ __forceinline__ float ldv<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
  return __bfloat162float(p[i]);
}
template <typename T> __device__ __forceinline__ void stv(T *p, size_t i, float x);
template <> __device__ __forceinline__ void stv<float>(float *p, size_t i, float x) { p[i] = x; }
template <> __device__ __forceinline__ void stv<__nv_bfloat16>(__nv_bfloat16 *p, size_t i, float x) {
  p[i] = __float2bfloat16_rn(x);
}

template <typename Tin, int DK>
__global__ void __launch_bounds__(160) step_kernel(const StepParams p) {
  __shared__ float sq[DK], sk[DK], sa[DK];
  __shared__ float sden;
  const int bh = blockIdx.x, h = bh % p.H, j = threadIdx.x;
  const int dv = p.dv, kind = p.kind;
  const bool elu = kind == kElu1, delta = kind == kGdn || kind == kKda, outer = kind == kOuter;
  const int W = dv + (elu ? 1 : 0);
  const Tin *q = static_cast<const Tin *>(p.q);
  const Tin *k = static_cast<const Tin *>(p.k);
  const Tin *v = static_cast<const Tin *>(p.v);

  for (int c = j; c < DK; c += blockDim.x) {
    float qc = ldv(q, (size_t)bh * DK + c), kc = ldv(k, (size_t)bh * DK + c);
    if (elu) {
      qc = qc > 0.f ? qc + 1.f : __expf(qc);
      kc = kc > 0.f ? kc + 1.f : __expf(kc);
    }
    sq[c] = qc;
    sk[c] = kc;
    float a = 1.f;
    if (kind == kRetnet) a = __expf(__ldg(p.g + h));
    else if (kind == kGla || kind == kKda || outer) a = __expf(__ldg(p.g + (size_t)bh * DK + c));
    else if (kind == kScalar || (kind == kGdn && p.g)) a = __expf(__ldg(p.g + bh));
    sa[c] = a;
  }
  __syncthreads();
  const bool active = j < W;
  float out = 0.f;
  if (active) {
    float *S = p.S + (size_t)bh * DK * W + j;
    float s[DK];
    // outer-product gate: this value column's factor beta_j (log-gate in p.beta)
    const float av = (outer && j < dv) ? __expf(__ldg(p.beta + (size_t)bh * dv + j)) : 1.f;
#pragma unroll
    for (int c = 0; c < DK; ++c) s[c] = S[(size_t)c * W] * (sa[c] * av);   // decay first
    float w = (j < dv) ? ldv(v, (size_t)bh * dv + j) : 1.f;
    if (delta) {
      float r = 0.f;
#pragma unroll
      for (int c = 0; c < DK; ++c) r = fmaf(s[c], sk[c], r);
      const float b = p.beta ? __ldg(p.beta + bh) : 1.f;
      w = b * (w - r);
    }
#pragma unroll
    for (int c = 0; c < DK; ++c) {
      s[c] = fmaf(sk[c], w, s[c]);
      S[(size_t)c * W] = s[c];
      out = fmaf(s[c], sq[c], out);
    }
  }
  if (elu) {
    if (j == dv) sden = out;
    __syncthreads();
    if (j < dv) stv(static_cast<Tin *>(p.o), (size_t)bh * dv + j, out / sden);
  } else if (active) {
    stv(static_cast<Tin *>(p.o), (size_t)bh * dv + j, out);
  }
}

template <typename Tin>
int launch_typed(const StepParams &p, cudaStream_t stream) {
  const int W = p.dv + (p.kind == kElu1 ? 1 : 0);
  const int threads = ((W + 31) / 32) * 32;
  if (p.dk == 64) step_kernel<Tin, 64><<<p.B * p.H, threads, 0, stream>>>(p);
  else step_kernel<Tin, 128><<<p.B * p.H, threads, 0, stream>>>(p);
  return 0;
}

}  // namespace

int launch_step(const StepParams &p, cudaStream_t stream) {
  if (p.f32) launch_typed<float>(p, stream);
  else launch_typed<__nv_bfloat16>(p, stream);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("la_recurrent_step: launch failed: %s", cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  return LA_OK;
}

}  // namespace la
