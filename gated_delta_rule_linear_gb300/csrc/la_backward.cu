// la_chunk_bwd: the backward pass of la_chunk_fwd for plain linear attention,
// RetNet's fixed decay and the data-dependent scalar decay ("Talk Linear
// Attention" sections 2.1 and 5.2; the states are recomputed, as section
// 4.1.2 describes, not stored). With alpha = 1 or gamma_h (for the scalar
// decay, alpha^(t-s) reads as the product of the gates of s+1 .. t),
//
//   dq_t = alpha^(t+1) S0 dO_t + sum_{s<=t} alpha^(t-s) (dO_t . v_s) k_s
//   dk_s = sum_{t>=s} alpha^(t-s) (dO_t . v_s) q_t + alpha^(T-1-s) dS v_s
//   dv_s = sum_{t>=s} alpha^(t-s) (q_t . k_s) dO_t + alpha^(T-1-s) dS^T k_s
//   dS0  = sum_t alpha^(t+1) q_t dO_t^T + alpha^T dS
//
// Each line is itself a causal linear attention with the same decay, so the
// backward runs the forward kernels three times: dq directly (queries dO,
// keys v, values k, initial state S0^T); dk and dv on the time-reversed
// sequences (queries v / k, keys dO / q, values q / dO, initial states
// dS^T / alpha and dS / alpha), and dS0 = alpha times the last pass's final
// state. The reversed passes are the forward kernels' reversed runs, which
// read and write the tensors in stored order, so nothing is copied; this file
// adds the initial-state preparation. For the scalar decay the reversed runs
// take each position's gate from the stored token after it, so the initial
// states need no division, dS0 = alpha_0 times the last pass's final state,
// and the log-gate gradient is a suffix sum,
//
//   dg_tau = sum_{u >= tau} (q_u . dq_u - k_u . dk_u) + sum(dS_final ⊙ S_final),
//
// with S_final from a fourth (forward) pass. GLA ("Talk Linear Attention"
// section 5.1) is the same channel by channel: its decay acts on the key
// channels, which are the value axis of the dq and dk passes, so those run on
// the outer-product gate (unit gates on their key axis, g on their value
// axis) and dv on GLA itself; dS0[c] = exp(g_0[c]) times row c of the last
// pass's final state, and dg[c] is the suffix sum of q[c] dq[c] - k[c] dk[c]
// plus row c's sum of dS_final ⊙ S_final.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdint>

#include "la_internal.h"

namespace la {
namespace {

// Initial states of the three passes, per head (alpha = exp(g_h) for RetNet, 1 otherwise):
// s0t = S0^T, dst = dS^T / alpha, dss = dS / alpha   ([B*H][.][.] float32)
__global__ void __launch_bounds__(256) state_prep_kernel(const float *__restrict__ S0, const float *__restrict__ dS,
                                                         const float *__restrict__ g, int H, int dk, int dv,
                                                         float *__restrict__ s0t, float *__restrict__ dst,
                                                         float *__restrict__ dss) {
  const int bh = blockIdx.y;
  const float inv = g ? expf(-__ldg(g + bh % H)) : 1.f;  // g: RetNet's per-head log-decay, else NULL
  const size_t base = (size_t)bh * dk * dv;
  for (int i = blockIdx.x * 256 + threadIdx.x; i < dk * dv; i += gridDim.x * 256) {
    const int c = i / dv, v = i % dv;  // element (c, v) of a [dk][dv] state
    if (S0) s0t[base + (size_t)v * dk + c] = S0[base + i];
    if (dS) {
      const float x = dS[base + i] * inv;
      dst[base + (size_t)v * dk + c] = x;
      dss[base + i] = x;
    }
  }
}

// dS0 = alpha * S, per head: alpha = exp(g[h]) (RetNet, gstride 0) or the
// first token's gate exp(g[bh * gstride]) (scalar decay, gstride T)
__global__ void __launch_bounds__(256) scale_state_kernel(const float *__restrict__ S, const float *__restrict__ g,
                                                          int H, long long gstride, int n, float *__restrict__ out) {
  const int bh = blockIdx.y;
  const float a = g ? expf(__ldg(g + (gstride ? (size_t)bh * gstride : (size_t)(bh % H)))) : 1.f;
  for (int i = blockIdx.x * 256 + threadIdx.x; i < n; i += gridDim.x * 256)
    out[(size_t)bh * n + i] = a * S[(size_t)bh * n + i];
}

template <typename T> __device__ __forceinline__ float ldf(const T *p);
template <> __device__ __forceinline__ float ldf<float>(const float *p) { return __ldg(p); }
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

// dg for the scalar decay in two launches. dg_tile_kernel, one CTA per
// (b, h, 256-token tile): w_u = q_u . dq_u - k_u . dk_u (a warp per token,
// lanes over the channels, coalesced) and the suffix sum of w inside the tile,
// written to dg, with the tile's total in `tot`. dg_carry_kernel, one CTA per
// (b, h): the final-state term c = sum(dS ⊙ S_final) plus the totals of the
// later tiles, added to every token of a tile.
template <typename Tin>
__global__ void __launch_bounds__(256) dg_tile_kernel(const Tin *__restrict__ q, const Tin *__restrict__ dq,
                                                      const Tin *__restrict__ k, const Tin *__restrict__ dk, int T,
                                                      int dkk, float *__restrict__ dg, float *__restrict__ tot) {
  __shared__ float red[8];
  __shared__ float wt[256];
  const int bh = blockIdx.x, tile = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t base = (size_t)bh * T;
  const int t0 = tile * 256, per = dkk / 32;  // channels per lane (2 or 4)
#pragma unroll 4
  for (int i = warp; i < 256; i += 8) {
    const int u = t0 + i;
    float x = 0.f;
    if (u < T) {
      const size_t r = (base + u) * dkk + (size_t)lane * per;
      for (int e = 0; e < per; ++e) x += ldf(q + r + e) * ldf(dq + r + e) - ldf(k + r + e) * ldf(dk + r + e);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    if (lane == 0) wt[i] = x;
  }
  __syncthreads();
  float w = wt[tid];
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {  // inclusive suffix sum within the warp
    const float y = __shfl_down_sync(0xffffffffu, w, off);
    if (lane + off < 32) w += y;
  }
  if (lane == 0) red[warp] = w;
  __syncthreads();
  float later = 0.f, all = 0.f;
#pragma unroll
  for (int wq = 0; wq < 8; ++wq) {
    all += red[wq];
    if (wq > warp) later += red[wq];
  }
  if (t0 + tid < T) dg[base + t0 + tid] = later + w;
  if (tid == 0) tot[(size_t)bh * gridDim.y + tile] = all;
}

__global__ void __launch_bounds__(256) dg_carry_kernel(const float *__restrict__ dS, const float *__restrict__ S_final,
                                                       const float *__restrict__ tot, int ntiles, int T, int n,
                                                       float *__restrict__ dg) {
  __shared__ float red[8];
  __shared__ float carry[1024];  // suffix sums of the tile totals, in chunks of 1024 tiles
  const int bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float c = 0.f;
  if (dS)
    for (int i = tid; i < n; i += 256) c = fmaf(dS[(size_t)bh * n + i], S_final[(size_t)bh * n + i], c);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
  if (lane == 0) red[warp] = c;
  __syncthreads();
  c = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) c += red[w];
  // tiles from the end, 1024 at a time: carry of tile j = c + totals of tiles j+1 ..
  for (int j1 = ntiles; j1 > 0; j1 -= 1024) {
    const int j0 = j1 > 1024 ? j1 - 1024 : 0;
    __syncthreads();
    if (tid == 0) {
      float acc = c;
      for (int j = j1 - 1; j >= j0; --j) {
        carry[j - j0] = acc;
        acc += tot[(size_t)bh * ntiles + j];
      }
      red[0] = acc;
    }
    __syncthreads();
    for (int u = j0 * 256 + tid; u < j1 * 256 && u < T; u += 256) dg[(size_t)bh * T + u] += carry[u / 256 - j0];
    c = red[0];
  }
}

// GLA: dS0[c][j] = exp(g_0[c]) * S[c][j], the first token's per-channel gate
__global__ void __launch_bounds__(256) scale_rows_kernel(const float *__restrict__ S, const float *__restrict__ g,
                                                         int T, int dkk, int dv, float *__restrict__ out) {
  const int bh = blockIdx.y;
  const size_t base = (size_t)bh * dkk * dv;
  for (int i = blockIdx.x * 256 + threadIdx.x; i < dkk * dv; i += gridDim.x * 256)
    out[base + i] = expf(__ldg(g + (size_t)bh * T * dkk + i / dv)) * S[base + i];
}

// dg for GLA, per key channel, in three launches. dgc_tile_kernel, one CTA
// per (b, h, 256-token tile), one thread per channel: the suffix sum over the
// tile of q[c] dq[c] - k[c] dk[c] (coalesced over the channels), with the
// tile's totals in `tot`. dgc_suffix_kernel turns the totals into carries
// (row sums of dS ⊙ S_final plus the later tiles' totals); dgc_carry_kernel
// adds them to the tile's tokens.
template <typename Tin>
__global__ void __launch_bounds__(128) dgc_tile_kernel(const Tin *__restrict__ q, const Tin *__restrict__ dq,
                                                       const Tin *__restrict__ k, const Tin *__restrict__ dk, int T,
                                                       int dkk, float *__restrict__ dg, float *__restrict__ tot) {
  const int bh = blockIdx.x, tile = blockIdx.y, c = threadIdx.x;
  if (c >= dkk) return;
  const int t0 = tile * 256, t1 = min(t0 + 256, T);
  float acc = 0.f;
  for (int u1 = t1; u1 > t0; u1 -= 8) {  // eight tokens' loads in flight, then their suffix sums
    float w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int u = u1 - 1 - e;
      const size_t r = ((size_t)bh * T + u) * dkk + c;
      w[e] = (u >= t0) ? ldf(q + r) * ldf(dq + r) - ldf(k + r) * ldf(dk + r) : 0.f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int u = u1 - 1 - e;
      acc += w[e];
      if (u >= t0) dg[((size_t)bh * T + u) * dkk + c] = acc;
    }
  }
  tot[((size_t)bh * gridDim.y + tile) * dkk + c] = acc;
}

// One CTA per (b, h), a thread per channel: turns the per-tile totals into
// per-tile carries in place, tot[tile] <- sum(dS ⊙ S_final)[c] + the totals of
// the later tiles (a suffix sum, taken once per channel).
__global__ void __launch_bounds__(128) dgc_suffix_kernel(const float *__restrict__ dS, const float *__restrict__ S_final,
                                                         float *__restrict__ tot, int ntiles, int dkk, int dv) {
  const int bh = blockIdx.x, c = threadIdx.x;
  if (c >= dkk) return;
  float carry = 0.f;
  if (dS)
    for (int j = 0; j < dv; ++j) {
      const size_t i = ((size_t)bh * dkk + c) * dv + j;
      carry = fmaf(dS[i], S_final[i], carry);
    }
  for (int tl = ntiles - 1; tl >= 0; --tl) {
    float *t = tot + ((size_t)bh * ntiles + tl) * dkk + c;
    const float x = *t;
    *t = carry;
    carry += x;
  }
}

// One CTA per (b, h, tile): adds the tile's carry to its tokens.
__global__ void __launch_bounds__(128) dgc_carry_kernel(const float *__restrict__ tot, int ntiles, int T, int dkk,
                                                        float *__restrict__ dg) {
  const int bh = blockIdx.x, tile = blockIdx.y, c = threadIdx.x;
  if (c >= dkk) return;
  const float carry = tot[((size_t)bh * ntiles + tile) * dkk + c];
  const int t0 = tile * 256, t1 = min(t0 + 256, T);
  for (int u0 = t0; u0 < t1; u0 += 8) {  // eight tokens read, then written
    float x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = (u0 + e < t1) ? dg[((size_t)bh * T + u0 + e) * dkk + c] : 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (u0 + e < t1) dg[((size_t)bh * T + u0 + e) * dkk + c] = x[e] + carry;
  }
}

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The forward recurrence over the time-reversed sequence, through the
// kernels' reversed runs (tensor cores for bf16, CUDA cores for float32).
int run_reversed(const void *q, const void *k, const void *v, const float *g, const float *beta, void *o,
                 const float *S0, float *S_final, int B, int H, int T, int dk, int dv, int kind, bool f32,
                 cudaStream_t s) {
  ChunkParams p{q, k, v, g, beta, o, S0, S_final, B, H, T, dk, dv, 64, kind, f32 ? 1 : 0, status_word(), 1};
  if (!p.status) {
    set_error("la_chunk_bwd: no CUDA device available (%s)", cudaGetErrorString(cudaGetLastError()));
    return LA_ERR_CUDA;
  }
  return f32 ? launch_chunk_simt(p, s) : launch_chunk_ws(p, s);
}

}  // namespace
}  // namespace la

using namespace la;

extern "C" int la_chunk_bwd(const void *q, const void *k, const void *v, const float *g, const void *dO,
                            const float *dS_final, const float *S0, void *dq_out, void *dk_out, void *dv_out,
                            float *dS0, float *dg_out, int B, int H, int T, int dk, int dv, int C, int mode,
                            la_stream_t stream) {
  la::NvtxRange nvtx_range("la_chunk_bwd");
  void *dq = dq_out, *dkg = dk_out, *dvg = dv_out;
  const int dk_ = dk, dv_ = dv;
  const char *fn = "la_chunk_bwd";
  set_error("%s", "");
  const int kind = mode & 0xff;
  if (!q || !k || !v || !dO || !dq || !dkg || !dvg) {
    set_error("%s: q, k, v, dO, dq, dk and dv are required", fn);
    return LA_ERR_INVALID_ARG;
  }
  if (B < 1 || H < 1 || T < 1 || (long long)B * H > 65535) {
    set_error("%s: need B, H, T >= 1 and B*H <= 65535 (got %d, %d, %d)", fn, B, H, T);
    return LA_ERR_INVALID_ARG;
  }
  if ((dk_ != 64 && dk_ != 128) || (dv_ != 64 && dv_ != 128)) {
    set_error("%s: dk and dv must be 64 or 128 (got %d, %d)", fn, dk_, dv_);
    return LA_ERR_UNSUPPORTED;
  }
  if ((mode & ~(0xff | LA_F32)) != 0 ||
      (kind != LA_LINEAR && kind != LA_RETNET && kind != LA_SCALAR_GATE && kind != LA_GLA)) {
    set_error("%s: mode 0x%x: this entry point covers LA_LINEAR, LA_RETNET, LA_SCALAR_GATE and LA_GLA "
              "(optionally | LA_F32); LA_GDN has la_chunk_bwd_delta", fn, mode);
    return (mode & ~(0xff | LA_F32)) == 0 && kind >= LA_LINEAR && kind <= LA_OUTER_GATE ? LA_ERR_UNSUPPORTED
                                                                                  : LA_ERR_INVALID_ARG;
  }
  const bool scalar = kind == LA_SCALAR_GATE, gla = kind == LA_GLA;
  if ((kind == LA_LINEAR) != (g == nullptr)) {
    set_error("%s: LA_RETNET needs g (float32 [H]), LA_SCALAR_GATE g [B][H][T], LA_GLA g [B][H][T][dk]; "
              "LA_LINEAR takes none", fn);
    return LA_ERR_INVALID_ARG;
  }
  if (dg_out && !scalar && !gla) {
    set_error("%s: dg is the gradient of the data-dependent log-gates (LA_SCALAR_GATE, LA_GLA; NULL otherwise)", fn);
    return LA_ERR_INVALID_ARG;
  }
  if (gla && (mode & LA_F32)) {
    set_error("%s: the LA_GLA backward takes bfloat16 inputs only", fn);
    return LA_ERR_UNSUPPORTED;
  }
  if (C != 0 && C != 64) {
    set_error("%s: chunk length C=%d is not implemented in this build (use 0 or 64)", fn, C);
    return LA_ERR_UNSUPPORTED;
  }
  if (dg_out && (T + 255) / 256 > 65535) {  // dg's 256-token tiles index the grid's y dimension
    set_error("%s: dg covers T <= %d tokens (got %d)", fn, 65535 * 256, T);
    return LA_ERR_UNSUPPORTED;
  }
  const void *p16[] = {q, k, v, dO, dq, dkg, dvg};
  for (const void *ptr : p16)
    if (!al16(ptr)) {
      set_error("%s: q, k, v, dO, dq, dk and dv must be 16-byte aligned", fn);
      return LA_ERR_INVALID_ARG;
    }
  if ((S0 && !al16(S0)) || (dS_final && !al16(dS_final)) || (dS0 && !al16(dS0)) || (g && !al16(g)) ||
      (dg_out && !al16(dg_out))) {
    set_error("%s: S0, dS_final, dS0, g and dg must be 16-byte aligned", fn);
    return LA_ERR_INVALID_ARG;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool f32 = (mode & LA_F32) != 0;
  const size_t esz = f32 ? 4 : 2;
  const size_t BH = (size_t)B * H;
  // workspace: three initial states and the last pass's final state; for dg also the
  // forward's final state and a scratch output of the forward pass that produces it
  const size_t n_s = BH * dk_ * dv_ * 4;
  const int ntiles = (T + 255) / 256;  // dg's 256-token tiles
  const size_t ntot = (BH * ntiles * (gla ? dk_ : 1) + 3) & ~static_cast<size_t>(3);  // their totals (floats)
  // GLA: zero key-axis gates [B][H][T][dv] for the outer-product-gate passes (dq, dk)
  const size_t nzero = gla ? BH * (size_t)T * dv_ * 4 : 0;
  const size_t bytes = (dg_out ? 5 : 4) * n_s + (dg_out ? BH * (size_t)T * dv_ * esz + ntot * 4 : 0) + nzero;
  uint8_t *ws = nullptr;
  cudaMemPool_t pool = library_pool();
  if (!pool) {
    set_error("%s: could not create the workspace pool: %s", fn, cudaGetErrorString(cudaGetLastError()));
    return LA_ERR_CUDA;
  }
  cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&ws), bytes, pool, s);
  if (e != cudaSuccess) {
    set_error("%s: workspace allocation of %zu bytes failed: %s", fn, bytes, cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  float *s0t = reinterpret_cast<float *>(ws), *dst = s0t + BH * dk_ * dv_, *dss = dst + BH * dk_ * dv_,
        *sfin = dss + BH * dk_ * dv_, *sT = sfin + BH * dk_ * dv_;
  float *tiles = sT + BH * dk_ * dv_;  // dg's per-tile totals, then the forward's scratch output
  uint8_t *oscr = reinterpret_cast<uint8_t *>(tiles + (dg_out ? ntot : 0));
  float *zg = reinterpret_cast<float *>(oscr + (dg_out ? BH * (size_t)T * dv_ * esz : 0));
  int rc = LA_OK;
  auto fail = [&](const char *what) {
    if (rc == LA_OK) {
      set_error("%s: %s failed: %s", fn, what, la_last_error()[0] ? la_last_error() : cudaGetErrorString(cudaGetLastError()));
      rc = LA_ERR_CUDA;
    }
  };
  // RetNet's reversed passes use the unshifted per-head decay, so their initial
  // states carry 1 / gamma; the scalar decay's reversed runs shift the gates instead
  const float *g_head = kind == LA_RETNET ? g : nullptr;
  if (gla && cudaMemsetAsync(zg, 0, nzero, s) != cudaSuccess) fail("zero gates");
  if (S0 || dS_final) {
    state_prep_kernel<<<dim3(8, (unsigned)BH), 256, 0, s>>>(S0, dS_final, g_head, H, dk_, dv_, s0t, dst, dss);
    if (cudaGetLastError() != cudaSuccess) fail("initial-state preparation");
  }
  const int fwd_mode = mode & (0xff | LA_F32);
  // dq: queries dO, keys v, values k (key width dv, value width dk), initial state S0^T; for GLA the
  // decay acts on k's channels, the value axis of this pass: the outer-product gate with unit key gates
  if (rc == LA_OK) {
    const int r = gla ? la_chunk_fwd(dO, v, k, zg, g, dq, S0 ? s0t : nullptr, nullptr, B, H, T, dv_, dk_, C,
                                     LA_OUTER_GATE, stream)
                      : la_chunk_fwd(dO, v, k, g, nullptr, dq, S0 ? s0t : nullptr, nullptr, B, H, T, dv_, dk_, C,
                                     fwd_mode, stream);
    if (r != LA_OK) rc = r;
  }
  // dk (reversed run): queries v, keys dO, values q, initial state dS^T (/ gamma); GLA again on the value axis
  if (rc == LA_OK)
    rc = gla ? run_reversed(v, dO, q, zg, g, dkg, dS_final ? dst : nullptr, nullptr, B, H, T, dv_, dk_, kOuter, f32, s)
             : run_reversed(v, dO, q, g, nullptr, dkg, dS_final ? dst : nullptr, nullptr, B, H, T, dv_, dk_, kind, f32,
                            s);
  // dv (reversed run): queries k, keys q, values dO, initial state dS (/ gamma); its final state x alpha = dS0
  if (rc == LA_OK)
    rc = run_reversed(k, q, dO, g, nullptr, dvg, dS_final ? dss : nullptr, dS0 ? sfin : nullptr, B, H, T, dk_, dv_,
                      kind, f32, s);
  if (rc == LA_OK && dS0) {
    if (gla)
      scale_rows_kernel<<<dim3(8, (unsigned)BH), 256, 0, s>>>(sfin, g, T, dk_, dv_, dS0);
    else
      scale_state_kernel<<<dim3(8, (unsigned)BH), 256, 0, s>>>(sfin, g, H, scalar ? (long long)T : 0ll, dk_ * dv_,
                                                                dS0);
    if (cudaGetLastError() != cudaSuccess) fail("dS0 scaling");
  }
  if (rc == LA_OK && dg_out) {
    // the forward's final state (for the dS_final term of dg), then the suffix sums
    if (dS_final) {
      const int r = la_chunk_fwd(q, k, v, g, nullptr, oscr, S0, sT, B, H, T, dk_, dv_, C, fwd_mode, stream);
      if (r != LA_OK) rc = r;
    }
    if (rc == LA_OK && gla) {
      const dim3 grid((unsigned)BH, (unsigned)ntiles);
      dgc_tile_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(
          static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(dq),
          static_cast<const __nv_bfloat16 *>(k), static_cast<const __nv_bfloat16 *>(dkg), T, dk_, dg_out, tiles);
      if (cudaGetLastError() == cudaSuccess)
        dgc_suffix_kernel<<<(unsigned)BH, 128, 0, s>>>(dS_final, sT, tiles, ntiles, dk_, dv_);
      if (cudaGetLastError() == cudaSuccess)
        dgc_carry_kernel<<<grid, 128, 0, s>>>(tiles, ntiles, T, dk_, dg_out);
      if (cudaGetLastError() != cudaSuccess) fail("dg suffix sums");
    } else if (rc == LA_OK) {
      const dim3 grid((unsigned)BH, (unsigned)ntiles);
      if (f32)
        dg_tile_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float *>(q), static_cast<const float *>(dq),
                                                   static_cast<const float *>(k), static_cast<const float *>(dkg), T,
                                                   dk_, dg_out, tiles);
      else
        dg_tile_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(dq),
            static_cast<const __nv_bfloat16 *>(k), static_cast<const __nv_bfloat16 *>(dkg), T, dk_, dg_out, tiles);
      if (cudaGetLastError() == cudaSuccess)
        dg_carry_kernel<<<(unsigned)BH, 256, 0, s>>>(dS_final, sT, tiles, ntiles, T, dk_ * dv_, dg_out);
      if (cudaGetLastError() != cudaSuccess) fail("dg suffix sums");
    }
  }
  e = cudaFreeAsync(ws, s);
  if (rc == LA_OK && e != cudaSuccess) {
    set_error("%s: workspace release failed: %s", fn, cudaGetErrorString(e));
    rc = LA_ERR_CUDA;
  }
  return rc;
}
