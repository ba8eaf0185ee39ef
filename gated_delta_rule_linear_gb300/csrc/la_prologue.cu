// la_prologue: the per-token steps between the q/k/v/gate projections and the
// chunk forward pass, in one streaming pass over HBM:
//
//   short convolution  x~_t[c] = sum_{tau < K} w[h][c][tau] x_{t - tau}[c]  on q, k and v
//                      ("LLM attention optimisation: linear attention", DeltaNet
//                      section: a depthwise short convolution after the
//                      projections; K <= 4), history rows from the previous call
//   L2 normalisation   x / max(||x||_2, 1e-6) per token (q and/or k, optional)
//   gate activation    g = logsigmoid(a) / tau ("Talk Linear Attention" section
//                      5.1, log of sigmoid(.)^(1/tau)) or g = -softplus(a) / tau
//   write strength     beta = sigmoid(a_beta)
//
// Memory-bound: every byte is read and written once. One CTA of 256 threads
// per (b, h) and 128-token tile, two CTAs per SM. A tile's rows (and the K-1
// rows before it) of each of q, k and v are contiguous in memory, so one
// thread starts three bulk asynchronous copies into shared memory (one
// mbarrier each) and the CTA forms the gates and beta while they land. For a
// tensor of width d a thread then owns one 8-channel group (16 bytes of a row)
// of a block of consecutive rows and keeps the previous K-1 raw rows of its
// channels in registers; the threads of a row are consecutive lanes, so the L2
// norm's sum of squares is a shuffle reduction over d / 8 lanes. Outputs are
// written straight from registers (16 bytes a thread, coalesced).
#include <cuda_bf16.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "la_internal.h"
#include "la_sm100.cuh"

namespace la {
namespace {

using namespace sm100;

constexpr int kThreads = 256;
constexpr int kTile = 128;  // tokens per CTA
constexpr int kMaxK = 4;
constexpr int kHalo = kMaxK - 1;
constexpr uint32_t kSpinLimit = 1u << 22;  // polls (with back-off) before a copy is given up

struct ProParams {
  const __nv_bfloat16 *x[3];  // q, k, v projections
  const float *w[3];          // [H][d][K] or null (no convolution)
  __nv_bfloat16 *y[3];
  const __nv_bfloat16 *hist_in;  // [B][H][K-1][2 dk + dv] or null
  __nv_bfloat16 *hist_out;       // same layout or null
  const float *a_gate, *a_beta;
  float *g, *beta;
  unsigned *status;
  int B, H, T, K, gate_kind, gate_width, l2mask;
  float inv_tau;
  uint32_t wait_limit;  // polls before a copy is given up (kSpinLimit unless a test shortens it)
  int skip_k_copy;      // test hook, 0 in normal use: arm k's barrier but start no copy
};

__host__ __device__ constexpr uint32_t tile_bytes(int d) { return (uint32_t)(kTile + kHalo) * d * 2u; }
// the head's convolution weights in shared memory, [tensor][channel][tap], taps padded to kMaxK
__host__ __device__ constexpr uint32_t wts_bytes(int dk, int dv) { return (uint32_t)(2 * dk + dv) * kMaxK * 4u; }

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float *f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint4 f32_to_bf16x8(const float *f) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t *>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Rows t0-3 .. t0+kTile-1 of one tensor: row rr of the shared tile is token
// t0 - 3 + rr. The copy covers the tokens in [0, T); halo rows before token 0
// are filled from the history (or zero) by the threads after the copy lands.
template <int D>
__device__ __forceinline__ void issue_tile(const ProParams &p, int which, int bh, int t0, uint8_t *tile,
                                           uint64_t *bar) {
  const int lo = max(t0 - kHalo, 0), hi = min(t0 + kTile, p.T);
  const uint32_t bytes = (uint32_t)(hi - lo) * D * 2u;
  mbar_arrive_expect_tx(bar, bytes);
  // the test hook leaves k's barrier waiting for bytes that never come (no copy
  // is in flight when the wait gives up)
  if (p.skip_k_copy && which == 1) return;
  bulk_load(tile + (size_t)(lo - (t0 - kHalo)) * D * 2, p.x[which] + ((size_t)bh * p.T + lo) * D, bytes, bar);
}

// One tensor of one tile from shared memory: convolution, optional L2 norm, store.
template <int D>
__device__ __forceinline__ void conv_tile(const ProParams &p, int which, int bh, int t0, const uint8_t *tile,
                                          const float *wsm) {
  constexpr int G = D / 8;         // 16-byte channel groups per row
  constexpr int S = kThreads / G;  // row streams
  constexpr int R = kTile / S;     // consecutive rows per stream
  const int tid = threadIdx.x, cg = tid % G, st = tid / G, lane = tid & 31;
  const int T = p.T;
  __nv_bfloat16 *y = p.y[which] + (size_t)bh * T * D + cg * 8;
  const bool l2 = (p.l2mask >> which) & 1;
  const unsigned gmask = (G == 32 ? 0xffffffffu : ((1u << G) - 1u)) << (lane & ~(G - 1));
  float w[kMaxK][8];  // this thread's 8 channels, tap-major (16-byte rows in shared memory)
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float4 w4 = *reinterpret_cast<const float4 *>(wsm + (cg * 8 + e) * kMaxK);
    w[0][e] = w4.x;
    w[1][e] = w4.y;
    w[2][e] = w4.z;
    w[3][e] = w4.w;
  }
  const int r0 = st * R;  // first row of the block, relative to t0
  const uint8_t *trow = tile + (size_t)kHalo * D * 2 + cg * 16;  // row of token t0
  float win[kHalo][8];
#pragma unroll
  for (int j = 1; j <= kHalo; ++j) bf16x8_to_f32(*reinterpret_cast<const uint4 *>(trow + (r0 - j) * D * 2), win[j - 1]);
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int t = t0 + r0 + i;
    if (t >= T) break;  // uniform across the row's lanes
    float xc[8], acc[8];
    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(trow + (r0 + i) * D * 2), xc);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float a = w[0][e] * xc[e];
#pragma unroll
      for (int tau = 1; tau < kMaxK; ++tau) a = fmaf(w[tau][e], win[tau - 1][e], a);
      acc[e] = a;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {  // slide the window
#pragma unroll
      for (int tau = kHalo - 1; tau > 0; --tau) win[tau][e] = win[tau - 1][e];
      win[0][e] = xc[e];
    }
    if (l2) {
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(acc[e], acc[e], ss);
#pragma unroll
      for (int off = G / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(gmask, ss, off);
      const float sc = 1.f / fmaxf(sqrtf(ss), 1e-6f);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] *= sc;
    }
    *reinterpret_cast<uint4 *>(y + (size_t)t * D) = f32_to_bf16x8(acc);
  }
}

__device__ __forceinline__ float softplus_f(float a) { return fmaxf(a, 0.f) + log1pf(expf(-fabsf(a))); }

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 2) prologue_kernel(const ProParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  auto tile = [&](int which) { return smem + (which == 0 ? 0u : (which == 1 ? tile_bytes(DK) : 2u * tile_bytes(DK))); };
  float *wsm = reinterpret_cast<float *>(smem + 2 * tile_bytes(DK) + tile_bytes(DV));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 2 * tile_bytes(DK) + tile_bytes(DV) + wts_bytes(DK, DV));
  const int bh = blockIdx.y, t0 = blockIdx.x * kTile, T = p.T, K = p.K;
  const int hist_w = 2 * DK + DV;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    issue_tile<DK>(p, 0, bh, t0, tile(0), &bars[0]);
    issue_tile<DK>(p, 1, bh, t0, tile(1), &bars[1]);
    issue_tile<DV>(p, 2, bh, t0, tile(2), &bars[2]);
  }
  // the head's weights, taps padded with zeros (no weights: the identity)
  {
    const int h = bh % p.H;
    for (int i = threadIdx.x; i < (2 * DK + DV) * kMaxK; i += kThreads) {
      const int c = i / kMaxK, tau = i % kMaxK;
      const int which = c < DK ? 0 : (c < 2 * DK ? 1 : 2);
      const int D = which < 2 ? DK : DV, cc = c - (which == 0 ? 0 : (which == 1 ? DK : 2 * DK));
      const float *wp = p.w[which];
      wsm[i] = wp ? ((tau < K) ? __ldg(wp + ((size_t)h * D + cc) * K + tau) : 0.f) : (tau == 0 ? 1.f : 0.f);
    }
  }
  // gates and beta while the tiles land: loads in batches of independent
  // requests, then the activations and stores
  const int n = min(kTile, T - t0);
  const int tid = threadIdx.x;
  const float *__restrict__ a_beta = p.a_beta;
  const size_t bbase = (size_t)bh * T + t0;
  const float ba = (a_beta && tid < n) ? __ldg(a_beta + bbase + tid) : 0.f;
  if (p.gate_kind != LA_GATE_NONE) {
    constexpr int kBatch = 16;
    const float *__restrict__ a_gate = p.a_gate;
    float *__restrict__ g = p.g;
    const size_t base = ((size_t)bh * T + t0) * p.gate_width;
    const int cnt = n * p.gate_width;
    const bool logsig = p.gate_kind == LA_GATE_LOGSIGMOID;
    for (int i0 = tid; i0 < cnt; i0 += kThreads * kBatch) {
      float a[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int idx = i0 + j * kThreads;
        a[j] = idx < cnt ? __ldg(a_gate + base + idx) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int idx = i0 + j * kThreads;
        if (idx < cnt) g[base + idx] = -(logsig ? softplus_f(-a[j]) : softplus_f(a[j])) * p.inv_tau;
      }
    }
  }
  if (a_beta && tid < n) p.beta[bbase + tid] = 1.f / (1.f + expf(-ba));
  // halo rows before token 0 (first tile only): the history, or zero
  if (t0 == 0) {
    for (int i = threadIdx.x; i < kHalo * (hist_w / 8); i += kThreads) {
      const int rr = i / (hist_w / 8), c8 = (i % (hist_w / 8)) * 8, tt = rr - kHalo;  // token -3 .. -1
      const int which = c8 < DK ? 0 : (c8 < 2 * DK ? 1 : 2);
      const int D = which < 2 ? DK : DV, c = c8 - (which == 0 ? 0 : (which == 1 ? DK : 2 * DK));
      uint4 u = make_uint4(0, 0, 0, 0);
      if (p.hist_in && tt >= -(K - 1))
        u = *reinterpret_cast<const uint4 *>(p.hist_in + ((size_t)bh * (K - 1) + (K - 1) + tt) * hist_w + c8);
      *reinterpret_cast<uint4 *>(tile(which) + ((size_t)rr * D + c) * 2) = u;
    }
  }
  __syncthreads();  // barrier initialisation and halo rows visible to every thread
  bool ok = true;
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    if (threadIdx.x == 0 && !mbar_wait_bounded(&bars[i], 0, p.wait_limit)) {
      atomicOr(p.status, kStatusTimeout);
      ok = false;
    }
  }
  ok = __syncthreads_and(ok);
  if (ok) {
    conv_tile<DK>(p, 0, bh, t0, tile(0), wsm);
    conv_tile<DK>(p, 1, bh, t0, tile(1), wsm + DK * kMaxK);
    conv_tile<DV>(p, 2, bh, t0, tile(2), wsm + 2 * DK * kMaxK);
  }
  // the last K-1 raw rows of history ++ x, by the CTA holding the last token
  if (p.hist_out && K > 1 && t0 + kTile >= T) {
    const int K1 = K - 1, G = hist_w / 8;
    for (int i = threadIdx.x; i < K1 * G; i += kThreads) {
      const int j = i / G, c8 = (i % G) * 8, tt = T - K1 + j;
      const int which = c8 < DK ? 0 : (c8 < 2 * DK ? 1 : 2);
      const int D = which < 2 ? DK : DV, c = c8 - (which == 0 ? 0 : (which == 1 ? DK : 2 * DK));
      uint4 u = make_uint4(0, 0, 0, 0);
      if (tt >= 0)
        u = __ldg(reinterpret_cast<const uint4 *>(p.x[which] + ((size_t)bh * T + tt) * D + c));
      else if (p.hist_in)
        u = *reinterpret_cast<const uint4 *>(p.hist_in + ((size_t)bh * K1 + K1 + tt) * hist_w + c8);
      *reinterpret_cast<uint4 *>(p.hist_out + ((size_t)bh * K1 + j) * hist_w + c8) = u;
    }
  }
}

template <int DK, int DV>
int launch_prologue(const ProParams &p, cudaStream_t s) {
  const size_t smem = 2 * tile_bytes(DK) + tile_bytes(DV) + wts_bytes(DK, DV) + 64;
  // set on every launch: the attribute belongs to the current device's context
  if (cudaFuncSetAttribute(prologue_kernel<DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return LA_ERR_CUDA;
  const dim3 grid((p.T + kTile - 1) / kTile, p.B * p.H);
  prologue_kernel<DK, DV><<<grid, kThreads, smem, s>>>(p);
  return LA_OK;
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

}  // namespace
}  // namespace la

using namespace la;

extern "C" int la_prologue(const void *xq, const void *xk, const void *xv, const float *wq, const float *wk,
                           const float *wv, int K, const void *hist_in, void *hist_out, const float *a_gate,
                           int gate_kind, int gate_width, float tau, const float *a_beta, void *q, void *k,
                           void *v, float *g, float *beta, int B, int H, int T, int dk, int dv, int flags,
                           la_stream_t stream) {
  la::NvtxRange nvtx_range("la_prologue");
  const char *fn = "la_prologue";
  set_error("%s", "");
  if (!xq || !xk || !xv || !q || !k || !v) {
    set_error("%s: xq, xk, xv, q, k and v are required", fn);
    return LA_ERR_INVALID_ARG;
  }
  if (B < 1 || H < 1 || T < 1 || (long long)B * H > 65535) {
    set_error("%s: need B, H, T >= 1 and B*H <= 65535 (got %d, %d, %d)", fn, B, H, T);
    return LA_ERR_INVALID_ARG;
  }
  if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128)) {
    set_error("%s: dk and dv must be 64 or 128 (got %d, %d)", fn, dk, dv);
    return LA_ERR_UNSUPPORTED;
  }
  if (K < 1 || K > kMaxK) {
    set_error("%s: convolution length K must be 1..%d (got %d)", fn, kMaxK, K);
    return LA_ERR_INVALID_ARG;
  }
  if ((flags & ~(LA_PRO_L2NORM_Q | LA_PRO_L2NORM_K)) != 0) {
    set_error("%s: unknown flags 0x%x", fn, flags);
    return LA_ERR_INVALID_ARG;
  }
  if (gate_kind != LA_GATE_NONE && gate_kind != LA_GATE_LOGSIGMOID && gate_kind != LA_GATE_NEG_SOFTPLUS) {
    set_error("%s: unknown gate kind %d", fn, gate_kind);
    return LA_ERR_INVALID_ARG;
  }
  if (gate_kind != LA_GATE_NONE &&
      (!a_gate || !g || (gate_width != 1 && gate_width != dk) || !(tau > 0.f) || !(tau < 3.0e38f))) {
    set_error("%s: a gate needs a_gate, g, gate_width 1 or dk and a finite tau > 0", fn);
    return LA_ERR_INVALID_ARG;
  }
  if ((a_beta == nullptr) != (beta == nullptr)) {
    set_error("%s: a_beta and beta go together", fn);
    return LA_ERR_INVALID_ARG;
  }
  if (K > 1 && hist_out && hist_out == hist_in) {
    set_error("%s: hist_out must not alias hist_in", fn);
    return LA_ERR_INVALID_ARG;
  }
  const void *ptrs16[] = {xq, xk, xv, q, k, v, hist_in, hist_out};
  for (const void *ptr : ptrs16)
    if (ptr && !aligned16(ptr)) {
      set_error("%s: q/k/v pointers and the histories must be 16-byte aligned", fn);
      return LA_ERR_INVALID_ARG;
    }
  ProParams p{};
  p.x[0] = static_cast<const __nv_bfloat16 *>(xq);
  p.x[1] = static_cast<const __nv_bfloat16 *>(xk);
  p.x[2] = static_cast<const __nv_bfloat16 *>(xv);
  p.w[0] = wq;
  p.w[1] = wk;
  p.w[2] = wv;
  p.y[0] = static_cast<__nv_bfloat16 *>(q);
  p.y[1] = static_cast<__nv_bfloat16 *>(k);
  p.y[2] = static_cast<__nv_bfloat16 *>(v);
  p.hist_in = K > 1 ? static_cast<const __nv_bfloat16 *>(hist_in) : nullptr;
  p.hist_out = K > 1 ? static_cast<__nv_bfloat16 *>(hist_out) : nullptr;
  p.a_gate = a_gate;
  p.a_beta = a_beta;
  p.g = g;
  p.beta = beta;
  p.B = B;
  p.H = H;
  p.T = T;
  p.K = K;
  p.gate_kind = gate_kind;
  p.gate_width = gate_kind == LA_GATE_NONE ? 1 : gate_width;
  p.l2mask = flags;
  p.inv_tau = gate_kind == LA_GATE_NONE ? 1.f : 1.f / tau;
  p.wait_limit = kSpinLimit;
  p.skip_k_copy = 0;
  {
    // Failure-detection test hook, off unless the environment asks for it:
    // LA_TEST_FAULT=prologue_wait makes every CTA arm k's copy barrier without
    // starting the copy and give up after a short bounded wait, so the call
    // reports LA_ERR_TIMEOUT through la_stream_status without faulting.
    const char *f = getenv("LA_TEST_FAULT");
    if (f && strcmp(f, "prologue_wait") == 0) {
      p.skip_k_copy = 1;
      p.wait_limit = 4096;
    }
  }
  p.status = status_word();
  if (!p.status) {
    set_error("%s: no CUDA device available (%s)", fn, cudaGetErrorString(cudaGetLastError()));
    return LA_ERR_CUDA;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rc;
  if (dk == 128 && dv == 128) rc = launch_prologue<128, 128>(p, s);
  else if (dk == 128) rc = launch_prologue<128, 64>(p, s);
  else if (dv == 128) rc = launch_prologue<64, 128>(p, s);
  else rc = launch_prologue<64, 64>(p, s);
  if (rc != LA_OK) {
    set_error("%s: could not set the kernel's shared-memory size: %s", fn, cudaGetErrorString(cudaGetLastError()));
    return rc;
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("%s: launch failed: %s", fn, cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  return LA_OK;
}
