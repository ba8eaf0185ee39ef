// Chunkwise forward on CUDA cores in float32 (the LA_F32 path).
//
// One CTA owns one (b, h) and one tile of value columns, walks the sequence
// chunk by chunk ("Talk Linear Attention" section 3.2) and keeps its slice of
// the state S[dk][tile] in shared memory between chunks. Inside a chunk of
// n <= 64 tokens with inclusive log-gate prefix b_r (section 5.2):
//
//   P  = (Q K^T) ⊙ exp(b_r - b_s) ⊙ M           local, decay-masked scores
//   U  = V, or for the delta rule U = T (diag(beta) V - diag(beta e^b) K S)
//        with T = (I + A)^-1, A_rs = beta_r e^{b_r - b_s} k_r.k_s (s < r)
//        (the WY/UT form of the DeltaNet update, section 6.2)
//   O  = Diag(e^b) Q S + P U                    inter-chunk + local output
//   S <- Diag(e^{b_last}) S + (Diag(e^{b_last - b}) K)^T U
//
// GLA gates are per key channel; their exp(b_r - b_s) is factored around the
// chunk midpoint m as exp(b_r - b_m) exp(b_m - b_s) so that P stays a plain
// product. The elu+1 mode applies phi to q, k and carries the normaliser z as
// one extra state column whose value input is 1 (then o = num / den).
//
// All arithmetic is float32; this kernel is the float32-input path and is
// written for clarity over speed (the bf16 path runs on the tensor cores).
// With p.rev it runs the same recurrence over the stored sequence read from
// its end (token t is memory row T-1-t, for every input and the output): the
// anti-causal passes of the backward. Scalar data-dependent gates are then
// taken from the stored token after each position (index T - t, none at
// t = 0), the decay those passes need.
#include <cuda_bf16.h>

#include "la_internal.h"

namespace la {
namespace {

constexpr int kC = 64;          // chunk length of this kernel
constexpr int kThreads = 256;
constexpr int kMid = kC / 2 - 1;

template <typename T> __device__ __forceinline__ float ld_in(const T *p);
template <> __device__ __forceinline__ float ld_in<float>(const float *p) { return __ldg(p); }
template <> __device__ __forceinline__ float ld_in<__nv_bfloat16>(const __nv_bfloat16 *p) {
  return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ void st_out(T *p, float x);
template <> __device__ __forceinline__ void st_out<float>(float *p, float x) { *p = x; }
template <> __device__ __forceinline__ void st_out<__nv_bfloat16>(__nv_bfloat16 *p, float x) {
  *p = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float phi(float x) { return x > 0.f ? x + 1.f : __expf(x); }

struct SimtLayout {
  int pk;   // row pitch of Q, K (dk + 1, avoids bank conflicts)
  int pw;   // row pitch of V, S, R, U (W + 1)
  int pc;   // row pitch of P, A, Tm (C + 1)
  int offQ, offK, offV, offS, offP, offA, offT, offR, offU, offB, offVec, total;
};

__host__ __device__ inline SimtLayout simt_layout(int dk, int W, bool gla, bool delta) {
  SimtLayout L;
  L.pk = dk + 1;
  L.pw = W + 1;
  L.pc = kC + 1;
  int o = 0;
  L.offQ = o; o += kC * L.pk;
  L.offK = o; o += kC * L.pk;
  L.offV = o; o += kC * L.pw;
  L.offS = o; o += dk * L.pw;
  L.offP = o; o += kC * L.pc;
  L.offA = o; o += delta ? kC * L.pc : 0;
  L.offT = o; o += delta ? kC * L.pc : 0;
  L.offR = o; o += kC * L.pw;
  L.offU = o; o += delta ? kC * L.pw : 0;
  L.offB = o; o += gla ? kC * dk : kC;
  L.offVec = o; o += 3 * dk + kC;
  L.total = o;
  return L;
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads)
chunk_simt_kernel(const ChunkParams p, int tile_w) {
  extern __shared__ float sm[];
  const int tid = threadIdx.x;
  const int bh = blockIdx.x;
  const int h = bh % p.H;
  const int j0 = blockIdx.y * tile_w;
  const int dk = p.dk, dv = p.dv, T = p.T;
  const int kind = p.kind;
  const bool elu = kind == kElu1, gla = kind == kGla, delta = kind == kGdn;
  const int wv = min(tile_w, dv - j0);          // real value columns in this tile
  const int W = wv + (elu ? 1 : 0);             // + normaliser column
  const int Wfull = dv + (elu ? 1 : 0);          // state row length in memory
  const SimtLayout L = simt_layout(dk, tile_w + (elu ? 1 : 0), gla, delta);

  float *Q = sm + L.offQ, *K = sm + L.offK, *V = sm + L.offV, *S = sm + L.offS;
  float *P = sm + L.offP, *A = sm + L.offA, *Tm = sm + L.offT, *R = sm + L.offR;
  float *U = sm + L.offU, *Bg = sm + L.offB, *vec = sm + L.offVec;
  float *ebm = vec, *eblast = vec + dk, *elm = vec + 2 * dk, *bet = vec + 3 * dk;

  const Tin *q = static_cast<const Tin *>(p.q) + (size_t)bh * T * dk;
  const Tin *k = static_cast<const Tin *>(p.k) + (size_t)bh * T * dk;
  const Tin *v = static_cast<const Tin *>(p.v) + (size_t)bh * T * dv;
  Tin *o = static_cast<Tin *>(p.o) + (size_t)bh * T * dv;
  // memory row of token t: reversed runs walk the stored sequence from its end
  const auto row = [&](int t) { return (size_t)(p.rev ? T - 1 - t : t); };

  // Initial state slice.
  for (int i = tid; i < dk * W; i += kThreads) {
    const int c = i / W, j = i % W;
    float s = 0.f;
    if (p.S0) {
      const float *s0 = p.S0 + ((size_t)bh * dk + c) * Wfull;
      s = (j < wv) ? s0[j0 + j] : s0[dv];
    }
    S[c * L.pw + j] = s;
  }

  for (int t0 = 0; t0 < T; t0 += kC) {
    const int n = min(kC, T - t0);
    __syncthreads();
    // ---- stage the chunk (zero rows past the end of the sequence) ----
    for (int i = tid; i < kC * dk; i += kThreads) {
      const int r = i / dk, c = i % dk;
      float qv = 0.f, kv = 0.f;
      if (r < n) {
        qv = ld_in(q + row(t0 + r) * dk + c);
        kv = ld_in(k + row(t0 + r) * dk + c);
        if (elu) { qv = phi(qv); kv = phi(kv); }
      }
      Q[r * L.pk + c] = qv;
      K[r * L.pk + c] = kv;
    }
    for (int i = tid; i < kC * W; i += kThreads) {
      const int r = i / W, j = i % W;
      float x = 0.f;
      if (r < n) x = (j < wv) ? ld_in(v + row(t0 + r) * dv + j0 + j) : 1.f;
      V[r * L.pw + j] = x;
    }
    if (gla) {
      for (int i = tid; i < kC * dk; i += kThreads) {
        const int r = i / dk, c = i % dk;
        Bg[i] = (r < n) ? __ldg(p.g + ((size_t)bh * T + row(t0 + r)) * dk + c) : 0.f;
      }
    } else if (tid < kC) {
      const int r = tid;
      float lg = 0.f;
      if (r < n) {
        if (kind == kRetnet) lg = __ldg(p.g + h);
        else if (kind == kScalar && p.rev)  // reversed: the gate of the stored token after it
          lg = (t0 + r >= 1) ? __ldg(p.g + (size_t)bh * T + (T - t0 - r)) : 0.f;
        else if (kind == kScalar || (kind == kGdn && p.g)) lg = __ldg(p.g + (size_t)bh * T + row(t0 + r));
      }
      Bg[r] = lg;
      bet[r] = (r < n) ? (p.beta ? __ldg(p.beta + (size_t)bh * T + row(t0 + r)) : 1.f) : 0.f;
    }
    __syncthreads();
    // ---- inclusive log-gate prefix ----
    if (gla) {
      for (int c = tid; c < dk; c += kThreads) {
        float acc = 0.f;
        for (int r = 0; r < kC; ++r) { acc += Bg[r * dk + c]; Bg[r * dk + c] = acc; }
        ebm[c] = __expf(Bg[kMid * dk + c]);
        eblast[c] = __expf(acc);
        elm[c] = __expf(acc - Bg[kMid * dk + c]);
      }
    } else if (tid == 0) {
      float acc = 0.f;
      for (int r = 0; r < kC; ++r) { acc += Bg[r]; Bg[r] = acc; }
    }
    __syncthreads();
    if (gla) {  // Q <- Q e^{b - b_m}, K <- K e^{b_m - b}
      for (int i = tid; i < kC * dk; i += kThreads) {
        const int r = i / dk, c = i % dk;
        const float d = Bg[r * dk + c] - Bg[kMid * dk + c];
        Q[r * L.pk + c] *= __expf(d);
        K[r * L.pk + c] *= __expf(-d);
      }
      __syncthreads();
    }
    // ---- local scores P (and A for the delta rule) ----
    for (int i = tid; i < kC * kC; i += kThreads) {
      const int r = i / kC, s = i % kC;
      float pv = 0.f, av = 0.f;
      if (s <= r && r < n) {
        float dq = 0.f, dkk = 0.f;
        const float *qr = Q + r * L.pk, *kr = K + r * L.pk, *ks = K + s * L.pk;
        for (int c = 0; c < dk; ++c) {
          dq = fmaf(qr[c], ks[c], dq);
          if (delta) dkk = fmaf(kr[c], ks[c], dkk);
        }
        const float gam = gla ? 1.f : __expf(Bg[r] - Bg[s]);
        pv = dq * gam;
        if (delta && s < r) av = bet[r] * gam * dkk;
      }
      P[r * L.pc + s] = pv;
      if (delta) A[r * L.pc + s] = av;
    }
    __syncthreads();
    const float *Uc = V;
    if (delta) {
      // T = (I + A)^-1 by forward substitution, one column per thread.
      if (tid < kC) {
        const int j = tid;
        for (int r = 0; r < kC; ++r) {
          float acc = (r == j) ? 1.f : 0.f;
          for (int s = j; s < r; ++s) acc = fmaf(-A[r * L.pc + s], Tm[s * L.pc + j], acc);
          Tm[r * L.pc + j] = (r < j) ? 0.f : acc;
        }
      }
      // R = diag(beta) V - diag(beta e^b) K S
      for (int i = tid; i < kC * W; i += kThreads) {
        const int r = i / W, j = i % W;
        float ks = 0.f;
        const float *kr = K + r * L.pk;
        for (int c = 0; c < dk; ++c) ks = fmaf(kr[c], S[c * L.pw + j], ks);
        R[r * L.pw + j] = bet[r] * (V[r * L.pw + j] - __expf(Bg[r]) * ks);
      }
      __syncthreads();
      for (int i = tid; i < kC * W; i += kThreads) {
        const int r = i / W, j = i % W;
        float u = 0.f;
        for (int s = 0; s <= r; ++s) u = fmaf(Tm[r * L.pc + s], R[s * L.pw + j], u);
        U[r * L.pw + j] = u;
      }
      __syncthreads();
      Uc = U;
    }
    // ---- output O = Diag(e^b) Q S + P U (into R as scratch) ----
    float *O = R;
    for (int i = tid; i < kC * W; i += kThreads) {
      const int r = i / W, j = i % W;
      if (r >= n) continue;
      float inter = 0.f;
      const float *qr = Q + r * L.pk;
      if (gla) {
        for (int c = 0; c < dk; ++c) inter = fmaf(qr[c] * ebm[c], S[c * L.pw + j], inter);
      } else {
        for (int c = 0; c < dk; ++c) inter = fmaf(qr[c], S[c * L.pw + j], inter);
        inter *= __expf(Bg[r]);
      }
      float loc = 0.f;
      for (int s = 0; s <= r; ++s) loc = fmaf(P[r * L.pc + s], Uc[s * L.pw + j], loc);
      O[r * L.pw + j] = inter + loc;
    }
    __syncthreads();
    for (int i = tid; i < kC * wv; i += kThreads) {
      const int r = i / wv, j = i % wv;
      if (r >= n) continue;
      float x = O[r * L.pw + j];
      if (elu) x = x / O[r * L.pw + wv];
      st_out(o + row(t0 + r) * dv + j0 + j, x);
    }
    // ---- state passing ----
    for (int i = tid; i < dk * W; i += kThreads) {
      const int c = i / W, j = i % W;
      float acc = 0.f;
      for (int s = 0; s < kC; ++s) {
        float kx = K[s * L.pk + c];
        if (!gla) kx *= __expf(Bg[kC - 1] - Bg[s]);
        acc = fmaf(kx, Uc[s * L.pw + j], acc);
      }
      const float dec = gla ? eblast[c] : __expf(Bg[kC - 1]);
      const float scl = gla ? elm[c] : 1.f;
      S[c * L.pw + j] = fmaf(dec, S[c * L.pw + j], scl * acc);
    }
  }
  __syncthreads();
  if (p.S_final) {
    for (int i = tid; i < dk * W; i += kThreads) {
      const int c = i / W, j = i % W;
      float *sf = p.S_final + ((size_t)bh * dk + c) * Wfull;
      if (j < wv) sf[j0 + j] = S[c * L.pw + j];
      else if (blockIdx.y == 0) sf[dv] = S[c * L.pw + j];
    }
  }
}

}  // namespace

int launch_chunk_simt(const ChunkParams &p, cudaStream_t stream) {
  // elu+1 keeps every value column in one CTA so that the shared normaliser
  // column is read and written by a single CTA (S_final may alias S0).
  const int tile_w = (p.kind == kElu1) ? p.dv : 32;
  const int ntiles = (p.dv + tile_w - 1) / tile_w;
  const SimtLayout L = simt_layout(p.dk, tile_w + (p.kind == kElu1 ? 1 : 0), p.kind == kGla,
                                   p.kind == kGdn);
  const size_t smem = sizeof(float) * (size_t)L.total;
  if (smem > 227 * 1024) {
    set_error("la_chunk_fwd: float32 path needs %zu bytes of shared memory for dk=%d dv=%d",
              smem, p.dk, p.dv);
    return LA_ERR_UNSUPPORTED;
  }
  dim3 grid(p.B * p.H, ntiles);
  cudaError_t e;
  if (p.f32) {
    e = cudaFuncSetAttribute(chunk_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e == cudaSuccess) chunk_simt_kernel<float><<<grid, kThreads, smem, stream>>>(p, tile_w);
  } else {
    e = cudaFuncSetAttribute(chunk_simt_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
      chunk_simt_kernel<__nv_bfloat16><<<grid, kThreads, smem, stream>>>(p, tile_w);
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("la_chunk_fwd: float32-path launch failed: %s", cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  return LA_OK;
}

}  // namespace la
