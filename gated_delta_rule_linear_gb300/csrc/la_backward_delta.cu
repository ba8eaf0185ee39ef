// la_chunk_bwd_delta: the backward pass of the delta-rule forward (Gated
// DeltaNet: S_t = (I - beta_t k_t k_t^T) alpha_t S_{t-1} + beta_t k_t v_t^T,
// o_t = S_t^T q_t; "LLM attention optimisation" page, Gated DeltaNet section;
// "Talk Linear Attention" sections 6.2 and 4.1.2), chunkwise with C = 64.
//
// Per chunk with local prefix b_r of the log-gates (gamma_r = e^{b_r}, gL = the
// last one, Gamma_rs = e^{b_r - b_s}), entering state S and the gradient
// E = dL/dS at the chunk's end, the forward's WY form is
//
//   L = strict_lower(Gamma ⊙ K K^T),  T = (I + Diag(beta) L)^{-1}
//   Z = V - Diag(gamma) K S,  U = T Diag(beta) Z,  P = lower(Gamma ⊙ Q K^T)
//   O = Diag(gamma) Q S + P U,  S_next = gL S + Kt^T U,  Kt = Diag(gL / gamma) K
//
// and its reverse, read off line by line:
//
//   dU = Kt E + P^T dO,  Y = T^T dU,  dZ = Diag(beta) Y = dV
//   dbeta_r = Y_r . Z_r + sum_s dA_rs L_rs,  dA = -strict_lower(Y U^T)
//   dP = lower(dO U^T),  F = Diag(beta) dA ⊙ Gamma,  H = dP ⊙ Gamma
//   dQ = Diag(gamma) dO S^T + H K
//   dK = -Diag(gamma) dZ S^T + (gL / gamma) U E^T + F K + F^T K + H^T Q
//   db_r = gamma_r (dO_r . (S^T q_r) - dZ_r . (S^T k_r)) + row/column sums of
//          Diag(beta) dA ⊙ L and dP ⊙ P - (gL / gamma_r) k_r . (U E^T)_r,
//          plus gL <S, E> + sum_r (gL / gamma_r) k_r . (U E^T)_r at the last row
//   dg = the suffix sum of db inside the chunk
//   E_prev = gL E + Q^T Diag(gamma) dO - K^T Diag(gamma) dZ
//
// Four launches:
//   bd_pre_kernel   every chunk in parallel: L and P from one [Q; K] K^T
//                   product, T by substitution; T and P to the workspace.
//   bd_fwd_kernel   per (b, h) and 16 value columns, the chunks in order: S
//                   entering each chunk to the workspace.
//   bd_bwd_kernel   per (b, h) and 16 value columns, the chunks in reverse: E
//                   at each chunk's end to the workspace; dS0.
//   bd_grad_kernel  every chunk in parallel: the gradients above, the value
//                   axis in blocks of 16 with dQ, dK, dA and dP held in
//                   registers across the blocks.
// Products are warp-level tf32 MMAs (16 x 8 x 8, fp32 accumulate) on tiles in
// shared memory; bf16 inputs enter exactly (a bf16 is a tf32), fp32 operands
// are rounded to the nearest tf32. A tail chunk is padded with zero rows, zero
// gates and beta = 0, which leaves every real row's result unchanged.
#include <cuda_bf16.h>

#include <cstdint>

#include "la_internal.h"
#include "la_warp_mma.cuh"

namespace la {
namespace {

using namespace wm;

// Per-chunk scalars: gamma_r = e^{b_r}, e^{bL - b_r}, beta_r and b_r (b the
// inclusive prefix of the chunk's log-gates); rows past the end get zero gates
// and beta = 0. One warp: gate_loads issues the loads (two rows per lane),
// gate_scan forms the prefix when they are needed.
struct Scal {
  float gam[kCh], glr[kCh], bet[kCh], b[kCh];
};
struct Gates {
  float x0, x1, b0, b1;
};
__device__ __forceinline__ Gates gate_loads(const float *g, const float *beta, size_t base, int n, int lane) {
  Gates r{0.f, 0.f, 0.f, 0.f};
  if (g) {
    if (lane < n) r.x0 = __ldg(g + base + lane);
    if (lane + 32 < n) r.x1 = __ldg(g + base + lane + 32);
  }
  r.b0 = lane < n ? (beta ? __ldg(beta + base + lane) : 1.f) : 0.f;
  r.b1 = lane + 32 < n ? (beta ? __ldg(beta + base + lane + 32) : 1.f) : 0.f;
  return r;
}
__device__ __forceinline__ void gate_scan(Scal &s, Gates gt, int lane) {
  float x0 = gt.x0, x1 = gt.x1;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float a0 = __shfl_up_sync(0xffffffffu, x0, off), a1 = __shfl_up_sync(0xffffffffu, x1, off);
    if (lane >= off) {
      x0 += a0;
      x1 += a1;
    }
  }
  x1 += __shfl_sync(0xffffffffu, x0, 31);
  const float bl = __shfl_sync(0xffffffffu, x1, 31);
  s.b[lane] = x0;
  s.b[lane + 32] = x1;
  s.gam[lane] = __expf(x0);
  s.gam[lane + 32] = __expf(x1);
  s.glr[lane] = __expf(bl - x0);
  s.glr[lane + 32] = __expf(bl - x1);
  s.bet[lane] = gt.b0;
  s.bet[lane + 32] = gt.b1;
}

// ============================================================ pre-pass
template <int DK>
struct PreSmem {
  __nv_bfloat16 q[kCh * Pitch<DK>::h], k[kCh * Pitch<DK>::h];
  float a[kCh * kPf];
  Scal s;
};

template <int DK>
__global__ void __launch_bounds__(128) bd_pre_kernel(const __nv_bfloat16 *__restrict__ q,
                                                     const __nv_bfloat16 *__restrict__ k,
                                                     const float *__restrict__ g, const float *__restrict__ beta,
                                                     int T, float *__restrict__ Tw, float *__restrict__ Pw,
                                                     __nv_bfloat16 *__restrict__ Tb, __nv_bfloat16 *__restrict__ Pb) {
  constexpr int PH = Pitch<DK>::h;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  PreSmem<DK> &sm = *reinterpret_cast<PreSmem<DK> *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = blockIdx.x, bh = blockIdx.y, nch = gridDim.x;
  const int t0 = i * kCh, n = min(kCh, T - t0);
  const size_t row0 = (size_t)bh * T + t0;
  rows_async<DK, PH>(sm.q, q + row0 * DK, n, tid, 128);
  rows_async<DK, PH>(sm.k, k + row0 * DK, n, tid, 128);
  cp_commit();
  if (warp == 0) gate_scan(sm.s, gate_loads(g, beta, row0, n, lane), lane);
  cp_wait<0>();
  __syncthreads();
  // [Q; K] K^T: warps 0, 1 the rows of Q (P), warps 2, 3 the rows of K (A)
  const __nv_bfloat16 *src = warp < 2 ? sm.q : sm.k;
  const int rbase = (warp & 1) * 32;
  float acc[2][8][4];
  const size_t cbase = ((size_t)bh * nch + i) * kCh * kCh;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    zero(acc[h]);
    wmma(acc[h], rbase + 16 * h, 0, DK, [&](int m, int kk) { return bfbits(src + m * PH + kk); },
         [&](int kk, int nn) { return bfbits(sm.k + nn * PH + kk); }, lane);
    if (warp < 2) {
      each(acc[h], rbase + 16 * h, 0, lane, [&](int r, int s, float &v) {
        const float x = s <= r ? __expf(sm.s.b[r] - sm.s.b[s]) * v : 0.f;
        Pw[cbase + r * kCh + s] = x;
        Pb[cbase + r * kCh + s] = __float2bfloat16_rn(x);
      });
    } else {
      each(acc[h], rbase + 16 * h, 0, lane, [&](int r, int s, float &v) {
        cc(sm.a, r, s) = s < r ? sm.s.bet[r] * __expf(sm.s.b[r] - sm.s.b[s]) * v : 0.f;
      });
    }
  }
  __syncthreads();
  // T = (I + A)^{-1}, unit lower triangular: column j by forward substitution, in registers
  if (tid < kCh) {
    const int j = tid;
    float tc[kCh];
#pragma unroll
    for (int r = 0; r < kCh; ++r) {
      // four partial sums, so the row's FMAs do not form one dependent chain
      float x[4] = {r == j ? 1.f : 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < r; ++s) x[s & 3] = fmaf(-cc(sm.a, r, s), tc[s], x[s & 3]);
      tc[r] = r < j ? 0.f : (x[0] + x[1]) + (x[2] + x[3]);
    }
#pragma unroll
    for (int r = 0; r < kCh; ++r) {
      Tw[cbase + r * kCh + j] = tc[r];
      Tb[cbase + r * kCh + j] = __float2bfloat16_rn(tc[r]);
    }
  }
}

// ============================================================ state chains
// Both chains run per (b, h) and 64 value columns on eight warps (warp w: token
// rows 16 (w % 4) of the chunk products, value columns 32 (w / 4) .. + 31), the
// state (or its gradient) in fp32 registers with a bf16 copy of its transpose
// as an MMA operand; bf16 m16n8k16 warp MMAs, the token-major operands through
// ldmatrix.trans; two tile buffers, so that the next chunk's copies run during
// the whole current one.
constexpr int kBW = 64;        // value columns per chain CTA
constexpr int kBP = kBW + 8;   // row pitch (bf16) of the chains' [64][64] tiles

// a [64][64] bf16 image (dense rows) into a tile of pitch kBP
__device__ __forceinline__ void img_async(__nv_bfloat16 *dst, const __nv_bfloat16 *src, int tid) {
  for (int e = tid; e < kCh * 8; e += 256) cpa16(dst + (e >> 3) * kBP + (e & 7) * 8, src + e * 8, true);
}
// value columns [c0, c0 + 64) of a [T][DV] bf16 tensor from the chunk's first token (n valid rows)
template <int DV>
__device__ __forceinline__ void vcols_async(__nv_bfloat16 *dst, const __nv_bfloat16 *src, int c0, int n, int tid) {
  for (int e = tid; e < kCh * 8; e += 256) {
    const int r = e >> 3, c = (e & 7) * 8;
    const bool ok = r < n;
    cpa16(dst + r * kBP + c, src + (ok ? (size_t)r * DV + c0 + c : 0), ok);
  }
}
// the thread's share of a state tile set (rows 16 (rh + 4 rt), columns n0 ..): fp32 to
// the image (row-major [DK][DV]) and its bf16 transpose (value column, key channel)
template <int DK, int DV, int RT>
__device__ __forceinline__ void state_out(const float (&X)[RT][4][4], float *img, __nv_bfloat16 *xt, int rh,
                                          int n0, int c0, int lane) {
  constexpr int PH = Pitch<DK>::h;
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int rt = 0; rt < RT; ++rt) {
    const int m0 = 16 * (rh + 4 * rt);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = n0 + 8 * j + 2 * t, r = m0 + g;
      *reinterpret_cast<float2 *>(img + (size_t)r * DV + c0 + c) = make_float2(X[rt][j][0], X[rt][j][1]);
      *reinterpret_cast<float2 *>(img + (size_t)(r + 8) * DV + c0 + c) = make_float2(X[rt][j][2], X[rt][j][3]);
      xt[c * PH + r] = __float2bfloat16_rn(X[rt][j][0]);
      xt[(c + 1) * PH + r] = __float2bfloat16_rn(X[rt][j][1]);
      xt[c * PH + r + 8] = __float2bfloat16_rn(X[rt][j][2]);
      xt[(c + 1) * PH + r + 8] = __float2bfloat16_rn(X[rt][j][3]);
    }
  }
}
// rows 16 rh, columns n0 .. n0 + 31 of a product, scaled per row, as bf16 into a [64][kBP] tile
template <class F>
__device__ __forceinline__ void tile_out(const float (&a)[4][4], __nv_bfloat16 *dst, int rh, int n0, int lane, F f) {
  const int g = lane >> 2, t = lane & 3, r = 16 * rh + g;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = n0 + 8 * j + 2 * t;
    *reinterpret_cast<__nv_bfloat162 *>(dst + r * kBP + c) =
        __floats2bfloat162_rn(f(r, c, a[j][0]), f(r, c + 1, a[j][1]));
    *reinterpret_cast<__nv_bfloat162 *>(dst + (r + 8) * kBP + c) =
        __floats2bfloat162_rn(f(r + 8, c, a[j][2]), f(r + 8, c + 1, a[j][3]));
  }
}

// ---- forward state chain: S entering each chunk to the workspace. KDA = true
// (Kimi Delta Attention): k is the pre-pass's image of K e^B (so the gates of
// the Gated DeltaNet form are absent: g = NULL), k2 its image of K e^{B_L - B}
// for the state update, and the decay e^{B_L} acts per key channel.
template <int DK, bool KDA>
struct FwdTiles {
  __nv_bfloat16 k[kCh * Pitch<DK>::h], v[kCh * kBP], t[kCh * kBP];
  __nv_bfloat16 k2[KDA ? kCh * Pitch<DK>::h : 8];
  float gl[KDA ? DK : 4];
};
template <int DK, bool KDA>
struct FwdSmem {
  FwdTiles<DK, KDA> x[2];
  __nv_bfloat16 st[kBW * Pitch<DK>::h], z[kCh * kBP], u[kCh * kBP];
  Scal sc[2];
};

// the per-chunk images of the KDA pre-pass: [BH][nch][64][DK] bf16 and [BH][nch][DK] e^{B_L}
struct KdaImages {
  const __nv_bfloat16 *kh, *kt, *qh;
  const float *gl;
};

template <int DK, int DV, bool KDA>
__global__ void __launch_bounds__(256) bd_fwd_kernel(const __nv_bfloat16 *__restrict__ k,
                                                     const __nv_bfloat16 *__restrict__ v,
                                                     const float *__restrict__ g, const float *__restrict__ beta,
                                                     const float *__restrict__ S0, int T,
                                                     const __nv_bfloat16 *__restrict__ Tb, float *__restrict__ Sin,
                                                     KdaImages img) {
  constexpr int PH = Pitch<DK>::h, NCB = DV / kBW, RT = DK / 64;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  FwdSmem<DK, KDA> &sm = *reinterpret_cast<FwdSmem<DK, KDA> *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rh = warp & 3, n0 = (warp >> 2) * 32;
  const int bh = blockIdx.x / NCB, c0 = (blockIdx.x % NCB) * kBW;
  const int nch = (T + kCh - 1) / kCh;
  auto issue = [&](int i, FwdTiles<DK, KDA> &x) {
    const int t0 = i * kCh, n = min(kCh, T - t0);
    const size_t row0 = (size_t)bh * T + t0, ci = (size_t)bh * nch + i;
    if constexpr (KDA) {
      rows_async<DK, PH>(x.k, img.kh + ci * kCh * DK, kCh, tid, 256);
      rows_async<DK, PH>(x.k2, img.kt + ci * kCh * DK, kCh, tid, 256);
      for (int e = tid; e < DK / 4; e += 256) cpa16(x.gl + 4 * e, img.gl + ci * DK + 4 * e, true);
    } else {
      rows_async<DK, PH>(x.k, k + row0 * DK, n, tid, 256);
    }
    vcols_async<DV>(x.v, v + row0 * DV, c0, n, tid);
    img_async(x.t, Tb + ((size_t)bh * nch + i) * kCh * kCh, tid);
    cp_commit();
  };
  auto gates = [&](int i) { return gate_loads(g, beta, (size_t)bh * T + i * kCh, min(kCh, T - i * kCh), lane); };
  float S[RT][4][4];
#pragma unroll
  for (int rt = 0; rt < RT; ++rt) {
    zero(S[rt]);
    if (S0)
      each(S[rt], 16 * (rh + 4 * rt), n0, lane,
           [&](int r, int c, float &x) { x = __ldg(S0 + ((size_t)bh * DK + r) * DV + c0 + c); });
  }
  issue(0, sm.x[0]);
  if (warp == 0) gate_scan(sm.sc[0], gates(0), lane);
  for (int i = 0; i < nch; ++i) {
    const FwdTiles<DK, KDA> &x = sm.x[i & 1];
    const Scal &sc = sm.sc[i & 1];
    const bool more = i + 1 < nch;
    Gates nxt{};
    if (more) {
      issue(i + 1, sm.x[(i + 1) & 1]);
      if (warp == 0) nxt = gates(i + 1);
    }
    state_out<DK, DV>(S, Sin + ((size_t)bh * nch + i) * DK * DV, sm.st, rh, n0, c0, lane);
    if (more)
      cp_wait<1>();
    else
      cp_wait<0>();
    __syncthreads();
    // Z' = Diag(beta) (V - Diag(gamma) K S)
    {
      float a[4][4];
      zero(a);
      wmma16(a, 16 * rh, n0, DK, x.k, PH, sm.st, PH, lane);
      tile_out(a, sm.z, rh, n0, lane,
               [&](int r, int c, float y) { return sc.bet[r] * (bf(x.v + r * kBP + c) - sc.gam[r] * y); });
    }
    __syncthreads();
    // U' = Diag(gL / gamma) T Z'
    {
      float a[4][4];
      zero(a);
      wmma16_bt(a, 16 * rh, n0, kCh, x.t, kBP, sm.z, kBP, lane);
      tile_out(a, sm.u, rh, n0, lane, [&](int r, int, float y) { return sc.glr[r] * y; });
    }
    __syncthreads();
    // S <- gL S + K^T U' (KDA: Diag(e^{B_L}) S + (K e^{B_L - B})^T U')
    const float gL = sc.gam[kCh - 1];
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
      const int m0 = 16 * (rh + 4 * rt);
      if constexpr (KDA) {
        each(S[rt], m0, n0, lane, [&](int r, int, float &y) { y *= x.gl[r]; });
        wmma16_atbt(S[rt], m0, n0, kCh, x.k2, PH, sm.u, kBP, lane);
      } else {
        each(S[rt], 0, 0, lane, [&](int, int, float &y) { y *= gL; });
        wmma16_atbt(S[rt], m0, n0, kCh, x.k, PH, sm.u, kBP, lane);
      }
    }
    if (warp == 0 && more) gate_scan(sm.sc[(i + 1) & 1], nxt, lane);
    __syncthreads();
  }
}

// ---- reverse chain of E = dL/dS at each chunk's end; dS0. KDA = true: q is the
// image of Q e^B, k that of K e^{B_L - B} (read by dU), k2 that of K e^B (the
// state-gradient update), the decay e^{B_L} per key channel, g = NULL.
template <int DK, bool KDA>
struct BwdTiles {
  __nv_bfloat16 q[kCh * Pitch<DK>::h], k[kCh * Pitch<DK>::h], o[kCh * kBP], t[kCh * kBP], p[kCh * kBP];
  __nv_bfloat16 k2[KDA ? kCh * Pitch<DK>::h : 8];
  float gl[KDA ? DK : 4];
};
template <int DK, bool KDA>
struct BwdSmem {
  BwdTiles<DK, KDA> x[2];
  __nv_bfloat16 et[kBW * Pitch<DK>::h], og[kCh * kBP], du[kCh * kBP], y[kCh * kBP];
  Scal sc[2];
};

template <int DK, int DV, bool KDA>
__global__ void __launch_bounds__(256) bd_bwd_kernel(const __nv_bfloat16 *__restrict__ q,
                                                     const __nv_bfloat16 *__restrict__ k,
                                                     const __nv_bfloat16 *__restrict__ dO,
                                                     const float *__restrict__ g, const float *__restrict__ beta,
                                                     const float *__restrict__ dS, int T,
                                                     const __nv_bfloat16 *__restrict__ Tb,
                                                     const __nv_bfloat16 *__restrict__ Pb, float *__restrict__ Eout,
                                                     float *__restrict__ dS0, KdaImages img) {
  constexpr int PH = Pitch<DK>::h, NCB = DV / kBW, RT = DK / 64;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  BwdSmem<DK, KDA> &sm = *reinterpret_cast<BwdSmem<DK, KDA> *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rh = warp & 3, n0 = (warp >> 2) * 32;
  const int bh = blockIdx.x / NCB, c0 = (blockIdx.x % NCB) * kBW;
  const int nch = (T + kCh - 1) / kCh;
  auto issue = [&](int i, BwdTiles<DK, KDA> &x) {
    const int t0 = i * kCh, n = min(kCh, T - t0);
    const size_t row0 = (size_t)bh * T + t0, ci = (size_t)bh * nch + i, cb = ci * kCh * kCh;
    if constexpr (KDA) {
      rows_async<DK, PH>(x.q, img.qh + ci * kCh * DK, kCh, tid, 256);
      rows_async<DK, PH>(x.k, img.kt + ci * kCh * DK, kCh, tid, 256);
      rows_async<DK, PH>(x.k2, img.kh + ci * kCh * DK, kCh, tid, 256);
      for (int e = tid; e < DK / 4; e += 256) cpa16(x.gl + 4 * e, img.gl + ci * DK + 4 * e, true);
    } else {
      rows_async<DK, PH>(x.q, q + row0 * DK, n, tid, 256);
      rows_async<DK, PH>(x.k, k + row0 * DK, n, tid, 256);
    }
    vcols_async<DV>(x.o, dO + row0 * DV, c0, n, tid);
    img_async(x.t, Tb + cb, tid);
    img_async(x.p, Pb + cb, tid);
    cp_commit();
  };
  auto gates = [&](int i) { return gate_loads(g, beta, (size_t)bh * T + i * kCh, min(kCh, T - i * kCh), lane); };
  float E[RT][4][4];
#pragma unroll
  for (int rt = 0; rt < RT; ++rt) {
    zero(E[rt]);
    if (dS)
      each(E[rt], 16 * (rh + 4 * rt), n0, lane,
           [&](int r, int c, float &x) { x = __ldg(dS + ((size_t)bh * DK + r) * DV + c0 + c); });
  }
  issue(nch - 1, sm.x[(nch - 1) & 1]);
  if (warp == 0) gate_scan(sm.sc[(nch - 1) & 1], gates(nch - 1), lane);
  for (int i = nch - 1; i >= 0; --i) {
    const BwdTiles<DK, KDA> &x = sm.x[i & 1];
    const Scal &sc = sm.sc[i & 1];
    const bool more = i > 0;
    Gates nxt{};
    if (more) {
      issue(i - 1, sm.x[(i - 1) & 1]);
      if (warp == 0) nxt = gates(i - 1);
    }
    state_out<DK, DV>(E, Eout + ((size_t)bh * nch + i) * DK * DV, sm.et, rh, n0, c0, lane);
    if (more)
      cp_wait<1>();
    else
      cp_wait<0>();
    __syncthreads();
    // Diag(gamma) dO for the state update (thread: a row, eight columns)
    {
      const int r = tid >> 2, cq = (tid & 3) * 16;
      const float gm = sc.gam[r];
#pragma unroll
      for (int e = 0; e < 16; e += 2) {
        const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(x.o + r * kBP + cq + e);
        *reinterpret_cast<__nv_bfloat162 *>(sm.og + r * kBP + cq + e) =
            __floats2bfloat162_rn(gm * __low2float(h), gm * __high2float(h));
      }
    }
    // dU = Diag(gL / gamma) K E + P^T dO
    {
      float a[4][4];
      zero(a);
      wmma16(a, 16 * rh, n0, DK, x.k, PH, sm.et, PH, lane);
      each(a, 16 * rh, n0, lane, [&](int r, int, float &y) { y *= sc.glr[r]; });
      wmma16_atbt(a, 16 * rh, n0, kCh, x.p, kBP, x.o, kBP, lane);
      tile_out(a, sm.du, rh, n0, lane, [&](int, int, float y) { return y; });
    }
    __syncthreads();
    // -Diag(gamma) dZ = -Diag(gamma beta) T^T dU
    {
      float a[4][4];
      zero(a);
      wmma16_atbt(a, 16 * rh, n0, kCh, x.t, kBP, sm.du, kBP, lane);
      tile_out(a, sm.y, rh, n0, lane, [&](int r, int, float y) { return -sc.gam[r] * sc.bet[r] * y; });
    }
    __syncthreads();
    // E <- gL E + Q^T Diag(gamma) dO - K^T Diag(gamma) dZ
    //   (KDA: Diag(e^{B_L}) E + (Q e^B)^T dO - (K e^B)^T dZ)
    const float gL = sc.gam[kCh - 1];
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
      const int m0 = 16 * (rh + 4 * rt);
      if constexpr (KDA)
        each(E[rt], m0, n0, lane, [&](int r, int, float &y) { y *= x.gl[r]; });
      else
        each(E[rt], 0, 0, lane, [&](int, int, float &y) { y *= gL; });
      wmma16_atbt(E[rt], m0, n0, kCh, x.q, PH, sm.og, kBP, lane);
      wmma16_atbt(E[rt], m0, n0, kCh, KDA ? x.k2 : x.k, PH, sm.y, kBP, lane);
    }
    if (warp == 0 && more) gate_scan(sm.sc[(i - 1) & 1], nxt, lane);
    __syncthreads();
  }
  if (dS0) {
#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
      each(E[rt], 16 * (rh + 4 * rt), n0, lane,
           [&](int r, int c, float &x) { dS0[((size_t)bh * DK + r) * DV + c0 + c] = x; });
  }
}

// ============================================================ gradients
// One CTA per chunk; the value axis in blocks of kGW = 32 columns (warp w: token
// rows 16 (w % 4), block columns 16 (w / 4) .. + 15 of the block products),
// double-buffered: the next block's S, E (float32) and v, dO columns land while
// this one computes.
constexpr int kGW = 32;       // value columns per gradient block
constexpr int kGP = kGW + 8;  // row pitch (bf16) of the block's v and dO tiles: 80-byte rows
// element (r, c) of a float32 x 32 tile (16-byte groups XOR-permuted by row)
__device__ __forceinline__ float &w32(float *p, int r, int c) { return fw<kGW>(p, r, c); }
// the D x 32 columns [c0, c0 + 32) of a [D][DV] float32 matrix into a w32 tile
template <int D, int DV>
__device__ __forceinline__ void state32_async(float *dst, const float *src, int c0, int tid) {
  for (int i = tid; i < D * 8; i += 256) {
    const int r = i >> 3, c = (i & 7) * 4;
    cpa16(dst + r * kGW + (c ^ swz64(r)), src + (size_t)r * DV + c0 + c, true);
  }
}
// the 64 x 32 columns [c0, c0 + 32) of a [T][DV] bf16 tensor (n valid rows), pitch kGP
template <int DV>
__device__ __forceinline__ void cols32_async(__nv_bfloat16 *dst, const __nv_bfloat16 *src, int c0, int n, int tid) {
  for (int i = tid; i < kCh * 4; i += 256) {
    const int r = i >> 2, c = (i & 3) * 8;
    const bool ok = r < n;
    cpa16(dst + r * kGP + c, src + (ok ? (size_t)r * DV + c0 + c : 0), ok);
  }
}

template <int DK>
struct GradBlk {
  float s[DK * kGW], e[DK * kGW];
  __nv_bfloat16 v[kCh * kGP], o[kCh * kGP];
};
template <int DK>
struct GradSmem {
  __nv_bfloat16 q[kCh * Pitch<DK>::h], k[kCh * Pitch<DK>::h];
  float t[kCh * kPf], p[kCh * kPf];
  union {
    struct {
      GradBlk<DK> b[2];
      float ks[kCh * kGW], qs[kCh * kGW], ke[kCh * kGW], z[kCh * kGW], u[kCh * kGW], du[kCh * kGW],
          y[kCh * kGW];
    } blk;
    struct {  // after the blocks: dA (then F), dP (then H), L
      float da[kCh * kPf], dp[kCh * kPf], l[kCh * kPf];
    } fin;
  } w;
  Scal sc;
  float db[kCh], dbeta[kCh], kd[kCh], red[8];
};

// acc_a += A B1, acc_b += A B2 with one A fragment per k step (NT 16 x 8 tiles each)
template <int NT, class GA, class GB1, class GB2>
__device__ __forceinline__ void wmma2(float (&acc_a)[NT][4], float (&acc_b)[NT][4], int m0, int n0, int K, GA ga,
                                      GB1 gb1, GB2 gb2, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int k0 = 0; k0 < K; k0 += 8) {
    uint32_t a[4] = {ga(m0 + g, k0 + t), ga(m0 + g + 8, k0 + t), ga(m0 + g, k0 + t + 4),
                     ga(m0 + g + 8, k0 + t + 4)};
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      uint32_t b1[2] = {gb1(k0 + t, n0 + 8 * j + g), gb1(k0 + t + 4, n0 + 8 * j + g)};
      uint32_t b2[2] = {gb2(k0 + t, n0 + 8 * j + g), gb2(k0 + t + 4, n0 + 8 * j + g)};
      mma_16x8x8_tf32(acc_a[j], a, b1);
      mma_16x8x8_tf32(acc_b[j], a, b2);
    }
  }
}

template <int DK, int DV>
__global__ void __launch_bounds__(256, 1) bd_grad_kernel(
    const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
    const __nv_bfloat16 *__restrict__ dO, const float *__restrict__ g, const float *__restrict__ beta, int T,
    const float *__restrict__ Tw, const float *__restrict__ Pw, const float *__restrict__ Sin,
    const float *__restrict__ Eout, __nv_bfloat16 *__restrict__ dq, __nv_bfloat16 *__restrict__ dk,
    __nv_bfloat16 *__restrict__ dv, float *__restrict__ dbeta, float *__restrict__ dg) {
  constexpr int PH = Pitch<DK>::h, NT = DK / 16;  // 16 x 8 tiles per warp across dQ, dK (DK / 2 columns)
  extern __shared__ __align__(16) uint8_t smem_raw[];
  GradSmem<DK> &sm = *reinterpret_cast<GradSmem<DK> *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = blockIdx.x, bh = blockIdx.y, nch = gridDim.x;
  const int t0 = i * kCh, n = min(kCh, T - t0);
  const size_t row0 = (size_t)bh * T + t0;
  const size_t cbase = ((size_t)bh * nch + i) * kCh * kCh, sbase = ((size_t)bh * nch + i) * DK * DV;
  auto& W = sm.w.blk;
  auto issue_blk = [&](int c0, GradBlk<DK> &b) {
    state32_async<DK, DV>(b.s, Sin + sbase, c0, tid);
    state32_async<DK, DV>(b.e, Eout + sbase, c0, tid);
    cols32_async<DV>(b.v, v + row0 * DV, c0, n, tid);
    cols32_async<DV>(b.o, dO + row0 * DV, c0, n, tid);
  };
  rows_async<DK, PH>(sm.q, q + row0 * DK, n, tid, 256);
  rows_async<DK, PH>(sm.k, k + row0 * DK, n, tid, 256);
  cc_async(sm.t, Tw + cbase, tid, 256);
  cc_async(sm.p, Pw + cbase, tid, 256);
  issue_blk(0, W.b[0]);
  cp_commit();
  if (warp == 0) gate_scan(sm.sc, gate_loads(g, beta, row0, n, lane), lane);
  if (tid < kCh) {
    sm.db[tid] = 0.f;
    sm.dbeta[tid] = 0.f;
    sm.kd[tid] = 0.f;
  }
  // register accumulators: dQ, dK (rows 16 (w & 3), columns (w >> 2) DK / 2 ..), dA, dP (columns (w >> 2) 32 ..)
  const int mr = 16 * (warp & 3), half = warp >> 2;
  const int nq = half * (DK / 2), na = half * 32;
  float aq[NT][4], ak[NT][4], aa[4][4], ap[4][4];
  zero(aq);
  zero(ak);
  zero(aa);
  zero(ap);
  float se = 0.f;  // <S, E> over this thread's share
  const int nc = 16 * half;  // block products: warp w owns rows 16 (w & 3), columns 16 (w >> 2) .. + 16
  for (int c0 = 0, cb = 0; c0 < DV; c0 += kGW, ++cb) {
    GradBlk<DK> &B = W.b[cb & 1];
    if (c0 + kGW < DV) {
      issue_blk(c0 + kGW, W.b[(cb + 1) & 1]);
      cp_commit();
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    for (int x = tid; x < DK * kGW; x += 256) se += w32(B.s, x >> 5, x & 31) * w32(B.e, x >> 5, x & 31);
    // ---- K S and Diag(gL / gamma) K E (one A fragment), Q S: two 16 x 8 tiles each per warp
    {
      float a[2][4], b[2][4], c[2][4];
      zero(a);
      zero(b);
      zero(c);
      wmma2(a, c, mr, nc, DK, [&](int m, int kk) { return bfbits(sm.k + m * PH + kk); },
            [&](int kk, int nn) { return tf(w32(B.s, kk, nn)); },
            [&](int kk, int nn) { return tf(w32(B.e, kk, nn)); }, lane);
      wmma(b, mr, nc, DK, [&](int m, int kk) { return bfbits(sm.q + m * PH + kk); },
           [&](int kk, int nn) { return tf(w32(B.s, kk, nn)); }, lane);
      each(a, mr, nc, lane, [&](int r, int col, float &x) { w32(W.ks, r, col) = x; });
      each(b, mr, nc, lane, [&](int r, int col, float &x) { w32(W.qs, r, col) = x; });
      each(c, mr, nc, lane, [&](int r, int col, float &x) { w32(W.ke, r, col) = sm.sc.glr[r] * x; });
    }
    __syncthreads();
    // ---- Z = V - Diag(gamma) K S; db += gamma dO . (Q S)  (thread: a row, eight columns)
    {
      const int r = tid >> 2, cq = (tid & 3) * 8;
      float part = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int c = cq + e;
        w32(W.z, r, c) = bf(B.v + r * kGP + c) - sm.sc.gam[r] * w32(W.ks, r, c);
        part += bf(B.o + r * kGP + c) * w32(W.qs, r, c);
      }
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      if ((tid & 3) == 0) sm.db[r] += sm.sc.gam[r] * part;
    }
    __syncthreads();
    // ---- U = T Diag(beta) Z; dU = Diag(gL / gamma) K E + P^T dO
    {
      float a[2][4], b[2][4];
      zero(a);
      wmma(a, mr, nc, kCh, [&](int m, int kk) { return tf(cc(sm.t, m, kk)); },
           [&](int kk, int nn) { return tf(sm.sc.bet[kk] * w32(W.z, kk, nn)); }, lane);
      each(a, mr, nc, lane, [&](int r, int col, float &x) { w32(W.u, r, col) = x; });
      each(b, mr, nc, lane, [&](int r, int col, float &x) { x = w32(W.ke, r, col); });
      wmma(b, mr, nc, kCh, [&](int m, int kk) { return tf(cc(sm.p, kk, m)); },
           [&](int kk, int nn) { return bfbits(B.o + kk * kGP + nn); }, lane);
      each(b, mr, nc, lane, [&](int r, int col, float &x) { w32(W.du, r, col) = x; });
    }
    __syncthreads();
    // ---- Y = T^T dU; dV = Diag(beta) Y; dbeta += Y . Z; db -= gamma dZ . (K S); kd += U . (Kt E)
    {
      float a[2][4];
      zero(a);
      wmma(a, mr, nc, kCh, [&](int m, int kk) { return tf(cc(sm.t, kk, m)); },
           [&](int kk, int nn) { return tf(w32(W.du, kk, nn)); }, lane);
      const int gg = lane >> 2;
      float pb[2] = {0.f, 0.f}, pd[2] = {0.f, 0.f}, pk[2] = {0.f, 0.f};
      each(a, mr, nc, lane, [&](int r, int col, float &y) {
        const int h = (r - mr - gg) >> 3;  // 0: row g, 1: row g + 8
        w32(W.y, r, col) = y;
        const float dz = sm.sc.bet[r] * y;
        if (r < n) dv[(row0 + r) * DV + c0 + col] = __float2bfloat16_rn(dz);
        pb[h] += y * w32(W.z, r, col);
        pd[h] += dz * w32(W.ks, r, col);
        pk[h] += w32(W.u, r, col) * w32(W.ke, r, col);
      });
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
          pb[h] += __shfl_xor_sync(0xffffffffu, pb[h], off);
          pd[h] += __shfl_xor_sync(0xffffffffu, pd[h], off);
          pk[h] += __shfl_xor_sync(0xffffffffu, pk[h], off);
        }
        if ((lane & 3) == 0) {
          const int r = mr + gg + 8 * h;
          atomicAdd(&sm.dbeta[r], pb[h]);
          atomicAdd(&sm.db[r], -sm.sc.gam[r] * pd[h]);
          atomicAdd(&sm.kd[r], pk[h]);
        }
      }
    }
    __syncthreads();
    // ---- dA -= Y U^T, dP += dO U^T, dQ += Diag(gamma) dO S^T,
    //      dK += -Diag(gamma beta) Y S^T + Diag(gL / gamma) U E^T (K = 32 each)
    wmma(aa, mr, na, kGW, [&](int m, int kk) { return tf(-w32(W.y, m, kk)); },
         [&](int kk, int nn) { return tf(w32(W.u, nn, kk)); }, lane);
    wmma(ap, mr, na, kGW, [&](int m, int kk) { return bfbits(B.o + m * kGP + kk); },
         [&](int kk, int nn) { return tf(w32(W.u, nn, kk)); }, lane);
    wmma(aq, mr, nq, kGW, [&](int m, int kk) { return tf(sm.sc.gam[m] * bf(B.o + m * kGP + kk)); },
         [&](int kk, int nn) { return tf(w32(B.s, nn, kk)); }, lane);
    wmma(ak, mr, nq, kGW, [&](int m, int kk) { return tf(-sm.sc.gam[m] * sm.sc.bet[m] * w32(W.y, m, kk)); },
         [&](int kk, int nn) { return tf(w32(B.s, nn, kk)); }, lane);
    wmma(ak, mr, nq, kGW, [&](int m, int kk) { return tf(sm.sc.glr[m] * w32(W.u, m, kk)); },
         [&](int kk, int nn) { return tf(w32(B.e, nn, kk)); }, lane);
    __syncthreads();
  }
  // ---- <S, E> over the block
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) se += __shfl_xor_sync(0xffffffffu, se, off);
  if (lane == 0) sm.red[warp] = se;
  // ---- dA, dP to shared memory; L = strict_lower(Gamma ⊙ K K^T)
  auto& Fn = sm.w.fin;
  each(aa, mr, na, lane, [&](int r, int s, float &x) { cc(Fn.da, r, s) = x; });
  each(ap, mr, na, lane, [&](int r, int s, float &x) { cc(Fn.dp, r, s) = x; });
  {
    float a[4][4];
    zero(a);
    wmma(a, mr, na, DK, [&](int m, int kk) { return bfbits(sm.k + m * PH + kk); },
         [&](int kk, int nn) { return bfbits(sm.k + nn * PH + kk); }, lane);
    each(a, mr, na, lane, [&](int r, int s, float &x) {
      cc(Fn.l, r, s) = s < r ? __expf(sm.sc.b[r] - sm.sc.b[s]) * x : 0.f;
    });
  }
  __syncthreads();
  // ---- F = Diag(beta) dA ⊙ Gamma, H = dP ⊙ Gamma (in place); dbeta and the row / column sums of db
  {
    const int r = tid >> 2;
    float rowp = 0.f, betp = 0.f;
    for (int jj = 0; jj < kCh / 4; ++jj) {
      const int s = (tid & 3) + 4 * jj;
      const float gm = s <= r ? __expf(sm.sc.b[r] - sm.sc.b[s]) : 0.f;
      const float a = s < r ? cc(Fn.da, r, s) : 0.f;
      const float l = cc(Fn.l, r, s);
      betp += a * l;
      const float dl = sm.sc.bet[r] * a, dll = dl * l;
      const float pp = s <= r ? cc(Fn.dp, r, s) : 0.f;
      const float ppp = pp * cc(sm.p, r, s);
      rowp += dll + ppp;
      if (dll + ppp != 0.f) atomicAdd(&sm.db[s], -(dll + ppp));
      cc(Fn.da, r, s) = dl * gm;
      cc(Fn.dp, r, s) = pp * gm;
    }
    rowp += __shfl_xor_sync(0xffffffffu, rowp, 1);
    rowp += __shfl_xor_sync(0xffffffffu, rowp, 2);
    betp += __shfl_xor_sync(0xffffffffu, betp, 1);
    betp += __shfl_xor_sync(0xffffffffu, betp, 2);
    if ((tid & 3) == 0) {
      atomicAdd(&sm.db[r], rowp);
      sm.dbeta[r] += betp;
    }
  }
  __syncthreads();
  // ---- dQ += H K; dK += F K + F^T K + H^T Q
  wmma(aq, mr, nq, kCh, [&](int m, int kk) { return tf(cc(Fn.dp, m, kk)); },
       [&](int kk, int nn) { return bfbits(sm.k + kk * PH + nn); }, lane);
  wmma(ak, mr, nq, kCh, [&](int m, int kk) { return tf(cc(Fn.da, m, kk)); },
       [&](int kk, int nn) { return bfbits(sm.k + kk * PH + nn); }, lane);
  wmma(ak, mr, nq, kCh, [&](int m, int kk) { return tf(cc(Fn.da, kk, m)); },
       [&](int kk, int nn) { return bfbits(sm.k + kk * PH + nn); }, lane);
  wmma(ak, mr, nq, kCh, [&](int m, int kk) { return tf(cc(Fn.dp, kk, m)); },
       [&](int kk, int nn) { return bfbits(sm.q + kk * PH + nn); }, lane);
  each(aq, mr, nq, lane, [&](int r, int c, float &x) {
    if (r < n) dq[(row0 + r) * DK + c] = __float2bfloat16_rn(x);
  });
  each(ak, mr, nq, lane, [&](int r, int c, float &x) {
    if (r < n) dk[(row0 + r) * DK + c] = __float2bfloat16_rn(x);
  });
  // ---- db: the Kt terms and gL <S, E> at the last row; dg = the suffix sum within the chunk
  if (warp == 0) {
    const float gL = sm.sc.gam[kCh - 1];
    float sE = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sE += sm.red[w];
    const float k0 = sm.kd[lane], k1 = sm.kd[lane + 32];
    float ksum = k0 + k1;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ksum += __shfl_xor_sync(0xffffffffu, ksum, off);
    float d0 = sm.db[lane] - k0, d1 = sm.db[lane + 32] - k1;
    if (lane == 31) d1 += ksum + gL * sE;
    // suffix sums over 64 rows: lane holds rows lane and lane + 32
    float s1 = d1, s0 = d0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float a1 = __shfl_down_sync(0xffffffffu, s1, off), a0 = __shfl_down_sync(0xffffffffu, s0, off);
      if (lane + off < 32) {
        s1 += a1;
        s0 += a0;
      }
    }
    s0 += __shfl_sync(0xffffffffu, s1, 0);
    if (dg) {
      if (lane < n) dg[row0 + lane] = s0;
      if (lane + 32 < n) dg[row0 + lane + 32] = s1;
    }
    if (dbeta) {
      if (lane < n) dbeta[row0 + lane] = sm.dbeta[lane];
      if (lane + 32 < n) dbeta[row0 + lane + 32] = sm.dbeta[lane + 32];
    }
  }
}

// ============================================================ Kimi Delta Attention
// The same four passes with the per-key-channel gate. Per chunk, with B[r][c]
// the inclusive prefix of the chunk's log-gates, b_m = B[31] (the fold's
// midpoint), B_L = B[63], EP = e^{B - b_m} and, in the chunk's products,
// K+ = K EP, K- = K / EP, Q+ = Q EP, K^ = K e^B, K~ = K e^{B_L - B}, Q^ = Q e^B:
//
//   L = strict_lower(K+ K-^T),  T = (I + Diag(beta) L)^{-1},  P = lower(Q+ K-^T)
//   Z = V - K^ S,  U = T Diag(beta) Z,  S_next = Diag(e^{B_L}) S + K~^T U
//   dU = K~ E + P^T dO,  Y = T^T dU,  dZ = Diag(beta) Y = dV
//   dA = -strict_lower(Y U^T),  dL = Diag(beta) dA,  dP = lower(dO U^T)
//   X1 = e^{b_m} (-dZ S^T) + dL K-,  X2 = e^{B_L - b_m} (U E^T) + dL^T K+ + dP^T Q+
//   dQ = EP (e^{b_m} dO S^T + dP K-),  dK = EP X1 + X2 / EP
//   dbeta_r = Y_r . Z_r + sum_s dA_rs L_rs
//   dB = Q dQ + K (EP X1 - X2 / EP), plus, at the last row, the column sums of
//        K e^{B_L - B} (U E^T) and e^{B_L} <S, E> per key channel
//   dg = the suffix sum of dB inside the chunk (per key channel)
//   E_prev = Diag(e^{B_L}) E + Q^T dO - K^T dZ
//
// (the chain rule through the exponentials: e^{B_r} enters Q^ and K^ with +,
// K~ and the column side of L and P with -, the last row also through
// S_next's decay). The chains are the Gated DeltaNet ones with the folded
// images; the pre-pass and the gradient kernel form the folds in float32.

// ---- pre-pass: the folds, P and T (float32 and bf16), the chains' images.
// 256 threads: each folds one key-channel pair over RPG rows (RG row groups, the
// prefix from the groups' gate sums), with paired bf16 and float loads and stores.
template <int DK>
struct KPreSmem {
  static constexpr int FP = DK + 4;  // float pitch: conflict-free tf32 fragment reads
  static constexpr int RG = 256 / (DK / 2), RPG = kCh / RG;  // thread: a key-channel pair, RPG rows
  union {
    float qp[kCh * FP];  // Q+, then A
    float a[kCh * kPf];
  } u;
  float kp[kCh * FP], km[kCh * FP];
  float bet[kCh], gsum[RG * DK];
};

template <int DK>
__global__ void __launch_bounds__(256, 2) bk_pre_kernel(const __nv_bfloat16 *__restrict__ q,
                                                        const __nv_bfloat16 *__restrict__ k,
                                                        const float *__restrict__ g, const float *__restrict__ beta,
                                                        int T, float *__restrict__ Tw, float *__restrict__ Pw,
                                                        __nv_bfloat16 *__restrict__ Tb, __nv_bfloat16 *__restrict__ Pb,
                                                        __nv_bfloat16 *__restrict__ kh, __nv_bfloat16 *__restrict__ kt,
                                                        __nv_bfloat16 *__restrict__ qh, float *__restrict__ gl) {
  using Sm = KPreSmem<DK>;
  constexpr int FP = Sm::FP, RG = Sm::RG, RPG = Sm::RPG;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Sm &sm = *reinterpret_cast<Sm *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = blockIdx.x, bh = blockIdx.y, nch = gridDim.x;
  const int t0 = i * kCh, n = min(kCh, T - t0);
  const size_t row0 = (size_t)bh * T + t0, ci = (size_t)bh * nch + i;
  if (tid < kCh) sm.bet[tid] = tid < n ? (beta ? __ldg(beta + row0 + tid) : 1.f) : 0.f;
  // ---- channels c, c + 1, rows r0 .. r0 + RPG - 1: the local prefix in registers (zero gates
  //      past the end)
  const int c = 2 * (tid % (DK / 2)), grp = tid / (DK / 2), r0 = grp * RPG;
  float2 bc[RPG];
  {
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int r = 0; r < RPG; ++r) {
      const float2 x = r0 + r < n ? __ldg(reinterpret_cast<const float2 *>(g + (row0 + r0 + r) * DK + c))
                                  : make_float2(0.f, 0.f);
      acc.x += x.x;
      acc.y += x.y;
      bc[r] = acc;
    }
    sm.gsum[grp * DK + c] = acc.x;
    sm.gsum[grp * DK + c + 1] = acc.y;
  }
  __syncthreads();
  {
    float2 off = make_float2(0.f, 0.f), bm = off, bl = off;
#pragma unroll
    for (int j = 0; j < RG; ++j) {
      const float x0 = sm.gsum[j * DK + c], x1 = sm.gsum[j * DK + c + 1];
      if (j < grp) {
        off.x += x0;
        off.y += x1;
      }
      if (j * RPG < kCh / 2) {  // B at row 31: the groups of rows 0 .. 31
        bm.x += x0;
        bm.y += x1;
      }
      bl.x += x0;
      bl.y += x1;
    }
    const float2 ebm = make_float2(__expf(bm.x), __expf(bm.y)), eblm = make_float2(__expf(bl.x - bm.x), __expf(bl.y - bm.y));
    if (grp == 0) *reinterpret_cast<float2 *>(gl + ci * DK + c) = make_float2(__expf(bl.x), __expf(bl.y));
    const size_t ib = ci * kCh * DK;
    __nv_bfloat162 *kh2 = reinterpret_cast<__nv_bfloat162 *>(kh + ib), *qh2 = reinterpret_cast<__nv_bfloat162 *>(qh + ib),
                   *kt2 = reinterpret_cast<__nv_bfloat162 *>(kt + ib);
#pragma unroll
    for (int r = 0; r < RPG; ++r) {
      const int R = r0 + r;
      const bool ok = R < n;
      const float2 qx = ok ? __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(q + (row0 + R) * DK + c))
                           : make_float2(0.f, 0.f);
      const float2 kx = ok ? __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(k + (row0 + R) * DK + c))
                           : make_float2(0.f, 0.f);
      const float d0 = off.x + bc[r].x - bm.x, d1 = off.y + bc[r].y - bm.y;
      const float ep0 = __expf(d0), ep1 = __expf(d1), em0 = __expf(-d0), em1 = __expf(-d1);
      *reinterpret_cast<float2 *>(sm.u.qp + R * FP + c) = make_float2(qx.x * ep0, qx.y * ep1);
      *reinterpret_cast<float2 *>(sm.kp + R * FP + c) = make_float2(kx.x * ep0, kx.y * ep1);
      *reinterpret_cast<float2 *>(sm.km + R * FP + c) = make_float2(kx.x * em0, kx.y * em1);
      // e^B = EP e^{b_m} and e^{B_L - B} = EM e^{B_L - b_m} for the chains' bf16 images
      kh2[(R * DK + c) >> 1] = __floats2bfloat162_rn(kx.x * (ep0 * ebm.x), kx.y * (ep1 * ebm.y));
      qh2[(R * DK + c) >> 1] = __floats2bfloat162_rn(qx.x * (ep0 * ebm.x), qx.y * (ep1 * ebm.y));
      kt2[(R * DK + c) >> 1] = __floats2bfloat162_rn(kx.x * (em0 * eblm.x), kx.y * (em1 * eblm.y));
    }
  }
  __syncthreads();
  // ---- [Q+; K+] K-^T: warps 0..3 the rows of Q+ (P, stored at once), warps 4..7 the rows of
  //      K+ (A = Diag(beta) L, held until Q+ is dead); warp w: rows 16 (w % 4)
  const float *src = warp < 4 ? sm.u.qp : sm.kp;
  const int m0 = 16 * (warp & 3);
  float acc[8][4];
  const size_t cbase = ci * kCh * kCh;
  zero(acc);
  wmma(acc, m0, 0, DK, [&](int m, int kk) { return tf(src[m * FP + kk]); },
       [&](int kk, int nn) { return tf(sm.km[nn * FP + kk]); }, lane);
  if (warp < 4)
    each(acc, m0, 0, lane, [&](int r, int s2, float &x) {
      const float y = s2 <= r ? x : 0.f;
      Pw[cbase + r * kCh + s2] = y;
      Pb[cbase + r * kCh + s2] = __float2bfloat16_rn(y);
    });
  __syncthreads();
  if (warp >= 4)
    each(acc, m0, 0, lane, [&](int r, int s2, float &x) { cc(sm.u.a, r, s2) = s2 < r ? sm.bet[r] * x : 0.f; });
  __syncthreads();
  // ---- T = (I + A)^{-1}: column j by forward substitution (as for Gated DeltaNet)
  if (tid < kCh) {
    const int j = tid;
    float tc[kCh];
#pragma unroll
    for (int r = 0; r < kCh; ++r) {
      float x[4] = {r == j ? 1.f : 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s2 = 0; s2 < r; ++s2) x[s2 & 3] = fmaf(-cc(sm.u.a, r, s2), tc[s2], x[s2 & 3]);
      tc[r] = r < j ? 0.f : (x[0] + x[1]) + (x[2] + x[3]);
    }
#pragma unroll
    for (int r = 0; r < kCh; ++r) {
      Tw[cbase + r * kCh + j] = tc[r];
      Tb[cbase + r * kCh + j] = __float2bfloat16_rn(tc[r]);
    }
  }
}

// ---- per-chunk gradients (tf32 warp MMAs, as bd_grad_kernel; the folds applied in
//      float32 as the operands are read: EP in shared memory, per-channel factors)
template <int DK>
struct KGradBlk {
  float s[DK * kPw], e[DK * kPw];
  __nv_bfloat16 v[kCh * kPh], o[kCh * kPh];
};
template <int DK>
struct KGradSmem {
  static constexpr int FP = DK + 4;
  __nv_bfloat16 q[kCh * Pitch<DK>::h], k[kCh * Pitch<DK>::h];
  float ep[kCh * FP], em[kCh * FP];  // e^{B - b_m} and e^{b_m - B}
  float t[kCh * kPf], p[kCh * kPf];
  union {
    struct {
      KGradBlk<DK> b[2];
      float ks[kCh * kPw], ke[kCh * kPw], z[kCh * kPw], u[kCh * kPw], du[kCh * kPw], y[kCh * kPw];
    } blk;
    struct {  // after the blocks: dA (then dL), dP, L; then dB
      float da[kCh * kPf], dp[kCh * kPf], l[kCh * kPf];
      float db[kCh * FP];
    } fin;
  } w;
  float bet[kCh], dbeta[kCh], ebm[DK], eblm[DK], ebl[DK], se[DK], dbl[DK];
};

template <int DK, int DV>
__global__ void __launch_bounds__(256, 1) bk_grad_kernel(
    const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
    const __nv_bfloat16 *__restrict__ dO, const float *__restrict__ g, const float *__restrict__ beta, int T,
    const float *__restrict__ Tw, const float *__restrict__ Pw, const float *__restrict__ Sin,
    const float *__restrict__ Eout, __nv_bfloat16 *__restrict__ dq, __nv_bfloat16 *__restrict__ dk,
    __nv_bfloat16 *__restrict__ dv, float *__restrict__ dbeta, float *__restrict__ dg) {
  constexpr int PH = Pitch<DK>::h, NT = DK / 16, FP = KGradSmem<DK>::FP;
  constexpr int TPC = 256 / DK, CPT = kCW / TPC;  // <S, E>: threads per key channel, columns per thread
  extern __shared__ __align__(16) uint8_t smem_raw[];
  KGradSmem<DK> &sm = *reinterpret_cast<KGradSmem<DK> *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = blockIdx.x, bh = blockIdx.y, nch = gridDim.x;
  const int t0 = i * kCh, n = min(kCh, T - t0);
  const size_t row0 = (size_t)bh * T + t0;
  const size_t cbase = ((size_t)bh * nch + i) * kCh * kCh, sbase = ((size_t)bh * nch + i) * DK * DV;
  auto &W = sm.w.blk;
  auto issue_blk = [&](int c0, KGradBlk<DK> &b) {
    state_async<DK, DV>(b.s, Sin + sbase, c0, tid, 256);
    state_async<DK, DV>(b.e, Eout + sbase, c0, tid, 256);
    cols_async<DV>(b.v, v + row0 * DV, c0, n, tid, 256);
    cols_async<DV>(b.o, dO + row0 * DV, c0, n, tid, 256);
  };
  rows_async<DK, PH>(sm.q, q + row0 * DK, n, tid, 256);
  rows_async<DK, PH>(sm.k, k + row0 * DK, n, tid, 256);
  cc_async(sm.t, Tw + cbase, tid, 256);
  cc_async(sm.p, Pw + cbase, tid, 256);
  issue_blk(0, W.b[0]);
  cp_commit();
  if (tid < kCh) {
    sm.bet[tid] = tid < n ? (beta ? __ldg(beta + row0 + tid) : 1.f) : 0.f;
    sm.dbeta[tid] = 0.f;
  }
  if (tid < DK) {  // channel c = tid: EP and the per-channel factors
    const int c = tid;
    float bc[kCh];
    float acc = 0.f;
#pragma unroll
    for (int r = 0; r < kCh; ++r) {
      acc += r < n ? __ldg(g + (row0 + r) * DK + c) : 0.f;
      bc[r] = acc;
    }
    const float bm = bc[kCh / 2 - 1], bl = bc[kCh - 1];
#pragma unroll
    for (int r = 0; r < kCh; ++r) {
      sm.ep[r * FP + c] = __expf(bc[r] - bm);
      sm.em[r * FP + c] = __expf(bm - bc[r]);
    }
    sm.ebm[c] = __expf(bm);
    sm.eblm[c] = __expf(bl - bm);
    sm.ebl[c] = __expf(bl);
    sm.dbl[c] = 0.f;
  }
  // folded operands read from the raw bf16 tiles
  auto kf = [&](int r, int c) { return bf(sm.k + r * PH + c); };
  auto qf = [&](int r, int c) { return bf(sm.q + r * PH + c); };
  const int mr = 16 * (warp & 3), half = warp >> 2;
  const int nq = half * (DK / 2), na = half * 32;
  float aq[NT][4], ak1[NT][4], ak2[NT][4], aa[4][4], ap[4][4];
  zero(aq);
  zero(ak1);
  zero(ak2);
  zero(aa);
  zero(ap);
  float se = 0.f;  // <S, E> over channel tid / TPC, this thread's columns
  const int nc = 8 * half;
  for (int c0 = 0, cb = 0; c0 < DV; c0 += kCW, ++cb) {
    KGradBlk<DK> &B = W.b[cb & 1];
    if (c0 + kCW < DV) {
      issue_blk(c0 + kCW, W.b[(cb + 1) & 1]);
      cp_commit();
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    {
      const int c = tid / TPC, j0 = (tid % TPC) * CPT;
#pragma unroll
      for (int j = 0; j < CPT; ++j) se += w16(B.s, c, j0 + j) * w16(B.e, c, j0 + j);
    }
    // ---- K^ S and K~ E: one 16 x 8 tile each per warp
    {
      float a[1][4], b[1][4];
      zero(a);
      zero(b);
      wmma(a, mr, nc, DK, [&](int m, int kk) { return tf(kf(m, kk) * sm.ep[m * FP + kk] * sm.ebm[kk]); },
           [&](int kk, int nn) { return tf(w16(B.s, kk, nn)); }, lane);
      wmma(b, mr, nc, DK, [&](int m, int kk) { return tf(kf(m, kk) * sm.eblm[kk] * sm.em[m * FP + kk]); },
           [&](int kk, int nn) { return tf(w16(B.e, kk, nn)); }, lane);
      each(a, mr, nc, lane, [&](int r, int col, float &x) { w16(W.ks, r, col) = x; });
      each(b, mr, nc, lane, [&](int r, int col, float &x) { w16(W.ke, r, col) = x; });
    }
    __syncthreads();
    // ---- Z = V - K^ S
    {
      const int r = tid >> 2, cq = (tid & 3) * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e) w16(W.z, r, cq + e) = bf(B.v + r * kPh + cq + e) - w16(W.ks, r, cq + e);
    }
    __syncthreads();
    // ---- U = T Diag(beta) Z; dU = K~ E + P^T dO
    {
      float a[1][4], b[1][4];
      zero(a);
      wmma(a, mr, nc, kCh, [&](int m, int kk) { return tf(cc(sm.t, m, kk)); },
           [&](int kk, int nn) { return tf(sm.bet[kk] * w16(W.z, kk, nn)); }, lane);
      each(a, mr, nc, lane, [&](int r, int col, float &x) { w16(W.u, r, col) = x; });
      each(b, mr, nc, lane, [&](int r, int col, float &x) { x = w16(W.ke, r, col); });
      wmma(b, mr, nc, kCh, [&](int m, int kk) { return tf(cc(sm.p, kk, m)); },
           [&](int kk, int nn) { return bfbits(B.o + kk * kPh + nn); }, lane);
      each(b, mr, nc, lane, [&](int r, int col, float &x) { w16(W.du, r, col) = x; });
    }
    __syncthreads();
    // ---- Y = T^T dU; dV = Diag(beta) Y; dbeta += Y . Z
    {
      float a[1][4];
      zero(a);
      wmma(a, mr, nc, kCh, [&](int m, int kk) { return tf(cc(sm.t, kk, m)); },
           [&](int kk, int nn) { return tf(w16(W.du, kk, nn)); }, lane);
      const int gg = lane >> 2;
      float pb[2] = {0.f, 0.f};
      each(a, mr, nc, lane, [&](int r, int col, float &y) {
        const int h = (r - mr - gg) >> 3;
        w16(W.y, r, col) = y;
        if (r < n) dv[(row0 + r) * DV + c0 + col] = __float2bfloat16_rn(sm.bet[r] * y);
        pb[h] += y * w16(W.z, r, col);
      });
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        pb[h] += __shfl_xor_sync(0xffffffffu, pb[h], 1);
        pb[h] += __shfl_xor_sync(0xffffffffu, pb[h], 2);
        if ((lane & 3) == 0) atomicAdd(&sm.dbeta[mr + gg + 8 * h], pb[h]);
      }
    }
    __syncthreads();
    // ---- dA -= Y U^T, dP += dO U^T; dO S^T, -dZ S^T = -Diag(beta) Y S^T, U E^T (K = 16 each)
    wmma(aa, mr, na, kCW, [&](int m, int kk) { return tf(-w16(W.y, m, kk)); },
         [&](int kk, int nn) { return tf(w16(W.u, nn, kk)); }, lane);
    wmma(ap, mr, na, kCW, [&](int m, int kk) { return bfbits(B.o + m * kPh + kk); },
         [&](int kk, int nn) { return tf(w16(W.u, nn, kk)); }, lane);
    wmma(aq, mr, nq, kCW, [&](int m, int kk) { return bfbits(B.o + m * kPh + kk); },
         [&](int kk, int nn) { return tf(w16(B.s, nn, kk)); }, lane);
    wmma(ak1, mr, nq, kCW, [&](int m, int kk) { return tf(-sm.bet[m] * w16(W.y, m, kk)); },
         [&](int kk, int nn) { return tf(w16(B.s, nn, kk)); }, lane);
    wmma(ak2, mr, nq, kCW, [&](int m, int kk) { return tf(w16(W.u, m, kk)); },
         [&](int kk, int nn) { return tf(w16(B.e, nn, kk)); }, lane);
    __syncthreads();
  }
  // ---- <S, E> per channel
#pragma unroll
  for (int off = 1; off < TPC; off <<= 1) se += __shfl_xor_sync(0xffffffffu, se, off);
  if (tid % TPC == 0) sm.se[tid / TPC] = se;
  // ---- dA, dP to shared memory; L = strict_lower(K+ K-^T)
  auto &Fn = sm.w.fin;
  each(aa, mr, na, lane, [&](int r, int s2, float &x) { cc(Fn.da, r, s2) = x; });
  each(ap, mr, na, lane, [&](int r, int s2, float &x) { cc(Fn.dp, r, s2) = x; });
  {
    float a[4][4];
    zero(a);
    wmma(a, mr, na, DK, [&](int m, int kk) { return tf(kf(m, kk) * sm.ep[m * FP + kk]); },
           [&](int kk, int nn) { return tf(kf(nn, kk) * sm.em[nn * FP + kk]); }, lane);
    each(a, mr, na, lane, [&](int r, int s2, float &x) { cc(Fn.l, r, s2) = s2 < r ? x : 0.f; });
  }
  __syncthreads();
  // ---- dL = Diag(beta) dA (strict lower), dP masked (lower); dbeta += sum_s dA L
  {
    const int r = tid >> 2;
    float betp = 0.f;
    for (int jj = 0; jj < kCh / 4; ++jj) {
      const int s2 = (tid & 3) + 4 * jj;
      const float a = s2 < r ? cc(Fn.da, r, s2) : 0.f;
      betp += a * cc(Fn.l, r, s2);
      cc(Fn.da, r, s2) = sm.bet[r] * a;
      cc(Fn.dp, r, s2) = s2 <= r ? cc(Fn.dp, r, s2) : 0.f;
    }
    betp += __shfl_xor_sync(0xffffffffu, betp, 1);
    betp += __shfl_xor_sync(0xffffffffu, betp, 2);
    if ((tid & 3) == 0) sm.dbeta[r] += betp;
  }
  __syncthreads();
  // ---- dQ/EP = e^{b_m} dO S^T + dP K-;  X1 = -e^{b_m} dZ S^T + dL K-;
  //      X2 = e^{B_L - b_m} U E^T (its K~-weighted column sums to dB's last row) + dL^T K+ + dP^T Q+
  each(aq, mr, nq, lane, [&](int, int c, float &x) { x *= sm.ebm[c]; });
  each(ak1, mr, nq, lane, [&](int, int c, float &x) { x *= sm.ebm[c]; });
  each(ak2, mr, nq, lane, [&](int, int c, float &x) { x *= sm.eblm[c]; });
  {
    // column sums over this warp's 16 rows of K (e^{B_L - B} U E^T) = K X2 / EP, per channel
    float cs[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) cs[j][0] = cs[j][1] = 0.f;
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = mr + g + 8 * (e >> 1), c = nq + 8 * j + 2 * t + (e & 1);
        cs[j][e & 1] += kf(r, c) * ak2[j][e] * sm.em[r * FP + c];
      }
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float x = cs[j][h];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
        if (g == 0) atomicAdd(&sm.dbl[nq + 8 * j + 2 * t + h], x);
      }
  }
  auto kmin = [&](int s2, int c) { return tf(kf(s2, c) * sm.em[s2 * FP + c]); };
  auto kplus = [&](int s2, int c) { return tf(kf(s2, c) * sm.ep[s2 * FP + c]); };
  auto qplus = [&](int s2, int c) { return tf(qf(s2, c) * sm.ep[s2 * FP + c]); };
  wmma(aq, mr, nq, kCh, [&](int m, int kk) { return tf(cc(Fn.dp, m, kk)); }, kmin, lane);
  wmma(ak1, mr, nq, kCh, [&](int m, int kk) { return tf(cc(Fn.da, m, kk)); }, kmin, lane);
  wmma(ak2, mr, nq, kCh, [&](int m, int kk) { return tf(cc(Fn.da, kk, m)); }, kplus, lane);
  wmma(ak2, mr, nq, kCh, [&](int m, int kk) { return tf(cc(Fn.dp, kk, m)); }, qplus, lane);
  // ---- dQ, dK; dB = Q dQ + K (EP X1 - X2 / EP) to shared memory
  {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = mr + g + 8 * (e >> 1), c = nq + 8 * j + 2 * t + (e & 1);
        const float epv = sm.ep[r * FP + c];
        const float dqv = epv * aq[j][e], x1 = epv * ak1[j][e], x2 = ak2[j][e] * sm.em[r * FP + c];
        if (r < n) {
          dq[(row0 + r) * DK + c] = __float2bfloat16_rn(dqv);
          dk[(row0 + r) * DK + c] = __float2bfloat16_rn(x1 + x2);
        }
        Fn.db[r * FP + c] = qf(r, c) * dqv + kf(r, c) * (x1 - x2);
      }
  }
  __syncthreads();
  // ---- dg: the suffix sum of dB per channel, the last row with its extra terms
  if (tid < DK) {
    const int c = tid;
    float run = sm.dbl[c] + sm.ebl[c] * sm.se[c];
    for (int r = kCh - 1; r >= 0; --r) {
      run += Fn.db[r * FP + c];
      if (dg && r < n) dg[(row0 + r) * DK + c] = run;
    }
  }
  if (dbeta && tid < n) dbeta[row0 + tid] = sm.dbeta[tid];
}

template <class Smem, class K>
cudaError_t set_smem(K kernel) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem));
}

template <int DK, int DV>
int launch_typed(const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                 const __nv_bfloat16 *dO, const float *g, const float *beta, const float *S0, const float *dS,
                 __nv_bfloat16 *dq, __nv_bfloat16 *dk, __nv_bfloat16 *dv, float *dbeta, float *dg, float *dS0,
                 int BH, int T, uint8_t *ws, cudaStream_t s) {
  const int nch = (T + kCh - 1) / kCh;
  const size_t ncc = (size_t)BH * nch * kCh * kCh, nss = (size_t)BH * nch * DK * DV;
  float *Tw = reinterpret_cast<float *>(ws), *Pw = Tw + ncc, *Sin = Pw + ncc, *Eout = Sin + nss;
  __nv_bfloat16 *Tb = reinterpret_cast<__nv_bfloat16 *>(Eout + nss), *Pb = Tb + ncc;
  cudaError_t e = set_smem<PreSmem<DK>>(bd_pre_kernel<DK>);
  if (e == cudaSuccess) e = set_smem<FwdSmem<DK, false>>(bd_fwd_kernel<DK, DV, false>);
  if (e == cudaSuccess) e = set_smem<BwdSmem<DK, false>>(bd_bwd_kernel<DK, DV, false>);
  if (e == cudaSuccess) e = set_smem<GradSmem<DK>>(bd_grad_kernel<DK, DV>);
  if (e == cudaSuccess) {
    bd_pre_kernel<DK><<<dim3(nch, BH), 128, sizeof(PreSmem<DK>), s>>>(q, k, g, beta, T, Tw, Pw, Tb, Pb);
    e = cudaGetLastError();
  }
  const unsigned nchain = (unsigned)(BH * (DV / kBW));
  if (e == cudaSuccess) {
    bd_fwd_kernel<DK, DV, false><<<nchain, 256, sizeof(FwdSmem<DK, false>), s>>>(k, v, g, beta, S0, T, Tb, Sin,
                                                                                KdaImages{});
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    bd_bwd_kernel<DK, DV, false><<<nchain, 256, sizeof(BwdSmem<DK, false>), s>>>(q, k, dO, g, beta, dS, T, Tb, Pb,
                                                                                Eout, dS0, KdaImages{});
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    bd_grad_kernel<DK, DV><<<dim3(nch, BH), 256, sizeof(GradSmem<DK>), s>>>(q, k, v, dO, g, beta, T, Tw, Pw, Sin,
                                                                           Eout, dq, dk, dv, dbeta, dg);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_error("la_chunk_bwd_delta: kernel launch failed: %s", cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  return LA_OK;
}

// Kimi Delta Attention: workspace per chunk -- T and P in float32 and bf16, the
// folded bf16 images K e^B, K e^{B_L - B}, Q e^B, e^{B_L}, and the S and E images
template <int DK, int DV>
int launch_kda(const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v, const __nv_bfloat16 *dO,
               const float *g, const float *beta, const float *S0, const float *dS, __nv_bfloat16 *dq,
               __nv_bfloat16 *dk, __nv_bfloat16 *dv, float *dbeta, float *dg, float *dS0, int BH, int T, uint8_t *ws,
               cudaStream_t s) {
  using bf = __nv_bfloat16;
  const int nch = (T + kCh - 1) / kCh;
  const size_t ncc = (size_t)BH * nch * kCh * kCh, nss = (size_t)BH * nch * DK * DV, nim = (size_t)BH * nch * kCh * DK;
  float *Tw = reinterpret_cast<float *>(ws), *Pw = Tw + ncc, *Sin = Pw + ncc, *Eout = Sin + nss, *gl = Eout + nss;
  bf *Tb = reinterpret_cast<bf *>(gl + (size_t)BH * nch * DK), *Pb = Tb + ncc, *kh = Pb + ncc, *kt = kh + nim,
     *qh = kt + nim;
  const KdaImages img{kh, kt, qh, gl};
  cudaError_t e = set_smem<KPreSmem<DK>>(bk_pre_kernel<DK>);
  if (e == cudaSuccess) e = set_smem<FwdSmem<DK, true>>(bd_fwd_kernel<DK, DV, true>);
  if (e == cudaSuccess) e = set_smem<BwdSmem<DK, true>>(bd_bwd_kernel<DK, DV, true>);
  if (e == cudaSuccess) e = set_smem<KGradSmem<DK>>(bk_grad_kernel<DK, DV>);
  if (e == cudaSuccess) {
    bk_pre_kernel<DK><<<dim3(nch, BH), 256, sizeof(KPreSmem<DK>), s>>>(q, k, g, beta, T, Tw, Pw, Tb, Pb, kh, kt, qh,
                                                                      gl);
    e = cudaGetLastError();
  }
  const unsigned nchain = (unsigned)(BH * (DV / kBW));
  if (e == cudaSuccess) {  // the chains take the gates through the images (g = NULL)
    bd_fwd_kernel<DK, DV, true><<<nchain, 256, sizeof(FwdSmem<DK, true>), s>>>(nullptr, v, nullptr, beta, S0, T, Tb,
                                                                               Sin, img);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    bd_bwd_kernel<DK, DV, true><<<nchain, 256, sizeof(BwdSmem<DK, true>), s>>>(nullptr, nullptr, dO, nullptr, beta, dS,
                                                                               T, Tb, Pb, Eout, dS0, img);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    bk_grad_kernel<DK, DV><<<dim3(nch, BH), 256, sizeof(KGradSmem<DK>), s>>>(q, k, v, dO, g, beta, T, Tw, Pw, Sin,
                                                                            Eout, dq, dk, dv, dbeta, dg);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_error("la_chunk_bwd_delta: kernel launch failed: %s", cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  return LA_OK;
}

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

size_t kda_bwd_workspace_bytes(int BH, int T, int dk, int dv) {
  const size_t nch = (size_t)(T + kCh - 1) / kCh;
  return (size_t)BH * nch *
         ((2 * kCh * kCh + 2 * (size_t)dk * dv + dk) * sizeof(float) + (2 * kCh * kCh + 3 * (size_t)kCh * dk) * 2);
}

size_t delta_bwd_workspace_bytes(int BH, int T, int dk, int dv) {
  const size_t nch = (size_t)(T + kCh - 1) / kCh;
  // float32 T, P, S and E images, then bfloat16 copies of T and P for the chains
  return (size_t)BH * nch * ((2 * kCh * kCh + 2 * (size_t)dk * dv) * sizeof(float) + 2 * kCh * kCh * 2);
}

}  // namespace la

using namespace la;

extern "C" int la_chunk_bwd_delta(const void *q, const void *k, const void *v, const float *g, const float *beta,
                                  const void *dO, const float *dS_final, const float *S0, void *dq_out,
                                  void *dk_out, void *dv_out, float *dbeta_out, float *dg_out, float *dS0,
                                  int B, int H, int T, int dk, int dv, int C, int mode, la_stream_t stream) {
  la::NvtxRange nvtx_range("la_chunk_bwd_delta");
  const char *fn = "la_chunk_bwd_delta";
  set_error("%s", "");
  if (!q || !k || !v || !dO || !dq_out || !dk_out || !dv_out) {
    set_error("%s: q, k, v, dO, dq, dk and dv are required", fn);
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
  const int kind = mode & 0xff;
  if ((mode & ~(0xff | LA_F32)) != 0 || kind < LA_LINEAR || kind > LA_OUTER_GATE) {
    set_error("%s: unknown mode 0x%x", fn, mode);
    return LA_ERR_INVALID_ARG;
  }
  if ((kind != LA_GDN && kind != LA_KDA) || (mode & LA_F32)) {
    set_error("%s: covers LA_GDN and LA_KDA with bfloat16 inputs (got mode 0x%x)", fn, mode);
    return LA_ERR_UNSUPPORTED;
  }
  const bool kda = kind == LA_KDA;
  if (kda && !g) {
    set_error("%s: LA_KDA needs the per-channel log-gates g", fn);
    return LA_ERR_INVALID_ARG;
  }
  if (dg_out && !g) {
    set_error("%s: dg needs the log-gates g (NULL g means alpha = 1, which has no gradient)", fn);
    return LA_ERR_INVALID_ARG;
  }
  if (C != 0 && C != 64) {
    set_error("%s: chunk length C=%d is not implemented (use 0 or 64)", fn, C);
    return LA_ERR_UNSUPPORTED;
  }
  const void *p16[] = {q, k, v, dO, dq_out, dk_out, dv_out};
  for (const void *ptr : p16)
    if (!al16(ptr)) {
      set_error("%s: q, k, v, dO, dq, dk and dv must be 16-byte aligned", fn);
      return LA_ERR_INVALID_ARG;
    }
  if ((S0 && !al16(S0)) || (dS_final && !al16(dS_final)) || (dS0 && !al16(dS0)) || (g && !al16(g)) ||
      (beta && !al16(beta)) || (dg_out && !al16(dg_out)) || (dbeta_out && !al16(dbeta_out))) {
    set_error("%s: g, beta, S0, dS_final, dS0, dg and dbeta must be 16-byte aligned", fn);
    return LA_ERR_INVALID_ARG;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int BH = B * H;
  const size_t bytes = kda ? kda_bwd_workspace_bytes(BH, T, dk, dv) : delta_bwd_workspace_bytes(BH, T, dk, dv);
  cudaMemPool_t pool = library_pool();
  if (!pool) {
    set_error("%s: could not create the workspace pool: %s", fn, cudaGetErrorString(cudaGetLastError()));
    return LA_ERR_CUDA;
  }
  uint8_t *ws = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&ws), bytes, pool, s);
  if (e != cudaSuccess) {
    set_error("%s: workspace allocation of %zu bytes failed: %s", fn, bytes, cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  using bf = __nv_bfloat16;
  auto qb = static_cast<const bf *>(q), kb = static_cast<const bf *>(k), vb = static_cast<const bf *>(v),
       ob = static_cast<const bf *>(dO);
  auto dqb = static_cast<bf *>(dq_out), dkb = static_cast<bf *>(dk_out), dvb = static_cast<bf *>(dv_out);
  int rc;
  if (kda) {
    if (dk == 128 && dv == 128)
      rc = launch_kda<128, 128>(qb, kb, vb, ob, g, beta, S0, dS_final, dqb, dkb, dvb, dbeta_out, dg_out, dS0, BH, T,
                                ws, s);
    else if (dk == 128)
      rc = launch_kda<128, 64>(qb, kb, vb, ob, g, beta, S0, dS_final, dqb, dkb, dvb, dbeta_out, dg_out, dS0, BH, T,
                               ws, s);
    else if (dv == 128)
      rc = launch_kda<64, 128>(qb, kb, vb, ob, g, beta, S0, dS_final, dqb, dkb, dvb, dbeta_out, dg_out, dS0, BH, T,
                               ws, s);
    else
      rc = launch_kda<64, 64>(qb, kb, vb, ob, g, beta, S0, dS_final, dqb, dkb, dvb, dbeta_out, dg_out, dS0, BH, T,
                              ws, s);
  } else if (dk == 128 && dv == 128)
    rc = launch_typed<128, 128>(qb, kb, vb, ob, g, beta, S0, dS_final, dqb, dkb, dvb, dbeta_out, dg_out, dS0, BH, T,
                                ws, s);
  else if (dk == 128)
    rc = launch_typed<128, 64>(qb, kb, vb, ob, g, beta, S0, dS_final, dqb, dkb, dvb, dbeta_out, dg_out, dS0, BH, T,
                               ws, s);
  else if (dv == 128)
    rc = launch_typed<64, 128>(qb, kb, vb, ob, g, beta, S0, dS_final, dqb, dkb, dvb, dbeta_out, dg_out, dS0, BH, T,
                               ws, s);
  else
    rc = launch_typed<64, 64>(qb, kb, vb, ob, g, beta, S0, dS_final, dqb, dkb, dvb, dbeta_out, dg_out, dS0, BH, T,
                              ws, s);
  e = cudaFreeAsync(ws, s);
  if (rc == LA_OK && e != cudaSuccess) {
    set_error("%s: workspace release failed: %s", fn, cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  return rc;
}
