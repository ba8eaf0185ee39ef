// Two-phase chunk forward of the generalised delta rule ("Talk Linear
// Attention", section 7.1: an identity-plus-rank-one transition between
// linear-attention steps), key-major,
//
//   S_t = (I - b_t a_t^T) S_{t-1} + k_t v_t^T,   o_t = S_t^T q_t,
//
// bf16 inputs on tf32 warp MMAs. Per chunk of C = 64 rows with incoming state
// S the retrieved values u_r = S_{r-1}^T a_r solve (I + L_ab) U = A S + L_ak V
// (L_ab[r,s] = a_r.b_s, L_ak[r,s] = a_r.k_s for s < r), so with
// T = (I + L_ab)^{-1}
//
//   U = W S + M V,           W = T A,  M = T L_ak
//   O = Q S + P1 V - P2 U,   P1 = lower(Q K^T), P2 = lower(Q B^T)
//   S <- S + K^T V - B^T U
//
// Phase 1 (gdw_pre_kernel, every chunk in parallel): P1, P2, L_ak, L_ab from
// two [Q; A] products, T by substitution, W and M; written to a workspace.
// Phase 2 (gdw_chain_kernel, per head and 16 value columns -- every value
// column of S evolves on its own): the chunks in order, S in registers, each
// chunk's tiles copied asynchronously while the previous chunk finishes.
// A tail chunk is padded with zero rows, which leaves every real row's result
// unchanged.
#include <cuda_bf16.h>

#include <cstdint>

#include "la_internal.h"
#include "la_warp_mma.cuh"

namespace la {
namespace {

using namespace wm;

// ============================================================ phase 1
template <int DK>
struct GwPreSmem {
  __nv_bfloat16 q[kCh * Pitch<DK>::h], k[kCh * Pitch<DK>::h], a[kCh * Pitch<DK>::h], b[kCh * Pitch<DK>::h];
  float lab[kCh * kPf], lak[kCh * kPf], t[kCh * kPf];
};

template <int DK>
__global__ void __launch_bounds__(128) gdw_pre_kernel(const __nv_bfloat16 *__restrict__ q,
                                                      const __nv_bfloat16 *__restrict__ k,
                                                      const __nv_bfloat16 *__restrict__ a,
                                                      const __nv_bfloat16 *__restrict__ b, int T,
                                                      float *__restrict__ Ww, float *__restrict__ Mw,
                                                      float *__restrict__ P1w, float *__restrict__ P2w) {
  constexpr int PH = Pitch<DK>::h;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  GwPreSmem<DK> &sm = *reinterpret_cast<GwPreSmem<DK> *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = blockIdx.x, bh = blockIdx.y, nch = gridDim.x;
  const int t0 = i * kCh, n = min(kCh, T - t0);
  const size_t row0 = (size_t)bh * T + t0;
  rows_async<DK, PH>(sm.q, q + row0 * DK, n, tid, 128);
  rows_async<DK, PH>(sm.k, k + row0 * DK, n, tid, 128);
  rows_async<DK, PH>(sm.a, a + row0 * DK, n, tid, 128);
  rows_async<DK, PH>(sm.b, b + row0 * DK, n, tid, 128);
  cp_commit();
  cp_wait<0>();
  __syncthreads();
  const size_t cbase = ((size_t)bh * nch + i) * kCh * kCh;
  // [Q; A] K^T and [Q; A] B^T: warps 0, 1 the rows of Q (P1, P2), warps 2, 3 the rows of A (L_ak, L_ab)
  const __nv_bfloat16 *src = warp < 2 ? sm.q : sm.a;
  const int rbase = (warp & 1) * 32;
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const __nv_bfloat16 *rhs = pass == 0 ? sm.k : sm.b;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float acc[8][4];
      zero(acc);
      wmma(acc, rbase + 16 * h, 0, DK, [&](int m, int kk) { return bfbits(src + m * PH + kk); },
           [&](int kk, int nn) { return bfbits(rhs + nn * PH + kk); }, lane);
      if (warp < 2) {
        float *P = pass == 0 ? P1w : P2w;
        each(acc, rbase + 16 * h, 0, lane, [&](int r, int s, float &x) { P[cbase + r * kCh + s] = s <= r ? x : 0.f; });
      } else {
        float *L = pass == 0 ? sm.lak : sm.lab;
        each(acc, rbase + 16 * h, 0, lane, [&](int r, int s, float &x) { cc(L, r, s) = s < r ? x : 0.f; });
      }
    }
  }
  __syncthreads();
  // T = (I + L_ab)^{-1}, unit lower triangular: column j by forward substitution, in registers
  if (tid < kCh) {
    const int j = tid;
    float tc[kCh];
#pragma unroll
    for (int r = 0; r < kCh; ++r) {
      // four partial sums, so the row's FMAs do not form one dependent chain
      float x[4] = {r == j ? 1.f : 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < r; ++s) x[s & 3] = fmaf(-cc(sm.lab, r, s), tc[s], x[s & 3]);
      tc[r] = r < j ? 0.f : (x[0] + x[1]) + (x[2] + x[3]);
    }
#pragma unroll
    for (int r = 0; r < kCh; ++r) cc(sm.t, r, j) = tc[r];
  }
  __syncthreads();
  // W = T A (64 x DK), M = T L_ak (64 x 64): warp w, rows 16 w
  {
    float acc[DK / 8][4];
    zero(acc);
    wmma(acc, 16 * warp, 0, kCh, [&](int m, int kk) { return tf(cc(sm.t, m, kk)); },
         [&](int kk, int nn) { return bfbits(sm.a + kk * PH + nn); }, lane);
    const size_t wbase = ((size_t)bh * nch + i) * kCh * DK;
    each(acc, 16 * warp, 0, lane, [&](int r, int c, float &x) { Ww[wbase + r * DK + c] = x; });
  }
  {
    float acc[8][4];
    zero(acc);
    wmma(acc, 16 * warp, 0, kCh, [&](int m, int kk) { return tf(cc(sm.t, m, kk)); },
         [&](int kk, int nn) { return tf(cc(sm.lak, kk, nn)); }, lane);
    each(acc, 16 * warp, 0, lane, [&](int r, int s, float &x) { Mw[cbase + r * kCh + s] = x; });
  }
}

// ============================================================ phase 2
template <int DK>
struct GwChainSmem {
  __nv_bfloat16 q[kCh * Pitch<DK>::h], k[kCh * Pitch<DK>::h], b[kCh * Pitch<DK>::h], v[kCh * kPh];
  float w[kCh * DK], m[kCh * kPf], p1[kCh * kPf], p2[kCh * kPf], s[DK * kPw], u[kCh * kPw];
};

template <int DK, int DV>
__global__ void __launch_bounds__(128) gdw_chain_kernel(
    const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
    const __nv_bfloat16 *__restrict__ b, __nv_bfloat16 *__restrict__ o, const float *__restrict__ S0,
    float *__restrict__ S_final, int T, const float *__restrict__ Ww, const float *__restrict__ Mw,
    const float *__restrict__ P1w, const float *__restrict__ P2w) {
  constexpr int PH = Pitch<DK>::h, NCB = DV / kCW, RT = DK / 64;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  GwChainSmem<DK> &sm = *reinterpret_cast<GwChainSmem<DK> *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x / NCB, c0 = (blockIdx.x % NCB) * kCW;
  const int nch = (T + kCh - 1) / kCh;
  // a chunk's tiles in two groups: q, W, M, P1 are read in phase 1 only, so the next
  // chunk's copies start once phase 1 is done; k, b, v and P2 after phase 2
  auto issue_a = [&](int i) {
    const int t0 = i * kCh, n = min(kCh, T - t0);
    const size_t row0 = (size_t)bh * T + t0, cb = ((size_t)bh * nch + i) * kCh * kCh;
    rows_async<DK, PH>(sm.q, q + row0 * DK, n, tid, 128);
    wide_async<DK>(sm.w, Ww + ((size_t)bh * nch + i) * kCh * DK, tid, 128);
    cc_async(sm.m, Mw + cb, tid, 128);
    cc_async(sm.p1, P1w + cb, tid, 128);
    cp_commit();
  };
  auto issue_b = [&](int i) {
    const int t0 = i * kCh, n = min(kCh, T - t0);
    const size_t row0 = (size_t)bh * T + t0, cb = ((size_t)bh * nch + i) * kCh * kCh;
    rows_async<DK, PH>(sm.k, k + row0 * DK, n, tid, 128);
    rows_async<DK, PH>(sm.b, b + row0 * DK, n, tid, 128);
    cols_async<DV>(sm.v, v + row0 * DV, c0, n, tid, 128);
    cc_async(sm.p2, P2w + cb, tid, 128);
    cp_commit();
  };
  float S[RT][2][4];
#pragma unroll
  for (int rt = 0; rt < RT; ++rt) {
    zero(S[rt]);
    if (S0)
      each(S[rt], 16 * (warp + 4 * rt), 0, lane,
           [&](int r, int c, float &x) { x = __ldg(S0 + ((size_t)bh * DK + r) * DV + c0 + c); });
  }
  issue_a(0);
  issue_b(0);
  for (int i = 0; i < nch; ++i) {
    const int t0 = i * kCh, n = min(kCh, T - t0);
    const size_t row0 = (size_t)bh * T + t0;
#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
      each(S[rt], 16 * (warp + 4 * rt), 0, lane, [&](int r, int c, float &x) { w16(sm.s, r, c) = x; });
    cp_wait<0>();
    __syncthreads();
    // ---- phase 1 (warp w, rows 16 w): U = W S + M V; R = Q S + P1 V
    float u[2][4], rr[2][4];
    zero(u);
    zero(rr);
    wmma(u, 16 * warp, 0, DK, [&](int m, int kk) { return tf(fw<DK>(sm.w, m, kk)); },
         [&](int kk, int nn) { return tf(w16(sm.s, kk, nn)); }, lane);
    wmma(u, 16 * warp, 0, kCh, [&](int m, int kk) { return tf(cc(sm.m, m, kk)); },
         [&](int kk, int nn) { return bfbits(sm.v + kk * kPh + nn); }, lane);
    wmma(rr, 16 * warp, 0, DK, [&](int m, int kk) { return bfbits(sm.q + m * PH + kk); },
         [&](int kk, int nn) { return tf(w16(sm.s, kk, nn)); }, lane);
    wmma(rr, 16 * warp, 0, kCh, [&](int m, int kk) { return tf(cc(sm.p1, m, kk)); },
         [&](int kk, int nn) { return bfbits(sm.v + kk * kPh + nn); }, lane);
    each(u, 16 * warp, 0, lane, [&](int r, int c, float &x) { w16(sm.u, r, c) = x; });
    __syncthreads();
    if (i + 1 < nch) issue_a(i + 1);
    // ---- phase 2: O = R - P2 U; S += K^T V - B^T U
    wmma(rr, 16 * warp, 0, kCh, [&](int m, int kk) { return tf(-cc(sm.p2, m, kk)); },
         [&](int kk, int nn) { return tf(w16(sm.u, kk, nn)); }, lane);
    each(rr, 16 * warp, 0, lane, [&](int r, int c, float &x) {
      if (r < n) o[(row0 + r) * DV + c0 + c] = __float2bfloat16_rn(x);
    });
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
      const int m0 = 16 * (warp + 4 * rt);
      wmma(S[rt], m0, 0, kCh, [&](int m, int kk) { return bfbits(sm.k + kk * PH + m); },
           [&](int kk, int nn) { return bfbits(sm.v + kk * kPh + nn); }, lane);
      wmma(S[rt], m0, 0, kCh, [&](int m, int kk) { return bfbits(sm.b + kk * PH + m); },
           [&](int kk, int nn) { return tf(-w16(sm.u, kk, nn)); }, lane);
    }
    __syncthreads();
    if (i + 1 < nch) issue_b(i + 1);
  }
  if (S_final) {
#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
      each(S[rt], 16 * (warp + 4 * rt), 0, lane,
           [&](int r, int c, float &x) { S_final[((size_t)bh * DK + r) * DV + c0 + c] = x; });
  }
}

template <class Smem, class K>
cudaError_t set_smem(K kernel) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem));
}

template <int DK, int DV>
int launch_typed(const GdeltaArgs &x, uint8_t *ws, cudaStream_t s) {
  using bf = __nv_bfloat16;
  const int BH = x.B * x.H, nch = (x.T + kCh - 1) / kCh;
  const size_t ncc = (size_t)BH * nch * kCh * kCh;
  float *Ww = reinterpret_cast<float *>(ws), *Mw = Ww + (size_t)BH * nch * kCh * DK, *P1w = Mw + ncc,
        *P2w = P1w + ncc;
  cudaError_t e = set_smem<GwPreSmem<DK>>(gdw_pre_kernel<DK>);
  if (e == cudaSuccess) e = set_smem<GwChainSmem<DK>>(gdw_chain_kernel<DK, DV>);
  if (e == cudaSuccess) {
    gdw_pre_kernel<DK><<<dim3(nch, BH), 128, sizeof(GwPreSmem<DK>), s>>>(
        static_cast<const bf *>(x.q), static_cast<const bf *>(x.k), static_cast<const bf *>(x.a),
        static_cast<const bf *>(x.b), x.T, Ww, Mw, P1w, P2w);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    gdw_chain_kernel<DK, DV><<<(unsigned)(BH * (DV / kCW)), 128, sizeof(GwChainSmem<DK>), s>>>(
        static_cast<const bf *>(x.q), static_cast<const bf *>(x.k), static_cast<const bf *>(x.v),
        static_cast<const bf *>(x.b), static_cast<bf *>(x.o), x.S0, x.S_final, x.T, Ww, Mw, P1w, P2w);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_error("la_chunk_fwd_gdelta: kernel launch failed: %s", cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  return LA_OK;
}

}  // namespace

size_t gdelta_wy_workspace_bytes(int BH, int T, int dk) {
  const size_t nch = (size_t)(T + kCh - 1) / kCh;
  return (size_t)BH * nch * ((size_t)kCh * dk + 3u * kCh * kCh) * sizeof(float);
}

int launch_gdelta_wy(const GdeltaArgs &x, void *workspace, cudaStream_t s) {
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  if (x.dk == 128 && x.dv == 128) return launch_typed<128, 128>(x, ws, s);
  if (x.dk == 128) return launch_typed<128, 64>(x, ws, s);
  if (x.dv == 128) return launch_typed<64, 128>(x, ws, s);
  return launch_typed<64, 64>(x, ws, s);
}

}  // namespace la
