// Two-phase chunk forward of the generalised delta rule ("Talk Linear
// Attention", section 7.1: an identity-plus-rank-one transition between
// linear-attention steps), key-major,
//
//   S_t = (I - b_t a_t^T) S_{t-1} + k_t v_t^T,   o_t = S_t^T q_t,
//
// bf16 inputs on bf16 warp MMAs (16 x 8 x 16, fp32 accumulate). Per chunk of
// C = 64 rows with incoming state
// S the retrieved values u_r = S_{r-1}^T a_r solve (I + L_ab) U = A S + L_ak V
// (L_ab[r,s] = a_r.b_s, L_ak[r,s] = a_r.k_s for s < r), so with
// T = (I + L_ab)^{-1}
//
//   U = W S + M V,           W = T A,  M = T L_ak
//   O = Q S + P1 V - P2 U,   P1 = lower(Q K^T), P2 = lower(Q B^T)
//   S <- S + K^T V - B^T U
//
// Phase 1 (gdw_pre_kernel, every chunk in parallel): P1, P2, L_ak, L_ab from
// two [Q; A] products, T from 16 x 16 diagonal blocks and three tf32 block
// levels, W and M; written to a workspace as bf16 operand images.
// Phase 2 (gdw_chain_kernel, per head and 16 value columns -- every value
// column of S evolves on its own): the chunks in order, S in registers (bf16
// copies of S^T and U^T feed the MMAs), v and the key rows as MMA operands
// through ldmatrix.trans, each chunk's tiles copied asynchronously while the
// previous chunk finishes.
// A tail chunk is padded with zero rows, which leaves every real row's result
// unchanged.
#include <cuda_bf16.h>

#include <cstdint>

#include "la_internal.h"
#include "la_warp_mma.cuh"

namespace la {
namespace {

using namespace wm;

constexpr int kCP = kCh + 8;   // row pitch (bf16) of C x C tiles
constexpr int kVP = kCW + 8;   // row pitch (bf16) of the chain's v tile

// Per-chunk workspace (bf16 images, dense rows): W [64][DK], M [64][64], P1 [64][64], P2 [64][64].
template <int DK>
struct GwOff {
  static constexpr size_t w = 0, m = (size_t)kCh * DK * 2, p1 = m + kCh * kCh * 2, p2 = p1 + kCh * kCh * 2,
                          bytes = p2 + kCh * kCh * 2;
};

// ============================================================ phase 1
// q and k are dead once the products are taken, b once the products are taken:
// L_ab (later T as bf16) and L_ak take the place of q and k, T that of b.
template <int DK>
struct GwPreSmem {
  static constexpr int PH = Pitch<DK>::h;
  __nv_bfloat16 a[kCh * PH];
  union {
    __nv_bfloat16 qk[2 * kCh * PH];
    struct {
      union {
        float lab[kCh * wy::kAp];  // L_ab (tf32) for the blocked solve
        __nv_bfloat16 tb[kCh * kCP];  // then T as a bf16 operand
      };
      __nv_bfloat16 lak[kCh * kCP];
    } s;
  } u1;
  union {
    __nv_bfloat16 b[kCh * PH];
    float tf[kCh * wy::kAp];
  } u2;
};

template <int DK>
__global__ void __launch_bounds__(128) gdw_pre_kernel(const __nv_bfloat16 *__restrict__ q,
                                                      const __nv_bfloat16 *__restrict__ k,
                                                      const __nv_bfloat16 *__restrict__ a,
                                                      const __nv_bfloat16 *__restrict__ b, int T,
                                                      uint8_t *__restrict__ ws) {
  constexpr int PH = Pitch<DK>::h;
  using O = GwOff<DK>;
  using bf16 = __nv_bfloat16;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  GwPreSmem<DK> &sm = *reinterpret_cast<GwPreSmem<DK> *>(smem_raw);
  bf16 *const sq = sm.u1.qk, *const sk = sm.u1.qk + kCh * PH;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = blockIdx.x, bh = blockIdx.y, nch = gridDim.x;
  const int t0 = i * kCh, n = min(kCh, T - t0);
  const size_t row0 = (size_t)bh * T + t0;
  uint8_t *wc = ws + ((size_t)bh * nch + i) * O::bytes;
  rows_async<DK, PH>(sq, q + row0 * DK, n, tid, 128);
  rows_async<DK, PH>(sk, k + row0 * DK, n, tid, 128);
  rows_async<DK, PH>(sm.a, a + row0 * DK, n, tid, 128);
  rows_async<DK, PH>(sm.u2.b, b + row0 * DK, n, tid, 128);
  cp_commit();
  cp_wait<0>();
  __syncthreads();
  // [Q; A] K^T and [Q; A] B^T: warps 0, 1 the rows of Q (P1, P2, stored at once),
  // warps 2, 3 the rows of A (L_ak, L_ab, held until every warp is done with q, k, b)
  const bf16 *src = warp < 2 ? sq : sm.a;
  const int rbase = (warp & 1) * 32;
  float lacc[2][2][8][4];
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const bf16 *rhs = pass == 0 ? sk : sm.u2.b;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      zero(lacc[pass][h]);
      wmma16(lacc[pass][h], rbase + 16 * h, 0, DK, src, PH, rhs, PH, lane);
      if (warp < 2) {
        __nv_bfloat162 *P = reinterpret_cast<__nv_bfloat162 *>(wc + (pass == 0 ? O::p1 : O::p2));
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = rbase + 16 * h + g, s = 8 * j + 2 * t;
          const float *x = lacc[pass][h][j];
          P[(r * kCh + s) >> 1] = __floats2bfloat162_rn(s <= r ? x[0] : 0.f, s + 1 <= r ? x[1] : 0.f);
          P[((r + 8) * kCh + s) >> 1] =
              __floats2bfloat162_rn(s <= r + 8 ? x[2] : 0.f, s + 1 <= r + 8 ? x[3] : 0.f);
        }
      }
    }
  }
  __syncthreads();
  if (warp >= 2) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      each(lacc[0][h], rbase + 16 * h, 0, lane,
           [&](int r, int s, float &x) { sm.u1.s.lak[r * kCP + s] = __float2bfloat16_rn(s < r ? x : 0.f); });
      each(lacc[1][h], rbase + 16 * h, 0, lane,
           [&](int r, int s, float &x) { sm.u1.s.lab[r * wy::kAp + s] = s < r ? wy::round_tf32(x) : 0.f; });
    }
  }
  __syncthreads();
  // T = (I + L_ab)^{-1}: 16 x 16 diagonal blocks, then three block levels (tf32 warp MMAs)
  float *const lab = sm.u1.s.lab, *const tf = sm.u2.tf;
  if (tid < kCh) wy::diag_inverse_16(lab, tf, tid >> 4, tid & 15);
  __syncthreads();
#pragma unroll 1
  for (int lvl = 1; lvl < 4; ++lvl) {
    if (warp < 4 - lvl) {
      const int ib = warp + lvl, jb = warp;
      float a2[2][4] = {};
      for (int kb = jb; kb < ib; ++kb)
        wy::block_mma_16(a2, lab + ib * 16 * wy::kAp + kb * 16, tf + kb * 16 * wy::kAp + jb * 16, lane);
      float *Tij = tf + ib * 16 * wy::kAp + jb * 16;
      wy::block_store_16(Tij, a2, 1.f, lane);
      __syncwarp();
      float a3[2][4] = {};
      wy::block_mma_16(a3, tf + ib * 16 * wy::kAp + ib * 16, Tij, lane);
      __syncwarp();
      wy::block_store_16(Tij, a3, -1.f, lane);
    }
    __syncthreads();
  }
  // T as bf16 (zero above the diagonal) in place of L_ab: thread tid owns row tid / 2, columns 32 (tid % 2) ..
  {
    const int r = tid >> 1, c0 = (tid & 1) * 32;
    bf16 *tb = sm.u1.s.tb;
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const int sc = c0 + e;
      const float x0 = sc <= r ? tf[r * wy::kAp + sc] : 0.f, x1 = sc + 1 <= r ? tf[r * wy::kAp + sc + 1] : 0.f;
      *reinterpret_cast<__nv_bfloat162 *>(tb + r * kCP + sc) = __floats2bfloat162_rn(x0, x1);
    }
  }
  __syncthreads();
  // W = T A (64 x DK), M = T L_ak (64 x 64): warp w, rows 16 w; B operands through ldmatrix.trans
  const int g = lane >> 2, t = lane & 3;
  {
    float acc[DK / 8][4];
    zero(acc);
    wmma16_bt(acc, 16 * warp, 0, kCh, sm.u1.s.tb, kCP, sm.a, PH, lane);
    __nv_bfloat162 *W = reinterpret_cast<__nv_bfloat162 *>(wc + O::w);
#pragma unroll
    for (int j = 0; j < DK / 8; ++j) {
      const int r = 16 * warp + g, c = 8 * j + 2 * t;
      W[(r * DK + c) >> 1] = __floats2bfloat162_rn(acc[j][0], acc[j][1]);
      W[((r + 8) * DK + c) >> 1] = __floats2bfloat162_rn(acc[j][2], acc[j][3]);
    }
  }
  {
    float acc[8][4];
    zero(acc);
    wmma16_bt(acc, 16 * warp, 0, kCh, sm.u1.s.tb, kCP, sm.u1.s.lak, kCP, lane);
    __nv_bfloat162 *M = reinterpret_cast<__nv_bfloat162 *>(wc + O::m);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = 16 * warp + g, c = 8 * j + 2 * t;
      M[(r * kCh + c) >> 1] = __floats2bfloat162_rn(acc[j][0], acc[j][1]);
      M[((r + 8) * kCh + c) >> 1] = __floats2bfloat162_rn(acc[j][2], acc[j][3]);
    }
  }
}

// ============================================================ phase 2
// One chunk's tiles; NB = 2 keeps two of them, so that chunk i + 1's copies run
// during all of chunk i.
template <int DK>
struct GwTiles {
  __nv_bfloat16 q[kCh * Pitch<DK>::h], k[kCh * Pitch<DK>::h], b[kCh * Pitch<DK>::h], w[kCh * Pitch<DK>::h];
  __nv_bfloat16 m[kCh * kCP], p1[kCh * kCP], p2[kCh * kCP], v[kCh * kVP];
};
template <int DK, int NB>
struct GwChainSmem {
  GwTiles<DK> x[NB];
  __nv_bfloat16 st[kCW * Pitch<DK>::h], ut[kCW * kCP];
};

template <int DK, int DV, int NB>
__global__ void __launch_bounds__(128) gdw_chain_kernel(
    const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
    const __nv_bfloat16 *__restrict__ b, __nv_bfloat16 *__restrict__ o, const float *__restrict__ S0,
    float *__restrict__ S_final, int T, const uint8_t *__restrict__ ws) {
  constexpr int PH = Pitch<DK>::h, NCB = DV / kCW, RT = DK / 64;
  using O = GwOff<DK>;
  using bf16 = __nv_bfloat16;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  GwChainSmem<DK, NB> &sm = *reinterpret_cast<GwChainSmem<DK, NB> *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x / NCB, c0 = (blockIdx.x % NCB) * kCW;
  const int nch = (T + kCh - 1) / kCh;
  const int g = lane >> 2, t = lane & 3;
  // group A (q, W, M, P1) is read in phase 1 only, group B (k, b, v, P2) in phase 2
  auto issue_a = [&](int i, GwTiles<DK> &x) {
    const int t0 = i * kCh, n = min(kCh, T - t0);
    const size_t row0 = (size_t)bh * T + t0;
    const uint8_t *wc = ws + ((size_t)bh * nch + i) * O::bytes;
    rows_async<DK, PH>(x.q, q + row0 * DK, n, tid, 128);
    rows_async<DK, PH>(x.w, reinterpret_cast<const bf16 *>(wc + O::w), kCh, tid, 128);
    rows_async<kCh, kCP>(x.m, reinterpret_cast<const bf16 *>(wc + O::m), kCh, tid, 128);
    rows_async<kCh, kCP>(x.p1, reinterpret_cast<const bf16 *>(wc + O::p1), kCh, tid, 128);
    cp_commit();
  };
  auto issue_b = [&](int i, GwTiles<DK> &x) {
    const int t0 = i * kCh, n = min(kCh, T - t0);
    const size_t row0 = (size_t)bh * T + t0;
    const uint8_t *wc = ws + ((size_t)bh * nch + i) * O::bytes;
    rows_async<DK, PH>(x.k, k + row0 * DK, n, tid, 128);
    rows_async<DK, PH>(x.b, b + row0 * DK, n, tid, 128);
    for (int e = tid; e < kCh * 2; e += 128) {
      const int r = e >> 1, c = (e & 1) * 8;
      const bool ok = r < n;
      cpa16(x.v + r * kVP + c, v + (ok ? (row0 + r) * DV + c0 + c : 0), ok);
    }
    rows_async<kCh, kCP>(x.p2, reinterpret_cast<const bf16 *>(wc + O::p2), kCh, tid, 128);
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
  issue_a(0, sm.x[0]);
  issue_b(0, sm.x[0]);
  for (int i = 0; i < nch; ++i) {
    const int t0 = i * kCh, n = min(kCh, T - t0);
    const size_t row0 = (size_t)bh * T + t0;
    GwTiles<DK> &x = sm.x[NB == 2 ? (i & 1) : 0];
    const bool more = i + 1 < nch;
    // NB = 2: the next chunk's copies go out now, into the buffer the previous chunk used
    if (NB == 2 && more) {
      issue_a(i + 1, sm.x[(i + 1) & 1]);
      issue_b(i + 1, sm.x[(i + 1) & 1]);
    }
    // S^T as bf16 (value column, key channel) for the MMAs
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
      const int m0 = 16 * (warp + 4 * rt);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int c = 8 * j + 2 * t;
        sm.st[c * PH + m0 + g] = __float2bfloat16_rn(S[rt][j][0]);
        sm.st[(c + 1) * PH + m0 + g] = __float2bfloat16_rn(S[rt][j][1]);
        sm.st[c * PH + m0 + g + 8] = __float2bfloat16_rn(S[rt][j][2]);
        sm.st[(c + 1) * PH + m0 + g + 8] = __float2bfloat16_rn(S[rt][j][3]);
      }
    }
    if (NB == 2 && more)
      cp_wait<2>();
    else
      cp_wait<0>();
    __syncthreads();
    // ---- phase 1 (warp w, rows 16 w): U = W S + M V; R = Q S + P1 V
    float u[2][4], rr[2][4];
    zero(u);
    zero(rr);
    wmma16(u, 16 * warp, 0, DK, x.w, PH, sm.st, PH, lane);
    wmma16_bt(u, 16 * warp, 0, kCh, x.m, kCP, x.v, kVP, lane);
    wmma16(rr, 16 * warp, 0, DK, x.q, PH, sm.st, PH, lane);
    wmma16_bt(rr, 16 * warp, 0, kCh, x.p1, kCP, x.v, kVP, lane);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int c = 8 * j + 2 * t, r = 16 * warp + g;
      sm.ut[c * kCP + r] = __float2bfloat16_rn(u[j][0]);
      sm.ut[(c + 1) * kCP + r] = __float2bfloat16_rn(u[j][1]);
      sm.ut[c * kCP + r + 8] = __float2bfloat16_rn(u[j][2]);
      sm.ut[(c + 1) * kCP + r + 8] = __float2bfloat16_rn(u[j][3]);
    }
    __syncthreads();
    if (NB == 1 && more) issue_a(i + 1, x);
    // ---- phase 2: O = R - P2 U; S += K^T V - B^T U
    wmma16<2, true>(rr, 16 * warp, 0, kCh, x.p2, kCP, sm.ut, kCP, lane);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int r = 16 * warp + g, c = c0 + 8 * j + 2 * t;
      if (r < n)
        *reinterpret_cast<__nv_bfloat162 *>(o + (row0 + r) * DV + c) = __floats2bfloat162_rn(rr[j][0], rr[j][1]);
      if (r + 8 < n)
        *reinterpret_cast<__nv_bfloat162 *>(o + (row0 + r + 8) * DV + c) =
            __floats2bfloat162_rn(rr[j][2], rr[j][3]);
    }
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
      const int m0 = 16 * (warp + 4 * rt);
      wmma16_atbt(S[rt], m0, 0, kCh, x.k, PH, x.v, kVP, lane);
      wmma16_at<2, true>(S[rt], m0, 0, kCh, x.b, PH, sm.ut, kCP, lane);
    }
    __syncthreads();
    if (NB == 1 && more) issue_b(i + 1, x);
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

template <int DK, int DV, int NB>
cudaError_t launch_chain(const GdeltaArgs &x, const uint8_t *ws, cudaStream_t s) {
  using bf = __nv_bfloat16;
  const int BH = x.B * x.H;
  cudaError_t e = set_smem<GwChainSmem<DK, NB>>(gdw_chain_kernel<DK, DV, NB>);
  if (e != cudaSuccess) return e;
  gdw_chain_kernel<DK, DV, NB><<<(unsigned)(BH * (DV / kCW)), 128, sizeof(GwChainSmem<DK, NB>), s>>>(
      static_cast<const bf *>(x.q), static_cast<const bf *>(x.k), static_cast<const bf *>(x.v),
      static_cast<const bf *>(x.b), static_cast<bf *>(x.o), x.S0, x.S_final, x.T, ws);
  return cudaGetLastError();
}

template <int DK, int DV>
int launch_typed(const GdeltaArgs &x, uint8_t *ws, cudaStream_t s) {
  using bf = __nv_bfloat16;
  const int BH = x.B * x.H, nch = (x.T + kCh - 1) / kCh;
  cudaError_t e = set_smem<GwPreSmem<DK>>(gdw_pre_kernel<DK>);
  if (e == cudaSuccess) {
    gdw_pre_kernel<DK><<<dim3(nch, BH), 128, sizeof(GwPreSmem<DK>), s>>>(
        static_cast<const bf *>(x.q), static_cast<const bf *>(x.k), static_cast<const bf *>(x.a),
        static_cast<const bf *>(x.b), x.T, ws);
    e = cudaGetLastError();
  }
  // the chain: double-buffered (one CTA an SM) when the grid fits on the SMs once,
  // else single-buffered (two CTAs an SM)
  if (e == cudaSuccess) {
    const long long grid = (long long)BH * (DV / kCW), sms = sm_count();
    e = grid <= sms ? launch_chain<DK, DV, 2>(x, ws, s) : launch_chain<DK, DV, 1>(x, ws, s);
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
  return (size_t)BH * nch * (dk == 128 ? GwOff<128>::bytes : GwOff<64>::bytes);
}

int launch_gdelta_wy(const GdeltaArgs &x, void *workspace, cudaStream_t s) {
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  if (x.dk == 128 && x.dv == 128) return launch_typed<128, 128>(x, ws, s);
  if (x.dk == 128) return launch_typed<128, 64>(x, ws, s);
  if (x.dv == 128) return launch_typed<64, 128>(x, ws, s);
  return launch_typed<64, 64>(x, ws, s);
}

}  // namespace la
