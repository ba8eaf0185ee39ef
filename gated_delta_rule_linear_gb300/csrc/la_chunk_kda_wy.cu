// Two-phase chunk forward of Kimi Delta Attention ("LLM attention
// optimisation" page, Kimi Delta Attention section: Gated DeltaNet with a
// per-key-channel gate), key-major,
//
//   S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,  o_t = S_t^T q_t,
//
// bf16 inputs, fp32 state, on bf16 warp MMAs (16 x 8 x 16, fp32 accumulate;
// the solve's block levels in tf32). Per chunk of C = 64 rows with
// the per-channel inclusive prefix B[r][c] of the log-gates, its midpoint row
// b_m[c] = B[31][c] and its last row B_L[c], the WY/UT form ("Talk Linear
// Attention" section 6.2) with the decay folded per channel is
//
//   A = Diag(beta) strict_lower(K+ K-^T),  T = (I + A)^{-1},  T' = T Diag(beta)
//   W = T' (K ⊙ e^B),  U = T' V - W S
//   O = (Q ⊙ e^B) S + P U,  P = lower(Q+ K-^T)
//   S <- Diag(e^{B_L}) S + (K ⊙ e^{B_L - B})^T U
//
// with Q+ = Q ⊙ e^{B - b_m}, K+ = K ⊙ e^{B - b_m}, K- = K ⊙ e^{b_m - B} (so
// that Q+ K-^T carries e^{B_r - B_s} channel by channel without forming it;
// a cumulative log-gate above ~80 within half a chunk overflows the fold, as
// in the fused kernels).
//
// Phase 1 (kdw_pre_kernel, every chunk in parallel): the prefix, the folded
// operands (bf16, as the fused kernels use them), A and P from one
// [Q+; K+] K-^T product, T by substitution, T', W;
// written to a workspace as bf16 operands (with Q ⊙ e^B and K ⊙ e^{B_L - B})
// and e^{B_L}. Phase 2 (kdw_chain_kernel, per head and 64 value columns -- each value
// column of S evolves on its own): the chunks in order, S in registers, eight
// warps (four row strips x two 32-column halves) sharing one copy of each
// chunk's images, the next chunk's tiles copied during the whole of the
// current one (two buffers). A tail chunk is
// padded with zero rows and zero gates, which leaves every real row's result
// unchanged.
#include <cuda_bf16.h>

#include <cstdint>

#include "la_internal.h"
#include "la_warp_mma.cuh"

namespace la {
namespace {

using namespace wm;

constexpr int kMid = kCh / 2 - 1;  // the fold's midpoint row
constexpr int kVW = 64;            // value columns per chain CTA (two halves of 32)
constexpr int kVP = kVW + 8;       // row pitch (bf16) of the chain's v tile
constexpr int kCP = kCh + 8;       // row pitch (bf16) of its C x C tiles

// Per-chunk workspace, in this order (bf16 operands, as the fused kernels use):
// T' [64][64], W [64][DK], P [64][64], Q e^B [64][DK], K e^{B_L - B} [64][DK]
// (all bf16, dense rows), e^{B_L} [DK] f32.
template <int DK>
struct KwOff {
  static constexpr size_t tp = 0, w = tp + kCh * kCh * 2, p = w + (size_t)kCh * DK * 2,
                          qt = p + kCh * kCh * 2, kt = qt + (size_t)kCh * DK * 2, gl = kt + (size_t)kCh * DK * 2,
                          bytes = gl + (size_t)DK * 4;
};

// ============================================================ phase 1
// One CTA per chunk, 128 threads, three operand tiles of shared memory (~53 KB
// at dk = 128: four CTAs per SM): a thread per key channel forms the channel's
// prefix in registers and folds Q and K in place (Q+, K+) and into K-; the
// products run on the bf16 operand tiles; T comes from 16 x 16 diagonal blocks
// and three block levels on tf32 warp MMAs (la_wy.cuh). Once the products are
// taken, A (held in registers across the barrier) replaces K-, T replaces Q+,
// and T' as bf16 replaces A.
template <int DK>
struct KwPreSmem {
  union {
    __nv_bfloat16 qp[kCh * Pitch<DK>::h];  // Q, folded in place into Q+
    float tf[kCh * wy::kAp];               // then T
  } r1;
  __nv_bfloat16 kp[kCh * Pitch<DK>::h];  // K, folded in place into K+
  union {
    __nv_bfloat16 km[kCh * Pitch<DK>::h];  // K-
    float af[kCh * wy::kAp];               // then A
    __nv_bfloat16 tpb[kCh * kCP];          // then T' (bf16), the W product's A operand
  } r3;
  float bet[kCh], bm[DK];
  float gsum[(128 / (DK / 2)) * DK];  // the fold's row groups' gate sums per key channel
};

template <int DK>
__global__ void __launch_bounds__(128, 4) kdw_pre_kernel(const __nv_bfloat16 *__restrict__ q,
                                                         const __nv_bfloat16 *__restrict__ k,
                                                         const float *__restrict__ g, const float *__restrict__ beta,
                                                         int T, uint8_t *__restrict__ ws) {
  constexpr int PH = Pitch<DK>::h;
  using O = KwOff<DK>;
  using bf16 = __nv_bfloat16;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  KwPreSmem<DK> &sm = *reinterpret_cast<KwPreSmem<DK> *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int i = blockIdx.x, bh = blockIdx.y, nch = gridDim.x;
  const int t0 = i * kCh, n = min(kCh, T - t0);
  const size_t row0 = (size_t)bh * T + t0;
  uint8_t *wc = ws + ((size_t)bh * nch + i) * O::bytes;
  rows_async<DK, PH>(sm.r1.qp, q + row0 * DK, n, tid, 128);
  rows_async<DK, PH>(sm.kp, k + row0 * DK, n, tid, 128);
  cp_commit();
  if (tid < kCh) sm.bet[tid] = tid < n ? (beta ? __ldg(beta + row0 + tid) : 1.f) : 0.f;
  // ---- the fold: thread tid owns the key-channel pair (2 cp, 2 cp + 1) and RPG consecutive
  //      rows; the prefix B[.][c] of its rows in registers, then the row groups' sums
  constexpr int NP = DK / 2, RG = 128 / NP, RPG = kCh / RG;
  const int cp = tid % NP, grp = tid / NP, r0 = grp * RPG, c = 2 * cp;
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
  cp_wait<0>();
  __syncthreads();
  // ---- folded rows: Q+, K+ (in place), K- (tiles), Q e^B and K e^{B_L - B} (workspace), e^{B_L}
  {
    float2 off = make_float2(0.f, 0.f), bmid = off, bl = off;
#pragma unroll
    for (int j = 0; j < RG; ++j) {
      const float x0 = sm.gsum[j * DK + c], x1 = sm.gsum[j * DK + c + 1];
      if (j < grp) {
        off.x += x0;
        off.y += x1;
      }
      if (j * RPG <= kMid) {  // the groups of rows 0 .. kMid
        bmid.x += x0;
        bmid.y += x1;
      }
      bl.x += x0;
      bl.y += x1;
    }
    if (grp == 0) {
      sm.bm[c] = bmid.x;
      sm.bm[c + 1] = bmid.y;
      *reinterpret_cast<float2 *>(wc + O::gl + 4 * c) = make_float2(__expf(bl.x), __expf(bl.y));
    }
    const float2 ebm = make_float2(__expf(bmid.x), __expf(bmid.y));
    const float2 eblm = make_float2(__expf(bl.x - bmid.x), __expf(bl.y - bmid.y));
    __nv_bfloat162 *qt = reinterpret_cast<__nv_bfloat162 *>(wc + O::qt),
                   *kt = reinterpret_cast<__nv_bfloat162 *>(wc + O::kt);
#pragma unroll
    for (int r = 0; r < RPG; ++r) {
      const int R = r0 + r;
      const float2 qx = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(sm.r1.qp + R * PH + c));
      const float2 kx = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(sm.kp + R * PH + c));
      const float d0 = off.x + bc[r].x - bmid.x, d1 = off.y + bc[r].y - bmid.y;
      const float ep0 = __expf(d0), ep1 = __expf(d1), em0 = __expf(-d0), em1 = __expf(-d1);
      *reinterpret_cast<__nv_bfloat162 *>(sm.r1.qp + R * PH + c) = __floats2bfloat162_rn(qx.x * ep0, qx.y * ep1);
      *reinterpret_cast<__nv_bfloat162 *>(sm.kp + R * PH + c) = __floats2bfloat162_rn(kx.x * ep0, kx.y * ep1);
      *reinterpret_cast<__nv_bfloat162 *>(sm.r3.km + R * PH + c) = __floats2bfloat162_rn(kx.x * em0, kx.y * em1);
      // e^B = EP e^{b_m}, e^{B_L - B} = EM e^{B_L - b_m}
      qt[(R * DK + c) >> 1] = __floats2bfloat162_rn(qx.x * (ep0 * ebm.x), qx.y * (ep1 * ebm.y));
      kt[(R * DK + c) >> 1] = __floats2bfloat162_rn(kx.x * (em0 * eblm.x), kx.y * (em1 * eblm.y));
    }
  }
  __syncthreads();
  // ---- [Q+; K+] K-^T: warps 0, 1 the rows of Q+ (P, stored at once), warps 2, 3 the
  //      rows of K+ (A, held until every warp is done with K-)
  const int rbase = (warp & 1) * 32;
  float acc[2][8][4];
  {
    const bf16 *src = warp < 2 ? sm.r1.qp : sm.kp;
    __nv_bfloat162 *P = reinterpret_cast<__nv_bfloat162 *>(wc + O::p);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      zero(acc[h]);
      wmma16(acc[h], rbase + 16 * h, 0, DK, src, PH, sm.r3.km, PH, lane);
      if (warp < 2) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = rbase + 16 * h + gq, sc = 8 * j + 2 * tq;
          const float *x = acc[h][j];
          P[(r * kCh + sc) >> 1] = __floats2bfloat162_rn(sc <= r ? x[0] : 0.f, sc + 1 <= r ? x[1] : 0.f);
          P[((r + 8) * kCh + sc) >> 1] =
              __floats2bfloat162_rn(sc <= r + 8 ? x[2] : 0.f, sc + 1 <= r + 8 ? x[3] : 0.f);
        }
      }
    }
  }
  __syncthreads();
  if (warp >= 2) {  // rounded to tf32 for the block MMAs of the solve
#pragma unroll
    for (int h = 0; h < 2; ++h)
      each(acc[h], rbase + 16 * h, 0, lane, [&](int r, int s, float &x) {
        sm.r3.af[r * wy::kAp + s] = s < r ? wy::round_tf32(sm.bet[r] * x) : 0.f;
      });
  }
  __syncthreads();
  // ---- T = (I + A)^{-1}: 16 x 16 diagonal blocks by forward substitution, then the
  //      off-diagonal blocks in three levels, T_ij = -T_ii sum_{j<=k<i} A_ik T_kj
  float *Af = sm.r3.af, *Tf = sm.r1.tf;
  if (tid < kCh) wy::diag_inverse_16(Af, Tf, tid >> 4, tid & 15);
  __syncthreads();
#pragma unroll 1
  for (int lvl = 1; lvl < 4; ++lvl) {
    if (warp < 4 - lvl) {
      const int ib = warp + lvl, jb = warp;
      float a2[2][4] = {};
      for (int kb = jb; kb < ib; ++kb)
        wy::block_mma_16(a2, Af + ib * 16 * wy::kAp + kb * 16, Tf + kb * 16 * wy::kAp + jb * 16, lane);
      float *Tij = Tf + ib * 16 * wy::kAp + jb * 16;
      wy::block_store_16(Tij, a2, 1.f, lane);
      __syncwarp();
      float a3[2][4] = {};
      wy::block_mma_16(a3, Tf + ib * 16 * wy::kAp + ib * 16, Tij, lane);
      __syncwarp();
      wy::block_store_16(Tij, a3, -1.f, lane);
    }
    __syncthreads();
  }
  // ---- T' = T Diag(beta) (zero above the diagonal) as bf16, to the workspace and, for the W
  //      product, in place of A (free since the last level): thread tid owns row tid / 2,
  //      columns 32 (tid % 2) .. + 31
  bf16 *tpb = sm.r3.tpb;
  {
    const int r = tid >> 1, c0 = (tid & 1) * 32;
    float x[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int sc = c0 + e;
      x[e] = sc <= r ? Tf[r * wy::kAp + sc] * sm.bet[sc] : 0.f;
    }
    __syncthreads();  // every thread has read its row of T before T' overwrites A
    bf16 *tp = reinterpret_cast<bf16 *>(wc + O::tp) + r * kCh + c0;
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(x[e], x[e + 1]);
      reinterpret_cast<__nv_bfloat162 *>(tp)[e >> 1] = h;
      *reinterpret_cast<__nv_bfloat162 *>(tpb + r * kCP + c0 + e) = h;
    }
  }
  __syncthreads();
  // ---- W = T' (K+ ⊙ e^{b_m}) = (T' K+) e^{b_m} per channel: warp w, rows 16 w
  {
    float wacc[DK / 8][4];
    zero(wacc);
    wmma16_bt(wacc, 16 * warp, 0, kCh, tpb, kCP, sm.kp, PH, lane);
    __nv_bfloat162 *W = reinterpret_cast<__nv_bfloat162 *>(wc + O::w);
#pragma unroll
    for (int j = 0; j < DK / 8; ++j) {
      const int r = 16 * warp + gq, c = 8 * j + 2 * tq;
      const float e0 = __expf(sm.bm[c]), e1 = __expf(sm.bm[c + 1]);
      W[(r * DK + c) >> 1] = __floats2bfloat162_rn(wacc[j][0] * e0, wacc[j][1] * e1);
      W[((r + 8) * DK + c) >> 1] = __floats2bfloat162_rn(wacc[j][2] * e0, wacc[j][3] * e1);
    }
  }
}

// ============================================================ phase 2
// bf16 m16n8k16 warp MMAs: S and U enter them as bf16 copies (S^T and U^T, k
// contiguous), the fp32 state stays in registers; the fragments of v (as B) and
// of K e^{B_L - B} (as the transposed A of the state update) come from
// ldmatrix.trans of their token-major tiles.
// One chunk's tiles of the chain; two of them, so that chunk i + 1's copies run
// during all of chunk i.
template <int DK>
struct KwTiles {
  float gl[DK];
  __nv_bfloat16 tp[kCh * kCP], p[kCh * kCP], w[kCh * Pitch<DK>::h], qt[kCh * Pitch<DK>::h],
      kt[kCh * Pitch<DK>::h], v[kCh * kVP];
};
template <int DK>
struct KwChainSmem {
  KwTiles<DK> x[2];
  __nv_bfloat16 st[kVW * Pitch<DK>::h], ut[kVW * kCP];
};

template <int DK, int DV>
__global__ void __launch_bounds__(256) kdw_chain_kernel(const __nv_bfloat16 *__restrict__ v,
                                                        __nv_bfloat16 *__restrict__ o, const float *__restrict__ S0,
                                                        float *__restrict__ S_final, int T,
                                                        const uint8_t *__restrict__ ws) {
  constexpr int PH = Pitch<DK>::h, NCB = DV / kVW, RT = DK / 64;
  using O = KwOff<DK>;
  using bf16 = __nv_bfloat16;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  KwChainSmem<DK> &sm = *reinterpret_cast<KwChainSmem<DK> *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rh = warp & 3, n0 = (warp >> 2) * 32;  // the warp's row strip and column half
  const int bh = blockIdx.x / NCB, c0 = (blockIdx.x % NCB) * kVW;
  const int nch = (T + kCh - 1) / kCh;
  // one chunk's tiles, one commit group
  auto issue = [&](int i, KwTiles<DK> &x) {
    const uint8_t *wc = ws + ((size_t)bh * nch + i) * O::bytes;
    const int t0 = i * kCh, n = min(kCh, T - t0);
    rows_async<kCh, kCP>(x.tp, reinterpret_cast<const bf16 *>(wc + O::tp), kCh, tid, 256);
    rows_async<DK, PH>(x.w, reinterpret_cast<const bf16 *>(wc + O::w), kCh, tid, 256);
    rows_async<DK, PH>(x.qt, reinterpret_cast<const bf16 *>(wc + O::qt), kCh, tid, 256);
    rows_async<kCh, kCP>(x.p, reinterpret_cast<const bf16 *>(wc + O::p), kCh, tid, 256);
    rows_async<DK, PH>(x.kt, reinterpret_cast<const bf16 *>(wc + O::kt), kCh, tid, 256);
    for (int e = tid; e < DK / 4; e += 256) cpa16(x.gl + 4 * e, wc + O::gl + 16 * e, true);
    const bf16 *vs = v + ((size_t)bh * T + t0) * DV + c0;
    for (int e = tid; e < kCh * (kVW / 8); e += 256) {
      const int r = e / (kVW / 8), c = (e % (kVW / 8)) * 8;
      const bool ok = r < n;
      cpa16(x.v + r * kVP + c, vs + (ok ? (size_t)r * DV + c : 0), ok);
    }
    cp_commit();
  };
  // S[:, c0 + n0 .. + 32) in registers: row tiles rh + 4 rt, four 8-column tiles
  float S[RT][4][4];
#pragma unroll
  for (int rt = 0; rt < RT; ++rt) {
    zero(S[rt]);
    if (S0)
      each(S[rt], 16 * (rh + 4 * rt), n0, lane,
           [&](int r, int c, float &x) { x = __ldg(S0 + ((size_t)bh * DK + r) * DV + c0 + c); });
  }
  issue(0, sm.x[0]);
  const int g = lane >> 2, t = lane & 3;
  for (int i = 0; i < nch; ++i) {
    const int t0 = i * kCh, n = min(kCh, T - t0);
    const size_t row0 = (size_t)bh * T + t0;
    KwTiles<DK> &x = sm.x[i & 1];
    const bool more = i + 1 < nch;
    // the buffer chunk i - 1 used is free (the barrier that ended it)
    if (more) issue(i + 1, sm.x[(i + 1) & 1]);
    // S^T as bf16 (value column, key channel)
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
      const int m0 = 16 * (rh + 4 * rt);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = n0 + 8 * j + 2 * t;
        sm.st[c * PH + m0 + g] = __float2bfloat16_rn(S[rt][j][0]);
        sm.st[(c + 1) * PH + m0 + g] = __float2bfloat16_rn(S[rt][j][1]);
        sm.st[c * PH + m0 + g + 8] = __float2bfloat16_rn(S[rt][j][2]);
        sm.st[(c + 1) * PH + m0 + g + 8] = __float2bfloat16_rn(S[rt][j][3]);
      }
    }
    if (more)
      cp_wait<1>();
    else
      cp_wait<0>();
    __syncthreads();
    // ---- phase 1 (rows 16 rh, columns n0 ..): U = T' V - W S; R = (Q ⊙ e^B) S
    float u[4][4], rr[4][4];
    zero(u);
    zero(rr);
    wmma16_bt(u, 16 * rh, n0, kCh, x.tp, kCP, x.v, kVP, lane);
    wmma16<4, true>(u, 16 * rh, n0, DK, x.w, PH, sm.st, PH, lane);
    wmma16(rr, 16 * rh, n0, DK, x.qt, PH, sm.st, PH, lane);
    // U^T as bf16 for the phase-2 MMAs (value column, token)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = n0 + 8 * j + 2 * t, r = 16 * rh + g;
      sm.ut[c * kCP + r] = __float2bfloat16_rn(u[j][0]);
      sm.ut[(c + 1) * kCP + r] = __float2bfloat16_rn(u[j][1]);
      sm.ut[c * kCP + r + 8] = __float2bfloat16_rn(u[j][2]);
      sm.ut[(c + 1) * kCP + r + 8] = __float2bfloat16_rn(u[j][3]);
    }
    __syncthreads();
    // ---- phase 2: O = R + P U; S <- Diag(e^{B_L}) S + (K ⊙ e^{B_L - B})^T U
    wmma16(rr, 16 * rh, n0, kCh, x.p, kCP, sm.ut, kCP, lane);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = 16 * rh + g, c = c0 + n0 + 8 * j + 2 * t;
      if (r < n)
        *reinterpret_cast<__nv_bfloat162 *>(o + (row0 + r) * DV + c) = __floats2bfloat162_rn(rr[j][0], rr[j][1]);
      if (r + 8 < n)
        *reinterpret_cast<__nv_bfloat162 *>(o + (row0 + r + 8) * DV + c) =
            __floats2bfloat162_rn(rr[j][2], rr[j][3]);
    }
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
      const int m0 = 16 * (rh + 4 * rt);
      each(S[rt], m0, n0, lane, [&](int r, int, float &y) { y *= x.gl[r]; });
      wmma16_at(S[rt], m0, n0, kCh, x.kt, PH, sm.ut, kCP, lane);
    }
    __syncthreads();
  }
  if (S_final) {
#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
      each(S[rt], 16 * (rh + 4 * rt), n0, lane,
           [&](int r, int c, float &y) { S_final[((size_t)bh * DK + r) * DV + c0 + c] = y; });
  }
}

template <class Smem, class K>
cudaError_t set_smem(K kernel) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem));
}

template <int DK, int DV>
int launch_typed(const ChunkParams &p, uint8_t *ws, cudaStream_t s) {
  using bf16 = __nv_bfloat16;
  const int BH = p.B * p.H, nch = (p.T + kCh - 1) / kCh;
  cudaError_t e = set_smem<KwPreSmem<DK>>(kdw_pre_kernel<DK>);
  if (e == cudaSuccess) e = set_smem<KwChainSmem<DK>>(kdw_chain_kernel<DK, DV>);
  if (e == cudaSuccess) {
    kdw_pre_kernel<DK><<<dim3(nch, BH), 128, sizeof(KwPreSmem<DK>), s>>>(
        static_cast<const bf16 *>(p.q), static_cast<const bf16 *>(p.k), p.g, p.beta, p.T, ws);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    kdw_chain_kernel<DK, DV><<<(unsigned)(BH * (DV / kVW)), 256, sizeof(KwChainSmem<DK>), s>>>(
        static_cast<const bf16 *>(p.v), static_cast<bf16 *>(p.o), p.S0, p.S_final, p.T, ws);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_error("la_chunk_fwd: LA_KDA kernel launch failed: %s", cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  return LA_OK;
}

}  // namespace

size_t kda_wy_workspace_bytes(const ChunkParams &p) {
  const size_t nch = (size_t)(p.T + kCh - 1) / kCh, BH = (size_t)p.B * p.H;
  return BH * nch * (p.dk == 128 ? KwOff<128>::bytes : KwOff<64>::bytes);
}

int launch_kda_wy(const ChunkParams &p, void *workspace, cudaStream_t stream) {
  if ((long long)p.B * p.H > 65535) {  // the pre-pass grid's y dimension
    set_error("la_chunk_fwd: LA_KDA takes B*H <= 65535 (got %lld)", (long long)p.B * p.H);
    return LA_ERR_UNSUPPORTED;
  }
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  if (p.dk == 128 && p.dv == 128) return launch_typed<128, 128>(p, ws, stream);
  if (p.dk == 128) return launch_typed<128, 64>(p, ws, stream);
  if (p.dv == 128) return launch_typed<64, 128>(p, ws, stream);
  return launch_typed<64, 64>(p, ws, stream);
}

}  // namespace la
