// Chunkwise forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA),
// bf16 inputs, fp32 accumulation and fp32 state.
//
// One CTA owns one (b, h) for the whole sequence ("non-materialised": the
// state never leaves the SM; "Talk Linear Attention" section 4.1.1 describes
// this variant). It walks the chunks of C = 64 tokens in order; q/k/v tiles
// of the next two chunks stream in by TMA while the current one is computed.
//
// Every contraction is written transposed so that its M dimension is a
// feature axis of 128 rows (dv for the value side, [Q;K] stacked for the
// scores) and C = 64 is N or K:
//
//   D1   = [Q; K] K^T            M=128 (64 q rows + 64 k rows), N=C, K=dk
//   O1^T = S^T Q^T               M=dv, N=C, K=dk      inter-chunk output
//   Y^T  = S^T K^T               M=dv, N=C, K=dk      (delta rule only)
//   U^T  = Z^T T^T               M=dv, N=C, K=C       (delta rule only)
//   O2^T = U^T P^T               M=dv, N=C, K=C       local output
//   S^T += U^T Kt                M=dv, N=dk, K=C      state passing
//
// with, for a chunk with inclusive log-gate prefix b ("Talk Linear Attention"
// section 5.2) and the masked local scores P = (Q K^T) ⊙ exp(b_r - b_s) ⊙ M
// (section 3.2):
//   non-delta: U = V;  delta: Z = diag(beta) V - diag(beta e^b) K S,
//   A_rs = beta_r e^{b_r - b_s} k_r.k_s (s < r), T = (I + A)^-1, U = T Z
//   (the WY/UT form of the DeltaNet update, section 6.2);
//   o = diag(e^b) O1 + O2 (elu+1: divided by q.z + P 1);
//   S <- Diag(e^{b_last}) S + Kt^T U,  Kt = Diag(e^{b_last - b}) K.
// S^T lives in TMEM (lane = value column, 128 fp32 columns = key axis) for
// the whole sequence; each chunk reads it once to make the bf16 operand copy
// and to apply the decay. GLA gates act per key channel and are folded into
// Q, K and the state copy around the chunk midpoint m:
// (Q e^{B - b_m})(K e^{b_m - B})^T gives the scores exactly.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "la_internal.h"
#include "la_sm100.cuh"
#include "la_tc_common.cuh"

namespace la {
namespace {

using namespace sm100;
using namespace tc;


constexpr int kThreads = 128;
constexpr int kMid = kC / 2 - 1;
constexpr uint32_t kSpin = 1u << 22;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColD1 = 128, kColO1 = 192, kColO2 = 256, kColY = 320, kColU = 384;
constexpr int kAp = kC + 1;  // fp32 pitch of the A / T work matrices

struct TcLayout {
  uint32_t qk[2], v[2], g[2], st, p, t, z, u, af, tf, x, klo, kb, misc, bar, total;
  int ns;  // q/k/v(/g) stages: two, one for Kimi Delta Attention (gate tile + solve buffers)
};

__host__ __device__ inline uint32_t up1k(uint32_t x) { return (x + 1023u) & ~1023u; }

__host__ __device__ inline TcLayout tc_layout(int dk, int dv, int kind) {
  (void)dv;
  TcLayout L;
  const bool kda = kind == kKda, pg = kind == kGla || kda, delta = kind == kGdn || kda;
  const uint32_t qk_bytes = (uint32_t)(dk / 64) * 16384u;
  L.ns = kda ? 1 : 2;
  uint32_t o = 0;
  for (int s = 0; s < 2; ++s) { L.qk[s] = (s < L.ns) ? o : L.qk[0]; o += (s < L.ns) ? qk_bytes : 0u; }
  for (int s = 0; s < 2; ++s) { L.v[s] = (s < L.ns) ? o : L.v[0]; o += (s < L.ns) ? 16384u : 0u; }  // second 8 KB: zero pad when dv = 64
  for (int s = 0; s < 2; ++s) {
    const uint32_t gb = pg ? up1k((uint32_t)kC * dk * 4u) : 0u;
    L.g[s] = (s < L.ns) ? o : L.g[0];
    o += (s < L.ns) ? gb : 0u;
  }
  L.st = o; o += qk_bytes;          // bf16 S^T operand copy: 128 rows x dk
  L.p = o; o += 8192u;              // P, 64 x 64 bf16
  L.t = o; o += delta ? 8192u : 0u;
  L.z = o; o += delta ? 16384u : 0u;
  L.u = o; o += delta ? 16384u : 0u;
  L.af = o; o += delta ? up1k(kC * kAp * 4u) : 0u;
  L.tf = o; o += delta ? up1k(kC * kAp * 4u) : 0u;
  L.x = o; o += delta ? up1k(3u * 256u * 4u) : 0u;
  L.klo = o; o += (kind == kElu1) ? (uint32_t)(dk / 64) * 8192u : 0u;  // low half of phi(k)
  L.kb = o; o += kda ? (uint32_t)(dk / 64) * 8192u : 0u;  // KDA: K e^{b_m - B}, then K e^{b_last - B}
  L.misc = o; o += up1k((7u * kC + 4u * 128u) * 4u);
  L.bar = o; o += 64u;
  L.total = o;
  return L;
}

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const ChunkParams p, const __grid_constant__ CUtensorMap tm_q,
                const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  const int kind = p.kind;
  const TcLayout L = tc_layout(DK, DV, kind);
  const bool elu = kind == kElu1, gla = kind == kGla, kda = kind == kKda;
  const bool pg = gla || kda;                // per-key-channel gates (midpoint fold)
  const bool delta = kind == kGdn || kda;
  const bool sgate = kind == kRetnet || kind == kScalar || (kind == kGdn && p.g != nullptr);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int bh = blockIdx.x, h = bh % p.H;
  const int T = p.T, nchunks = (T + kC - 1) / kC;
  const int Wmem = DV + (elu ? 1 : 0);

  uint64_t *bar_full = reinterpret_cast<uint64_t *>(sm + L.bar);
  uint64_t *bar_mma = bar_full + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_full + 3);
  float *sb = reinterpret_cast<float *>(sm + L.misc);  // b_r (scalar gates)
  float *seb = sb + kC;                                 // e^{b_r}
  float *sebl = seb + kC;                               // e^{b_last - b_r}
  float *sbeta = sebl + kC;                             // beta_r (0 past the end)
  float *sden = sbeta + kC;                             // elu+1 denominators
  float *sdec = sden + kC;                              // [0] = e^{b_last}
  float *sz = sdec + kC;                                // elu+1 normaliser z [dk]
  float *sbm = sz + 128;                                // GLA e^{b_m,c}
  float *sblast = sbm + 128;                            // GLA e^{b_last,c}
  float *selm = sblast + 128;                           // GLA e^{b_last,c - b_m,c}
  float *sqz = selm + 128;                              // elu+1: phi(q_r) . z
  float *Af = reinterpret_cast<float *>(sm + L.af);
  float *Tf = reinterpret_cast<float *>(sm + L.tf);
  float *Xs = reinterpret_cast<float *>(sm + L.x);

  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar_full[0], 1);
    mbar_init(&bar_full[1], 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    if (pg) prefetch_tmap(&tm_g);
  }
  if (DV == 64) {  // zero pad block above the 64 real value rows of each V stage
    for (int i = tid; i < 2 * 512; i += kThreads) {
      reinterpret_cast<uint4 *>(sm + L.v[i >> 9] + 8192)[i & 511] = make_uint4(0, 0, 0, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t tl = tbase + lane_base;  // this thread's TMEM lane, column 0

  const uint32_t stage_bytes = 2u * DK * kC * 2u + DV * kC * 2u + (pg ? DK * kC * 4u : 0u);
  auto issue_loads = [&](int chunk, int s) {
    const int t0 = chunk * kC;
    mbar_arrive_expect_tx(&bar_full[s], stage_bytes);
#pragma unroll
    for (int a = 0; a < DK / 64; ++a) {
      tma_load_3d(sm + L.qk[s] + a * 16384, &tm_q, &bar_full[s], 64 * a, t0, bh);
      tma_load_3d(sm + L.qk[s] + a * 16384 + 8192, &tm_k, &bar_full[s], 64 * a, t0, bh);
    }
#pragma unroll
    for (int a = 0; a < DV / 64; ++a)
      tma_load_3d(sm + L.v[s] + a * 8192, &tm_v, &bar_full[s], 64 * a, t0, bh);
    if (pg) tma_load_3d(sm + L.g[s], &tm_g, &bar_full[s], 0, t0, bh);
  };
  int pending[2] = {-1, -1};  // chunk whose copies are in flight per stage (thread 0)
  if (tid == 0) {
    for (int s = 0; s < L.ns && s < nchunks; ++s) {
      issue_loads(s, s);
      pending[s] = s;
    }
  }

  // Initial state into TMEM (S^T: lane = value column v, column = key c).
  {
    const int v = tid;
    for (int c0 = 0; c0 < DK; c0 += 16) {
      float vals[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        vals[i] = (p.S0 && v < DV) ? p.S0[((size_t)bh * DK + c0 + i) * Wmem + v] : 0.f;
      tmem_st16(tl + kColS + c0, vals);
    }
    if (elu && tid < DK) sz[tid] = p.S0 ? p.S0[((size_t)bh * DK + tid) * Wmem + DV] : 0.f;
    tmem_wait_st();
  }

  // Scalar gates / beta of the next chunk are prefetched into registers.
  auto load_gate = [&](int chunk, float &lg, float &bt) {
    const int r = tid, t = chunk * kC + r;
    lg = 0.f;
    bt = 0.f;
    if (r < kC && chunk < nchunks && t < T) {
      if (kind == kRetnet) lg = __ldg(p.g + h);
      else if (sgate) lg = __ldg(p.g + (size_t)bh * T + t);
      bt = p.beta ? __ldg(p.beta + (size_t)bh * T + t) : 1.f;
    }
  };
  float lg_next = 0.f, bt_next = 0.f;
  load_gate(0, lg_next, bt_next);

  uint32_t mma_phase = 0;
  bool abort = false;
  const uint32_t id_d1 = idesc_bf16_f32(128, 64, false, false);
  const uint32_t id_kk = idesc_bf16_f32(128, 64, false, false);
  const uint32_t id_o2 = idesc_bf16_f32(128, 64, !delta, false);
  const uint32_t id_su = idesc_bf16_f32(128, DK, !delta, true);

  for (int i = 0; i < nchunks; ++i) {
    const int t0 = i * kC, n = min(kC, T - t0), s = i % L.ns;
    const uint32_t fpar = (i / L.ns) & 1;
    uint8_t *qk = sm + L.qk[s];
    uint8_t *vt = sm + L.v[s];
    float *gt = reinterpret_cast<float *>(sm + L.g[s]);

    if (tid < kC) {
      sb[tid] = lg_next;
      sbeta[tid] = bt_next;
    }
    load_gate(i + 1, lg_next, bt_next);
    if (L.ns == 1 && tid == 0 && i + 1 < nchunks) {  // one stage: warm L2 with the next chunk's tiles
      const int tp = (i + 1) * kC;
#pragma unroll
      for (int a = 0; a < DK / 64; ++a) {
        tma_prefetch_3d(&tm_q, 64 * a, tp, bh);
        tma_prefetch_3d(&tm_k, 64 * a, tp, bh);
      }
#pragma unroll
      for (int a = 0; a < DV / 64; ++a) tma_prefetch_3d(&tm_v, 64 * a, tp, bh);
      if (pg) tma_prefetch_3d(&tm_g, 0, tp, bh);
    }
    bool ok = mbar_wait_bounded(&bar_full[s], fpar, kSpin);
    if (__syncthreads_or(!ok)) { abort = true; break; }
    if (tid == 0) pending[s] = -1;

    // ---- inclusive log-gate prefix ----------------------------------------
    if (pg) {
      if (tid < DK) {
        float acc = 0.f, bmid = 0.f;
        for (int r = 0; r < kC; ++r) {
          acc += gt[r * DK + tid];
          gt[r * DK + tid] = acc;
          if (r == kMid) bmid = acc;
        }
        sbm[tid] = __expf(bmid);
        sblast[tid] = __expf(acc);
        selm[tid] = __expf(acc - bmid);
      }
    } else if (warp == 0) {
      const int l = tid;
      float v0 = sb[l], v1 = sb[l + 32];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float a0 = __shfl_up_sync(0xffffffffu, v0, off);
        const float a1 = __shfl_up_sync(0xffffffffu, v1, off);
        if (l >= off) { v0 += a0; v1 += a1; }
      }
      v1 += __shfl_sync(0xffffffffu, v0, 31);
      const float blast = __shfl_sync(0xffffffffu, v1, 31);
      sb[l] = v0;
      sb[l + 32] = v1;
      seb[l] = __expf(v0);
      seb[l + 32] = __expf(v1);
      sebl[l] = __expf(blast - v0);
      sebl[l + 32] = __expf(blast - v1);
      if (l == 0) sdec[0] = __expf(blast);
    }
    __syncthreads();

    // ---- elementwise prologue on the Q / K tiles -------------------------
    if (elu || pg) {
      constexpr int kChunks = 2 * kC * DK / 8;  // 16-byte groups in [Q;K]
      for (int ci = tid; ci < kChunks; ci += kThreads) {
        const int g8 = ci % (DK / 8), row = ci / (DK / 8);  // row 0..127 of [Q;K]
        const int r = row & (kC - 1);
        const bool is_k = row >= kC;
        uint8_t *ptr = qk + (g8 >> 3) * 16384 + sw128_off(row, (g8 & 7) * 8);
        float f[8];
        bf16x8_to_f32(*reinterpret_cast<uint4 *>(ptr), f);
        if (elu) {
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = (r < n) ? (f[e] > 0.f ? f[e] + 1.f : __expf(f[e])) : 0.f;
          if (is_k) {  // phi(k) = hi + lo in bf16: the state update and z use both halves
            const uint4 hi = f32_to_bf16x8(f);
            float fh[8];
            bf16x8_to_f32(hi, fh);
#pragma unroll
            for (int e = 0; e < 8; ++e) fh[e] = f[e] - fh[e];
            *reinterpret_cast<uint4 *>(sm + L.klo + (g8 >> 3) * 8192 + sw128_off(r, (g8 & 7) * 8)) =
                f32_to_bf16x8(fh);
          }
        } else {
          // GLA: Q e^{B - b_m}, K e^{b_m - B}. KDA: Q and K rows both e^{B - b_m} (the A rows
          // of K K^T and the key side of Y = (K e^B) S), K e^{b_m - B} apart (scores' B operand)
          const float *brow = gt + r * DK + g8 * 8;
          const float *bmid = gt + kMid * DK + g8 * 8;
          float fo[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float d = brow[e] - bmid[e];
            fo[e] = f[e] * __expf(-d);
            f[e] *= __expf((is_k && !kda) ? -d : d);
          }
          if (kda && is_k)
            *reinterpret_cast<uint4 *>(sm + L.kb + (g8 >> 3) * 8192 + sw128_off(r, (g8 & 7) * 8)) =
                f32_to_bf16x8(fo);
        }
        *reinterpret_cast<uint4 *>(ptr) = f32_to_bf16x8(f);
      }
    }

    // ---- state round trip: bf16 operand copy, then decay in place --------
    {
      const bool decays = sgate || pg;
      for (int c0 = 0; c0 < DK; c0 += 16) {
        float vals[16], cp[16];
        tmem_ld16(tl + kColS + c0, vals);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) cp[e] = pg ? vals[e] * sbm[c0 + e] : vals[e];
        store_row16_bf16(sm + L.st, 16384, tid, c0, cp);
        if (decays) {
#pragma unroll
          for (int e = 0; e < 16; ++e) vals[e] *= pg ? sblast[c0 + e] : sdec[0];
          tmem_st16(tl + kColS + c0, vals);
        }
      }
      tmem_wait_st();
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- MMA group 1: scores, inter-chunk output, (delta) S^T K^T --------
    if (tid == 0) {
      tc_fence_after();
      const uint32_t a_qk = smem_u32(qk), a_st = smem_u32(sm + L.st), a_kb = smem_u32(sm + L.kb);
#pragma unroll
      for (int kk = 0; kk < DK / 16; ++kk) {
        const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint64_t dq = desc_sw128(a_qk + ko, 16, 1024);          // rows 0..127: [Q; K]
        const uint64_t dk_ = desc_sw128(a_qk + ko + 8192, 16, 1024);  // rows 0..63: K
        const uint64_t ds = desc_sw128(a_st + ko, 16, 1024);          // S^T copy
        const uint64_t dkb = kda ? desc_sw128(a_kb + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024) : dk_;
        mma_bf16(tbase + kColD1, dq, dkb, id_d1, kk > 0);
        mma_bf16(tbase + kColO1, ds, dq, id_kk, kk > 0);
        if (delta) mma_bf16(tbase + kColY, ds, dk_, id_kk, kk > 0);
      }
      mma_commit(bar_mma);
    }
    ok = mbar_wait_bounded(bar_mma, mma_phase, kSpin);
    mma_phase ^= 1;
    if (__syncthreads_or(!ok)) { abort = true; break; }
    tc_fence_after();

    // ---- epilogue 1: P (lanes 0..63), A (lanes 64..127), Z (delta) ------
    if (tid < kC) {
      const int r = tid;
      float rowsum = 0.f;
      for (int s0 = 0; s0 < kC; s0 += 16) {
        float d[16];
        tmem_ld16(tl + kColD1 + s0, d);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int sc = s0 + e;
          float x = (sc <= r && r < n) ? d[e] : 0.f;
          if (sgate && sc <= r) x *= __expf(sb[r] - sb[sc]);
          d[e] = __bfloat162float(__float2bfloat16_rn(x));
          rowsum += d[e];
        }
        store_row16_bf16(sm + L.p, 8192, r, s0, d);
      }
      if (elu) sden[r] = rowsum;
    } else {
      const int r = tid - kC;
      if (delta) {
        for (int s0 = 0; s0 < kC; s0 += 16) {
          float d[16];
          tmem_ld16(tl + kColD1 + s0, d);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int sc = s0 + e;
            float a = 0.f;
            if (sc < r && r < n) a = sbeta[r] * d[e] * (sgate ? __expf(sb[r] - sb[sc]) : 1.f);
            Af[r * kAp + sc] = a;
          }
        }
      }
      if (elu) {  // q_r . z with the rounded phi(q) the MMA used
        float acc = 0.f;
        for (int g8 = 0; g8 < DK / 8; ++g8) {
          float f[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4 *>(qk + (g8 >> 3) * 16384 +
                                                          sw128_off(r, (g8 & 7) * 8)), f);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc = fmaf(f[e], sz[g8 * 8 + e], acc);
        }
        sqz[r] = acc;
      }
    }
    if (delta) {  // Z^T[v][r] = beta_r (V[r][v] - e^{b_r} Y^T[v][r])
      const int v = tid;
      const uint8_t *vb = vt + (v >> 6) * 8192;
      for (int r0 = 0; r0 < kC; r0 += 16) {
        float y[16];
        tmem_ld16(tl + kColY + r0, y);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int r = r0 + e;
          const float ey = kda ? 1.f : seb[r];  // KDA: e^{B} is inside (K e^B) S already
          y[e] = (v < DV) ? sbeta[r] * (bf16_at(vb, sw128_off(r, v & 63)) - ey * y[e]) : 0.f;
        }
        store_row16_bf16(sm + L.z, 16384, v, r0, y);
      }
    }
    tc_fence_before();
    __syncthreads();
    if (L.ns == 1 && tid == 0 && i + 1 < nchunks) {  // the only stage is consumed: stream the next chunk
      issue_loads(i + 1, 0);
      pending[0] = i + 1;
    }

    // ---- K -> Kt in place (state-update operand); elu+1 z and den --------
    if (kda) {  // K e^{b_m - B} -> K e^{b_last - B}
      constexpr int kChunks = kC * DK / 8;
      for (int ci = tid; ci < kChunks; ci += kThreads) {
        const int g8 = ci % (DK / 8), r = ci / (DK / 8);
        uint8_t *ptr = sm + L.kb + (g8 >> 3) * 8192 + sw128_off(r, (g8 & 7) * 8);
        float f[8];
        bf16x8_to_f32(*reinterpret_cast<uint4 *>(ptr), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] *= selm[g8 * 8 + e];
        *reinterpret_cast<uint4 *>(ptr) = f32_to_bf16x8(f);
      }
    } else if (sgate || gla) {
      constexpr int kChunks = kC * DK / 8;
      for (int ci = tid; ci < kChunks; ci += kThreads) {
        const int g8 = ci % (DK / 8), r = ci / (DK / 8);
        uint8_t *ptr = qk + (g8 >> 3) * 16384 + 8192 + sw128_off(r, (g8 & 7) * 8);
        float f[8];
        bf16x8_to_f32(*reinterpret_cast<uint4 *>(ptr), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] *= gla ? selm[g8 * 8 + e] : sebl[r];
        *reinterpret_cast<uint4 *>(ptr) = f32_to_bf16x8(f);
      }
    }
    if (elu) {
      if (tid < kC) sden[tid] += sqz[tid];
      if (tid < DK) {
        float acc = 0.f;
        for (int r = 0; r < kC; ++r)
          acc += bf16_at(qk + (tid >> 6) * 16384 + 8192, sw128_off(r, tid & 63)) +
                 bf16_at(sm + L.klo + (tid >> 6) * 8192, sw128_off(r, tid & 63));
        sz[tid] += acc;
      }
    }
    // ---- delta rule: T = (I + A)^-1, 16x16 diagonal blocks then levels ----
    if (delta) {
      if (tid < kC) {  // diagonal blocks, one column per thread
        const int blk = tid >> 4, j = tid & 15, base = blk * 16;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float acc = (r == j) ? 1.f : 0.f;
#pragma unroll
          for (int m = 0; m < r; ++m)
            if (m >= j) acc = fmaf(-Af[(base + r) * kAp + base + m], x[m], acc);
          x[r] = (r < j) ? 0.f : acc;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Tf[(base + r) * kAp + base + j] = x[r];
      }
      __syncthreads();
      for (int lvl = 1; lvl < 4; ++lvl) {
        const int nblk = 4 - lvl;
        // X_i = sum_{k=j}^{i-1} A_ik T_kj for blocks (i, j = i - lvl)
        for (int e = tid; e < nblk * 256; e += kThreads) {
          const int bi = e >> 8, a = (e >> 4) & 15, bcol = e & 15;
          const int ib = bi + lvl, jb = bi;
          float acc = 0.f;
          for (int kb = jb; kb < ib; ++kb)
#pragma unroll
            for (int m = 0; m < 16; ++m)
              acc = fmaf(Af[(ib * 16 + a) * kAp + kb * 16 + m], Tf[(kb * 16 + m) * kAp + jb * 16 + bcol], acc);
          Xs[e] = acc;
        }
        __syncthreads();
        for (int e = tid; e < nblk * 256; e += kThreads) {
          const int bi = e >> 8, a = (e >> 4) & 15, bcol = e & 15;
          const int ib = bi + lvl, jb = bi;
          float acc = 0.f;
#pragma unroll
          for (int m = 0; m < 16; ++m)
            if (m <= a) acc = fmaf(Tf[(ib * 16 + a) * kAp + ib * 16 + m], Xs[(bi << 8) + m * 16 + bcol], acc);
          Tf[(ib * 16 + a) * kAp + jb * 16 + bcol] = -acc;
        }
        __syncthreads();
      }
      // bf16 T (upper triangle zero) as the K-major B operand [r][s]
      for (int ci = tid; ci < kC * 8; ci += kThreads) {
        const int r = ci >> 3, g8 = ci & 7;
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int sc = g8 * 8 + e;
          f[e] = (sc <= r) ? Tf[r * kAp + sc] : 0.f;
        }
        *reinterpret_cast<uint4 *>(sm + L.t + sw128_off(r, g8 * 8)) = f32_to_bf16x8(f);
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    if (delta) {  // ---- U^T = Z^T T^T ----
      if (tid == 0) {
        tc_fence_after();
        const uint32_t a_z = smem_u32(sm + L.z), a_t = smem_u32(sm + L.t);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tbase + kColU, desc_sw128(a_z + kk * 32, 16, 1024),
                   desc_sw128(a_t + kk * 32, 16, 1024), id_kk, kk > 0);
        mma_commit(bar_mma);
      }
      ok = mbar_wait_bounded(bar_mma, mma_phase, kSpin);
      mma_phase ^= 1;
      if (__syncthreads_or(!ok)) { abort = true; break; }
      tc_fence_after();
      for (int r0 = 0; r0 < kC; r0 += 16) {
        float u[16];
        tmem_ld16(tl + kColU + r0, u);
        tmem_wait_ld();
        store_row16_bf16(sm + L.u, 16384, tid, r0, u);
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();
    }

    // ---- MMA group 2: local output and state update ----------------------
    if (tid == 0) {
      tc_fence_after();
      const uint32_t a_p = smem_u32(sm + L.p), a_k = smem_u32(qk + 8192);
      const uint32_t a_u = delta ? smem_u32(sm + L.u) : smem_u32(vt);
#pragma unroll
      for (int kk = 0; kk < kC / 16; ++kk) {
        const uint64_t du = delta ? desc_sw128(a_u + kk * 32, 16, 1024)
                                  : desc_sw128(a_u + kk * 2048, 8192, 1024);
        mma_bf16(tbase + kColO2, du, desc_sw128(a_p + kk * 32, 16, 1024), id_o2, kk > 0);
        const uint64_t dkt = kda ? desc_sw128(smem_u32(sm + L.kb) + kk * 2048, 8192, 1024)
                                 : desc_sw128(a_k + kk * 2048, 16384, 1024);
        mma_bf16(tbase + kColS, du, dkt, id_su, 1);
        if (elu)
          mma_bf16(tbase + kColS, du, desc_sw128(smem_u32(sm + L.klo) + kk * 2048, 8192, 1024),
                   id_su, 1);
      }
      mma_commit(bar_mma);
    }
    ok = mbar_wait_bounded(bar_mma, mma_phase, kSpin);
    mma_phase ^= 1;
    if (__syncthreads_or(!ok)) { abort = true; break; }
    tc_fence_after();
    if (L.ns == 2 && tid == 0 && i + 2 < nchunks) {  // the stage is free: stream chunk i + 2 into it
      issue_loads(i + 2, s);
      pending[s] = i + 2;
    }

    // ---- output epilogue --------------------------------------------------
    {
      const int v = tid;
      __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o) + ((size_t)bh * T + t0) * DV + v;
      for (int r0 = 0; r0 < kC; r0 += 16) {
        float a[16], b[16];
        tmem_ld16(tl + kColO1 + r0, a);
        tmem_ld16(tl + kColO2 + r0, b);
        tmem_wait_ld();
        if (v < DV) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int r = r0 + e;
            if (r < n) {
              float x = (pg || !sgate) ? a[e] + b[e] : fmaf(seb[r], a[e], b[e]);
              if (elu) x = x / sden[r];
              o[(size_t)r * DV] = __float2bfloat16_rn(x);
            }
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  }

  if (!abort) {
    tc_fence_after();
    if (p.S_final) {
      const int v = tid;
      for (int c0 = 0; c0 < DK; c0 += 16) {
        float vals[16];
        tmem_ld16(tl + kColS + c0, vals);
        tmem_wait_ld();
        if (v < DV) {
#pragma unroll
          for (int e = 0; e < 16; ++e) p.S_final[((size_t)bh * DK + c0 + e) * Wmem + v] = vals[e];
        }
      }
      if (elu && tid < DK) p.S_final[((size_t)bh * DK + tid) * Wmem + DV] = sz[tid];
    }
  } else if (tid == 0) {
    atomicOr(p.status, kStatusTimeout);
    // let copies and MMAs already in flight land before the memory goes away
    for (int s = 0; s < L.ns; ++s)
      if (pending[s] >= 0) (void)mbar_wait_bounded(&bar_full[s], (pending[s] / L.ns) & 1, kSpin);
    (void)mbar_wait_bounded(bar_mma, mma_phase, kSpin);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

// ---------------------------------------------------------------- host side

template <int DK, int DV>
int launch_typed(const ChunkParams &p, cudaStream_t stream) {
  const TcLayout L = tc_layout(DK, DV, p.kind);
  const size_t smem = L.total + 1024;
  if (smem > 232448) {
    set_error("la_chunk_fwd: tensor-core kernel needs %zu bytes of shared memory", smem);
    return LA_ERR_UNSUPPORTED;
  }
  const int BH = p.B * p.H;
  CUtensorMap mq, mk, mv, mg;
  bool ok = make_map(&mq, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DK, p.T, BH, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&mk, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DK, p.T, BH, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&mv, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, p.T, BH, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  if (ok && (p.kind == kGla || p.kind == kKda))
    ok = make_map(&mg, p.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, DK, p.T, BH, DK,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
  else
    mg = mq;
  if (!ok) {
    set_error("la_chunk_fwd: cuTensorMapEncodeTiled rejected a tensor map");
    return LA_ERR_CUDA;
  }
  auto kern = chunk_tc_kernel<DK, DV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) {
    kern<<<BH, kThreads, smem, stream>>>(p, mq, mk, mv, mg);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_error("la_chunk_fwd: tensor-core kernel launch failed: %s", cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  return LA_OK;
}

}  // namespace

int launch_chunk_tc(const ChunkParams &p, cudaStream_t stream) {
  if (p.f32) {
    set_error("la_chunk_fwd: the tensor-core kernel takes bfloat16 inputs");
    return LA_ERR_UNSUPPORTED;
  }
  if (!encode_fn()) {
    set_error("la_chunk_fwd: cuTensorMapEncodeTiled is unavailable");
    return LA_ERR_CUDA;
  }
  if (p.kind == kKda) {  // Kimi Delta Attention: the sequential-phase kernel, one stage
    if (p.dk == 128 && p.dv == 128) return launch_typed<128, 128>(p, stream);
    if (p.dk == 128 && p.dv == 64) return launch_typed<128, 64>(p, stream);
    if (p.dk == 64 && p.dv == 128) return launch_typed<64, 128>(p, stream);
    return launch_typed<64, 64>(p, stream);
  }
  if (p.kind != kGdn) return launch_chunk_ws(p, stream);
  if (p.dk == 128 && p.dv == 128) {
    // two CTAs per head (value halves, alternate chunks' key side) while the
    // doubled grid still fits on the GPU at once; LA_DELTA = pair | single forces one
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 0;
    bool pair = 2LL * p.B * p.H <= sms;
    if (const char *env = getenv("LA_DELTA")) {
      if (strcmp(env, "pair") == 0) pair = true;
      if (strcmp(env, "single") == 0) pair = false;
    }
    return pair ? launch_chunk_delta_pair(p, stream) : launch_chunk_delta(p, stream);
  }
  if (p.dk == 128 && p.dv == 64) return launch_typed<128, 64>(p, stream);
  if (p.dk == 64 && p.dv == 128) return launch_typed<64, 128>(p, stream);
  return launch_typed<64, 64>(p, stream);
}

}  // namespace la
