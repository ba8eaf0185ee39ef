// Warp-specialised chunk forward for the gated delta rule (Gated DeltaNet;
// plain DeltaNet when g is absent) on tcgen05 + TMEM + TMA, bf16 inputs,
// fp32 state, dk = dv = 128.
//
// Per chunk of C = 64 tokens with inclusive log-gate prefix b (scalar per
// token) and the WY/UT form of the delta rule ("Talk Linear Attention"
// section 6.2; decay first, then the delta rule, as Gated DeltaNet writes it):
//
//   A_rs = beta_r e^{b_r - b_s} k_r.k_s (s < r),  T = (I + A)^-1
//   W    = T diag(beta e^b) K,  U = T diag(beta) V - W S_prev
//   O    = Diag(e^b) Q S_prev + P U,  P = (Q K^T) ⊙ e^{b_r - b_s} ⊙ M
//   S   <- e^{b_last} S_prev + Kt^T U,  Kt = Diag(e^{b_last - b}) K
//
// Everything that does not depend on S (scores, A, the triangular solve, W)
// is produced by the key group one chunk ahead; the S-dependent chain per
// chunk is: state round trip -> U MMAs -> U epilogue -> state-update MMA.
// In transposed form (M = 128 feature rows, C = 64 as N or K):
//   D1   = [Q; K] K^T            scores and K K^T
//   W^T  = K^T T''^T             T'' = T diag(beta e^b)          (key side)
//   U^T  = V^T T'^T + S^T (-W)^T T' = T diag(beta)             (state side)
//   O^T  = S^T Qt^T + U^T P^T,   S^T += U^T Kt
//
// Roles (384 threads): warp 0 producer (TMA tiles + gate/beta prefix),
// warp 1 key-side MMAs (D1, W), warp 2 state-side MMAs (U, O, state update),
// warp 3 TMEM owner, warps 4-7 state group (round trip, U epilogue, output
// epilogue), warps 8-11 key group (P, A, triangular solve, W epilogue,
// in-place Qt / Kt). All waits are bounded (device status word on expiry).
#include "la_tc_common.cuh"
#include "la_wy.cuh"

namespace la {
namespace {

using namespace sm100;
using namespace tc;
using namespace wy;

constexpr int kThreads = 384;
constexpr int DK = 128, DV = 128;
constexpr int kNS = 2;   // q/k/v stages
constexpr int kNM = 4;   // per-chunk scalar slots
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColD1 = 128, kColW = 192, kColU = 256, kColO = 320;  // O: 2 x 64
constexpr int kSG = 128, kKG = 256;
constexpr int kBarSG = 1, kBarKG = 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kFastLimit = 100.f;

// per-chunk scalars (floats)
constexpr int kMsB2 = 0, kMsEB = 64, kMsBeta = 128, kMsDec = 192, kMsB2L = 193, kMsFast = 194,
              kMsF = 256, kMsVS = 320, kMsBEB = 384, kMsAR = 448, kMsBytes = 2048;

__host__ __device__ inline uint32_t up1k(uint32_t x) { return (x + 1023u) & ~1023u; }

struct DLayout {
  uint32_t qk, v, stage;                       // inside a stage
  uint32_t p, st, af, tf, tp, tpp, wu, misc, bar, total;
};

__host__ __device__ inline DLayout d_layout() {
  DLayout L;
  uint32_t o = 0;
  L.qk = o; o += 32768u;
  L.v = o; o += 16384u;
  L.stage = o;
  o = L.stage * kNS;
  L.p = o; o += 2u * 8192u;               // scores P, two buffers
  L.st = o; o += 32768u;                  // bf16 S^T copy
  L.af = o; o += up1k(kC * kAp * 4u);     // A, fp32
  L.tf = o; o += up1k(kC * kAp * 4u);     // T, fp32
  L.tp = o; o += 8192u;                   // T' = T diag(beta), bf16 [r][s]
  L.tpp = o; o += 8192u;                  // T'' = T diag(beta e^b), bf16 [r][s]
  L.wu = o; o += 16384u;                  // -W (MN-major [c][r]), later U^T ([v][s])
  L.misc = o; o += kNM * kMsBytes;
  L.bar = o; o += 512u;
  L.total = o;
  return L;
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_delta_kernel(const ChunkParams p, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const DLayout L = d_layout();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x;
  const int T = p.T, nchunks = (T + kC - 1) / kC;
  const bool gated = p.g != nullptr;

  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.bar);
  uint64_t *full = bars, *empty = bars + 2, *key_ready = bars + 4, *mfree = bars + 6;   // [2],[2],[2],[4]
  uint64_t *d1_full = bars + 10, *d1_free = bars + 11, *t_ready = bars + 12, *w_full = bars + 13;
  uint64_t *s_ready = bars + 14, *u_full = bars + 15, *u_ready = bars + 16, *s_done = bars + 17;
  uint64_t *o_done = bars + 18, *o_free = bars + 20, *kfree = bars + 22, *drain = bars + 23;  // [2],[2],1,[2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 26);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  float *Af = reinterpret_cast<float *>(sm + L.af);
  float *Tf = reinterpret_cast<float *>(sm + L.tf);
  auto stage = [&](int s) { return sm + (uint32_t)s * L.stage; };
  auto mslot = [&](int j) { return reinterpret_cast<float *>(sm + L.misc + (uint32_t)(j % kNM) * kMsBytes); };

  if (warp == 3) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&full[s], 2);   // TMA bytes + the producer's gate prefix
      mbar_init(&empty[s], 1);  // state-side MMA commit after the chunk's last MMA
      mbar_init(&key_ready[s], 1);
    }
    for (int m = 0; m < kNM; ++m) mbar_init(&mfree[m], 1);
    mbar_init(d1_full, 1);
    mbar_init(d1_free, 1);
    mbar_init(t_ready, 1);
    mbar_init(w_full, 1);
    mbar_init(s_ready, 1);
    mbar_init(u_full, 1);
    mbar_init(u_ready, 1);
    mbar_init(s_done, 1);
    mbar_init(kfree, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&o_done[b], 1);
      mbar_init(&o_free[b], 1);
      mbar_init(&drain[b], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t tl = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    constexpr uint32_t bytes = 2u * DK * kC * 2u + DV * kC * 2u;
    int issued = 0;
    for (int j = 0; j < nchunks; ++j) {
      const int s = j % kNS, t0 = j * kC;
      int ok = 1;
      if (lane == 0) ok = wait_or_abort(&mfree[j % kNM], ((j / kNM) & 1) ^ 1, abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      {
        float *ms = mslot(j);
        const int t = t0 + lane;
        float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
        if (t < T) {
          g0 = gated ? __ldg(p.g + (size_t)bh * T + t) : 0.f;
          b0 = p.beta ? __ldg(p.beta + (size_t)bh * T + t) : 1.f;
        }
        if (t + 32 < T) {
          g1 = gated ? __ldg(p.g + (size_t)bh * T + t + 32) : 0.f;
          b1 = p.beta ? __ldg(p.beta + (size_t)bh * T + t + 32) : 1.f;
        }
        float v0 = g0 * kLog2e, v1 = g1 * kLog2e;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float a0 = __shfl_up_sync(0xffffffffu, v0, off);
          const float a1 = __shfl_up_sync(0xffffffffu, v1, off);
          if (lane >= off) { v0 += a0; v1 += a1; }
        }
        v1 += __shfl_sync(0xffffffffu, v0, 31);
        const float bl = __shfl_sync(0xffffffffu, v1, 31);
        const float e0 = exp2f(v0), e1 = exp2f(v1);
        const float f0 = exp2f(v0 - bl), f1 = exp2f(v1 - bl);
        ms[kMsB2 + lane] = v0;
        ms[kMsB2 + lane + 32] = v1;
        ms[kMsEB + lane] = e0;
        ms[kMsEB + lane + 32] = e1;
        ms[kMsBeta + lane] = b0;
        ms[kMsBeta + lane + 32] = b1;
        ms[kMsF + lane] = f0;
        ms[kMsF + lane + 32] = f1;
        ms[kMsVS + lane] = exp2f(bl - v0);
        ms[kMsVS + lane + 32] = exp2f(bl - v1);
        ms[kMsBEB + lane] = b0 * e0;
        ms[kMsBEB + lane + 32] = b1 * e1;
        ms[kMsAR + lane] = b0 * f0;
        ms[kMsAR + lane + 32] = b1 * f1;
        if (lane == 0) {
          ms[kMsDec] = exp2f(bl);
          ms[kMsB2L] = bl;
          ms[kMsFast] = (-bl < kFastLimit) ? 1.f : 0.f;
        }
        __syncwarp();
      }
      if (lane == 0) ok = wait_or_abort(&empty[s], ((j / kNS) & 1) ^ 1, abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      uint8_t *st = stage(s);
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          tma_load_3d(st + L.qk + a * 16384, &tm_q, &full[s], 64 * a, t0, bh);
          tma_load_3d(st + L.qk + a * 16384 + 8192, &tm_k, &full[s], 64 * a, t0, bh);
          tma_load_3d(st + L.v + a * 8192, &tm_v, &full[s], 64 * a, t0, bh);
        }
        mbar_arrive(&full[s]);
        // the load of chunk j + kNS waits for this chunk's last MMA; warm L2 now
        // so that it does not pay the DRAM latency then
        if (j + kNS < nchunks) {
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            tma_prefetch_3d(&tm_q, 64 * a, t0 + kNS * kC, bh);
            tma_prefetch_3d(&tm_k, 64 * a, t0 + kNS * kC, bh);
            tma_prefetch_3d(&tm_v, 64 * a, t0 + kNS * kC, bh);
          }
        }
      }
      issued = j + 1;
    }
    if (lane == 0)
      for (int j = (issued > kNS ? issued - kNS : 0); j < issued; ++j)
        (void)mbar_wait_bounded(&full[j % kNS], (j / kNS) & 1, kSpinLimit);
  } else if (warp == 1) {
    // ------------------------------------------------- key-side MMAs: D1, W
    if (lane == 0) {
      constexpr uint32_t id_d1 = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t id_w = idesc_bf16_f32(128, 64, true, false);
      const uint32_t a_tpp = smem_u32(sm + L.tpp);
      // scores of chunk j into the (single) D1 buffer once the key group read chunk j-1's
      auto issue_d1 = [&](int j) -> bool {
        const int s = j % kNS;
        if (!wait_or_abort(&full[s], (j / kNS) & 1, abort_flag, p.status)) return false;
        if (!wait_or_abort(d1_free, (j & 1) ^ 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint32_t a_qk = smem_u32(stage(s) + L.qk);
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16(tbase + kColD1, desc_sw128(a_qk + ko, 16, 1024), desc_sw128(a_qk + ko + 8192, 16, 1024),
                   id_d1, kk > 0);
        }
        mma_commit(d1_full);
        return true;
      };
      bool ok = nchunks > 0 && issue_d1(0);
      for (int j = 0; j < nchunks && ok; ++j) {
        if (j + 1 < nchunks && !issue_d1(j + 1)) break;
        // W^T = K^T T''^T: K rows as MN-major A (M = dk), T'' K-major
        if (!wait_or_abort(t_ready, j & 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t a_qk = smem_u32(stage(j % kNS) + L.qk);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tbase + kColW, desc_sw128(a_qk + 8192 + kk * 2048, 16384, 1024),
                   desc_sw128(a_tpp + kk * 32, 16, 1024), id_w, kk > 0);
        mma_commit(w_full);
      }
      mma_commit(&drain[0]);
      (void)mbar_wait_bounded(&drain[0], 0, kSpinLimit);
    }
  } else if (warp == 2) {
    // ------------------------------------- state-side MMAs: U, O, state update
    if (lane == 0) {
      constexpr uint32_t id_ut = idesc_bf16_f32(128, 64, true, false);   // V^T T'^T
      constexpr uint32_t id_us = idesc_bf16_f32(128, 64, false, true);   // S^T (-W)^T
      constexpr uint32_t id_o1 = idesc_bf16_f32(128, 64, false, false);  // S^T Qt^T
      constexpr uint32_t id_su = idesc_bf16_f32(128, DK, false, true);   // U^T Kt
      constexpr uint32_t id_o2 = idesc_bf16_f32(128, 64, false, false);  // U^T P^T
      const uint32_t a_st = smem_u32(sm + L.st), a_tp = smem_u32(sm + L.tp), a_wu = smem_u32(sm + L.wu);
      for (int i = 0; i < nchunks; ++i) {
        const int s = i % kNS;
        if (!wait_or_abort(&key_ready[s], (i / kNS) & 1, abort_flag, p.status)) break;
        if (!wait_or_abort(s_ready, i & 1, abort_flag, p.status)) break;
        if (!wait_or_abort(&o_free[i & 1], ((i >> 1) & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        uint8_t *st = stage(s);
        const uint32_t a_v = smem_u32(st + L.v), a_qk = smem_u32(st + L.qk);
        const uint32_t d_o = tbase + kColO + (uint32_t)(i & 1) * 64u;
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tbase + kColU, desc_sw128(a_v + kk * 2048, 8192, 1024), desc_sw128(a_tp + kk * 32, 16, 1024),
                   id_ut, kk > 0);
        // T' has been read (and T'' by the W MMA before s_ready): the key
        // group may write the next chunk's T' and T''
        mma_commit(kfree);
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16(tbase + kColU, desc_sw128(a_st + ko, 16, 1024), desc_sw128(a_wu + kk * 2048, 8192, 1024),
                   id_us, 1);
        }
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16(d_o, desc_sw128(a_st + ko, 16, 1024), desc_sw128(a_qk + ko, 16, 1024), id_o1, kk > 0);
        }
        mma_commit(u_full);
        if (!wait_or_abort(u_ready, i & 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t a_p = smem_u32(sm + L.p + (uint32_t)(i & 1) * 8192u);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(d_o, desc_sw128(a_wu + kk * 32, 16, 1024), desc_sw128(a_p + kk * 32, 16, 1024), id_o2, 1);
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tbase + kColS, desc_sw128(a_wu + kk * 32, 16, 1024),
                   desc_sw128(a_qk + 8192 + kk * 2048, 16384, 1024), id_su, 1);
        mma_commit(s_done);
        mma_commit(&o_done[i & 1]);
        mma_commit(&empty[s]);
      }
      mma_commit(&drain[1]);
      (void)mbar_wait_bounded(&drain[1], 0, kSpinLimit);
    }
  } else if (tid >= kSG && tid < kKG) {
    // ------------------------------------------------------------ state group
    const int v = tid - kSG;
    for (int c0 = 0; c0 < DK; c0 += 32) {
      float x[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) x[e] = p.S0 ? p.S0[((size_t)bh * DK + c0 + e) * DV + v] : 0.f;
      tmem_st32(tl + kColS + c0, x);
    }
    tmem_wait_st();
    bool alive = true;
    for (int i = 0; i <= nchunks && alive; ++i) {
      if (i < nchunks) {
        const int s = i % kNS;
        const float *ms = mslot(i);
        // W^T of this chunk is in TMEM, and the previous chunk's MMAs have
        // finished with the shared -W / U buffer and with the state
        bool ok = wait_or_abort(w_full, i & 1, abort_flag, p.status);
        if (ok && i > 0) ok = wait_or_abort(s_done, (i - 1) & 1, abort_flag, p.status);
        if (!group_all(ok, kBarSG)) { alive = false; break; }
        tc_fence_after();
        // -W as the MN-major B operand [c][r] (TMEM lane = key channel c)
#pragma unroll 1
        for (int r0 = 0; r0 < kC; r0 += 32) {
          float x[32];
          tmem_ld32(tl + kColW + r0, x);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = -x[e];
          store_row32_bf16(sm + L.wu, 16384, v, r0, x);
        }
        // Qt = Diag(e^b) Q, Kt = Diag(e^{b_last - b}) K in place (row v of [Q; K])
        if (gated) {
          uint8_t *qk = stage(s) + L.qk;
          const int r = v & (kC - 1);
          const float rs = (v < kC) ? ms[kMsEB + r] : ms[kMsVS + r];
#pragma unroll 1
          for (int g0 = 0; g0 < 16; g0 += 4) {  // rolled: keeps the hot loop's code small
            uint4 u[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
              u[q] = *reinterpret_cast<const uint4 *>(qk + ((g0 + q) >> 3) * 16384 + sw128_off(v, ((g0 + q) & 7) * 8));
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float f[8];
              unpack8(u[q], f);
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] *= rs;
              *reinterpret_cast<uint4 *>(qk + ((g0 + q) >> 3) * 16384 + sw128_off(v, ((g0 + q) & 7) * 8)) = pack8(f);
            }
          }
        }
        // state round trip: bf16 operand copy of S_prev, decay in place
        const float dec = ms[kMsDec];
#pragma unroll 1
        for (int c0 = 0; c0 < DK; c0 += 32) {
          float x[32];
          tmem_ld32(tl + kColS + c0, x);
          tmem_wait_ld();
          store_row32_bf16(sm + L.st, 16384, v, c0, x);
          if (gated) {
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] *= dec;
            tmem_st32(tl + kColS + c0, x);
          }
        }
        tmem_wait_st();
        fence_proxy_async();
        tc_fence_before();
        group_sync(kBarSG);
        if (v == 0) mbar_arrive(s_ready);
        // U epilogue: U^T (fp32, TMEM) -> bf16 K-major operand [v][s]
        ok = wait_or_abort(u_full, i & 1, abort_flag, p.status);
        if (!group_all(ok, kBarSG)) { alive = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int r0 = 0; r0 < kC; r0 += 32) {
          float x[32];
          tmem_ld32(tl + kColU + r0, x);
          tmem_wait_ld();
          store_row32_bf16(sm + L.wu, 16384, v, r0, x);
        }
        fence_proxy_async();
        tc_fence_before();
        group_sync(kBarSG);
        if (v == 0) mbar_arrive(u_ready);
      }
      if (i > 0) {
        // output epilogue of chunk c = i - 1 (overlaps the state update of chunk i)
        const int c = i - 1, ob = c & 1, n = min(kC, T - c * kC);
        bool ok = wait_or_abort(&o_done[ob], (c >> 1) & 1, abort_flag, p.status);
        if (!group_all(ok, kBarSG)) { alive = false; break; }
        tc_fence_after();
        __nv_bfloat16 *og = static_cast<__nv_bfloat16 *>(p.o) + ((size_t)bh * T + (size_t)c * kC) * DV;
        const bool odd = lane & 1;
#pragma unroll 1
        for (int r0 = 0; r0 < kC; r0 += 16) {
          float a[16];
          tmem_ld16(tl + kColO + ob * 64 + r0, a);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const float send = odd ? a[e] : a[e + 1];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
            const int r = r0 + e + (odd ? 1 : 0);
            const int col = v - (odd ? 1 : 0);
            const uint32_t w = odd ? pack_bf16(recv, a[e + 1]) : pack_bf16(a[e], recv);
            if (r < n) *reinterpret_cast<uint32_t *>(og + (size_t)r * DV + col) = w;
          }
        }
        tc_fence_before();
        group_sync(kBarSG);
        if (v == 0) {
          mbar_arrive(&o_free[ob]);
          mbar_arrive(&mfree[c % kNM]);
        }
      }
    }
    if (alive && p.S_final) {
      bool ok = wait_or_abort(s_done, (nchunks - 1) & 1, abort_flag, p.status);
      if (group_all(ok, kBarSG)) {
        tc_fence_after();
        for (int c0 = 0; c0 < DK; c0 += 32) {
          float x[32];
          tmem_ld32(tl + kColS + c0, x);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) p.S_final[((size_t)bh * DK + c0 + e) * DV + v] = x[e];
        }
      }
    }
  } else if (tid >= kKG) {
    // -------------------------------------------------------------- key group
    const int kg = tid - kKG;
    for (int j = 0; j < nchunks; ++j) {
      const int s = j % kNS, n = min(kC, T - j * kC);
      uint8_t *st = stage(s);
      float *ms = mslot(j);
      bool ok = wait_or_abort(&full[s], (j / kNS) & 1, abort_flag, p.status);
      if (ok) ok = wait_or_abort(d1_full, j & 1, abort_flag, p.status);
      if (!group_all(ok, kBarKG)) break;
      tc_fence_after();
      const bool fast = ms[kMsFast] != 0.f;
      // ---- P (TMEM lanes 0..63 = Q K^T rows) and A (lanes 64..127 = K K^T rows)
      bool okp = true;
      if (kg < kC) {
        // P buffer j & 1 is free once chunk j - 2's output MMA has read it
        okp = wait_or_abort(&o_done[j & 1], ((j >> 1) & 1) ^ 1, abort_flag, p.status);
      }
      if (kg < kC && okp) {
        const int r = kg;
        const float b2r = ms[kMsB2 + r], fr = ms[kMsF + r];
#pragma unroll 1
        for (int s0 = 0; s0 < kC; s0 += 32) {
          float d[32], fs[32];
          load32(ms + (fast ? kMsVS : kMsB2) + s0, fs);
          tmem_ld32(tl + kColD1 + s0, d);
          tmem_wait_ld();
          if (fast) {  // uniform per chunk: the common case issues no exponentials
#pragma unroll
            for (int e = 0; e < 32; ++e) d[e] = (s0 + e <= r && r < n) ? d[e] * (fr * fs[e]) : 0.f;
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int sc = s0 + e;
              d[e] = (sc <= r && r < n) ? d[e] * exp2f(b2r - fs[e]) : 0.f;
            }
          }
          store_row32_bf16(sm + L.p + (uint32_t)(j & 1) * 8192u, 8192, r, s0, d);
        }
      } else if (kg >= kC) {
        const int r = kg - kC;
        const float b2r = ms[kMsB2 + r], ar = ms[kMsAR + r], br = ms[kMsBeta + r];
#pragma unroll 1
        for (int s0 = 0; s0 < kC; s0 += 32) {
          float d[32], fs[32];
          load32(ms + (fast ? kMsVS : kMsB2) + s0, fs);
          tmem_ld32(tl + kColD1 + s0, d);
          tmem_wait_ld();
          if (fast) {
#pragma unroll
            for (int e = 0; e < 32; ++e) d[e] = (s0 + e < r && r < n) ? round_tf32(d[e] * (ar * fs[e])) : 0.f;
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int sc = s0 + e;
              d[e] = (sc < r && r < n) ? round_tf32(d[e] * (br * exp2f(b2r - fs[e]))) : 0.f;
            }
          }
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4 *>(Af + r * kAp + s0 + 4 * q) =
                make_float4(d[4 * q], d[4 * q + 1], d[4 * q + 2], d[4 * q + 3]);
        }
      }
      tc_fence_before();
      if (!group_all(okp, kBarKG)) break;
      if (kg == 0) mbar_arrive(d1_free);
      // ---- T = (I + A)^-1: 16x16 diagonal blocks, then three block levels
      if (kg < kC) diag_inverse_16(Af, Tf, kg >> 4, kg & 15);
      group_sync(kBarKG);
      // off-diagonal blocks level by level: T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj,
      // one warp per 16x16 output block (tf32 warp MMAs)
      {
        const int kw = kg >> 5;
#pragma unroll 1
        for (int lvl = 1; lvl < 4; ++lvl) {
          if (kw < 4 - lvl) {
            const int ib = kw + lvl, jb = kw;
            float acc[2][4] = {};
            for (int kb = jb; kb < ib; ++kb)
              block_mma_16(acc, Af + ib * 16 * kAp + kb * 16, Tf + kb * 16 * kAp + jb * 16, lane);
            float *Tij = Tf + ib * 16 * kAp + jb * 16;
            block_store_16(Tij, acc, 1.f, lane);  // X parked in its output block
            __syncwarp();
            float acc2[2][4] = {};
            block_mma_16(acc2, Tf + ib * 16 * kAp + ib * 16, Tij, lane);
            __syncwarp();
            block_store_16(Tij, acc2, -1.f, lane);
          }
          group_sync(kBarKG);
        }
      }
      // ---- T' and T'' (bf16) once chunk j-1 has finished with the buffers
      ok = wait_or_abort(kfree, (j & 1) ^ 1, abort_flag, p.status);
      if (!group_all(ok, kBarKG)) break;
      {
        const int r = kg >> 1, g0 = (kg & 1) * 4;
        float tv[32], bt[32], bb[32];
        load32(ms + kMsBeta + g0 * 8, bt);
        load32(ms + kMsBEB + g0 * 8, bb);
        load32(Tf + r * kAp + g0 * 8, tv);
#pragma unroll
        for (int e = 0; e < 32; ++e) tv[e] = (g0 * 8 + e <= r) ? tv[e] : 0.f;
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) {
          const int g8 = g0 + gi;
          float f1[8], f2[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            f1[e] = tv[gi * 8 + e] * bt[gi * 8 + e];
            f2[e] = tv[gi * 8 + e] * bb[gi * 8 + e];
          }
          *reinterpret_cast<uint4 *>(sm + L.tp + sw128_off(r, g8 * 8)) = pack8(f1);
          *reinterpret_cast<uint4 *>(sm + L.tpp + sw128_off(r, g8 * 8)) = pack8(f2);
        }
      }
      fence_proxy_async();
      group_sync(kBarKG);
      if (kg == 0) {
        mbar_arrive(t_ready);        // T'' for the W MMA
        mbar_arrive(&key_ready[s]);  // T' and P for the state side
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 3) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

int launch_chunk_delta(const ChunkParams &p, cudaStream_t stream) {
  if (p.dk != DK || p.dv != DV) {
    set_error("la_chunk_fwd: the pipelined delta-rule kernel takes dk = dv = 128");
    return LA_ERR_UNSUPPORTED;
  }
  if (!encode_fn()) {
    set_error("la_chunk_fwd: cuTensorMapEncodeTiled is unavailable");
    return LA_ERR_CUDA;
  }
  const DLayout L = d_layout();
  const size_t smem = L.total + 1024;
  if (smem > 232448) {
    set_error("la_chunk_fwd: delta-rule kernel needs %zu bytes of shared memory", smem);
    return LA_ERR_UNSUPPORTED;
  }
  const int BH = p.B * p.H;
  CUtensorMap mq, mk, mv;
  const bool ok = make_map(&mq, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DK, p.T, BH, 64,
                           CU_TENSOR_MAP_SWIZZLE_128B) &&
                  make_map(&mk, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DK, p.T, BH, 64,
                           CU_TENSOR_MAP_SWIZZLE_128B) &&
                  make_map(&mv, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, p.T, BH, 64,
                           CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) {
    set_error("la_chunk_fwd: cuTensorMapEncodeTiled rejected a tensor map");
    return LA_ERR_CUDA;
  }
  cudaError_t e =
      cudaFuncSetAttribute(chunk_delta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) {
    chunk_delta_kernel<<<BH, kThreads, smem, stream>>>(p, mq, mk, mv);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_error("la_chunk_fwd: delta-rule kernel launch failed: %s", cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  return LA_OK;
}

}  // namespace la
