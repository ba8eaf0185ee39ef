// Chunk forward for the gated delta rule on a pair of CTAs per head (a
// thread-block cluster of two), bf16 inputs, fp32 state, dk = dv = 128.
//
// Same arithmetic as the one-CTA kernel (la_chunk_delta.cu, "Talk Linear
// Attention" section 6.2, WY/UT form):
//
//   A_rs = beta_r e^{b_r - b_s} k_r.k_s (s < r),  T = (I + A)^-1
//   W    = T diag(beta e^b) K,  U = T diag(beta) V - W S_prev
//   O    = Diag(e^b) Q S_prev + P U,  S <- e^{b_last} S_prev + Kt^T U
//
// but split two ways:
//   * by value columns: every value column of S evolves on its own (U's
//     column v depends only on S's column v), so CTA r of the pair owns the
//     64 value columns 64r .. 64r + 63 of S, U and O;
//   * by chunks for the key side: the S-independent part of a chunk (P, A,
//     the triangular solve, T', W) is the same for both CTAs, so CTA (j mod 2)
//     computes it for chunk j and ships P, T' and -W to the other CTA's shared
//     memory with one bulk copy each (cluster address space, completion on
//     the receiver's mbarrier). Each key group therefore solves every other
//     chunk.
// The bf16 copy of S^T, the bf16 U^T and the key side's bf16 K^T are A
// operands taken from tensor memory (packed pairs along K), which keeps shared
// memory for the exchange buffers; the K^T copy frees the key side's [Q; K]
// buffer for the next own chunk as soon as the scores MMA has read it. Value
// rows 64..127 of the 128-row operands are zero.
//
// Roles (384 threads per CTA): warp 0 producer (TMA tiles, gate/beta prefix),
// warp 1 key-side MMAs (D1, W) for this CTA's chunks, warp 2 state-side MMAs
// (U, O, state update) for every chunk, warp 3 TMEM owner, warps 4-7 state
// group (in-place Qt, state round trip, U epilogue, output epilogue;
// warps 4-5 hold the 64 live value rows), warps 8-11 key group (P, A,
// triangular solve, T', T'', -W, the exchange). All waits are bounded.
#include <cstdlib>

#include "la_tc_common.cuh"
#include "la_wy.cuh"

namespace la {
namespace {

using namespace sm100;
using namespace tc;
using namespace wy;

constexpr int kThreads = 384;
constexpr int DK = 128, DV = 128, NV = 64;  // NV: value columns per CTA
constexpr int kNS = 2;                      // q/k/v stages (chunk j in stage j % 2)
constexpr int kNM = 3;                      // per-chunk scalar slots of the state side
constexpr uint32_t kTmemCols = 512;
// S fp32 (128), S^T bf16 copy (64 packed), D1 (64), W^T (64), U^T (64; the U
// epilogue packs U^T into its first 32 columns and U^T Diag(e^{b_last - b})
// into the other 32), O (64), K^T of the key side's chunk (32 packed)
constexpr uint32_t kColS = 0, kColSC = 128, kColD1 = 192, kColW = 256, kColU = 320, kColO = 384, kColKT = 448;
constexpr int kSG = 128, kKG = 256;
constexpr int kBarSG = 1, kBarKG = 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kFastLimit = 100.f;
constexpr uint32_t kKeyBytes = 8192u + 8192u + 16384u;  // P, T', -W of one chunk

// per-chunk scalars (floats) of the key side (own chunks, two slots)
constexpr int kMsB2 = 0, kMsBeta = 128, kMsFast = 194, kMsF = 256, kMsVS = 320, kMsBEB = 384, kMsAR = 448,
              kMsBytes = 2048;
// ... and of the state side (every chunk): e^b, e^{b_last - b}, e^{b_last}
constexpr int kSsEB = 0, kSsVS = 64, kSsDec = 128, kSsBytes = 1024;

__host__ __device__ inline uint32_t up1k(uint32_t x) { return (x + 1023u) & ~1023u; }

struct PLayout {
  uint32_t qk, v, stage;  // inside a stage
  uint32_t zero, p, tp, wn, kt, af, tf, misc, kms, bar, total;
};

// Identical in both CTAs of a pair: the exchange addresses one buffer in the
// other CTA by its own offset.
__host__ __device__ inline PLayout p_layout() {
  PLayout L;
  uint32_t o = 0;
  L.qk = o; o += 32768u;
  L.v = o; o += 8192u;  // this CTA's 64 value columns
  L.stage = o;
  o = L.stage * kNS;
  L.zero = o; o += 8192u;                // value rows 64..127 of V^T (MN-major atom of zeros)
  L.p = o; o += 2u * 8192u;              // P of chunks owned by CTA b: buffer b
  L.tp = o; o += 2u * 8192u;             // T' = T diag(beta), bf16 [r][s]
  L.wn = o; o += 2u * 16384u;            // -W, MN-major [c][r]
  L.kt = o; o += 32768u;                 // [Q; K] of this CTA's next chunk, for the key side
  L.af = o; o += up1k(kC * kAp * 4u);    // A, fp32; after the solve T'' = T diag(beta e^b), bf16
  L.tf = o; o += up1k(kC * kAp * 4u);    // T, fp32
  L.misc = o; o += kNM * kSsBytes;       // state-side scalars, every chunk
  L.kms = o; o += 2u * kMsBytes;         // key-side scalars, own chunks
  L.bar = o; o += 512u;
  L.total = o;
  return L;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
chunk_delta_pair_kernel(const ChunkParams p, const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const PLayout L = p_layout();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int bh = blockIdx.x >> 1, v_base = (int)rank * NV;
  const int T = p.T, nchunks = (T + kC - 1) / kC;
  const bool gated = p.g != nullptr;

  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.bar);
  uint64_t *full = bars, *empty = bars + 2, *mfree = bars + 4;                     // [2], [2], [4]
  uint64_t *d1_full = bars + 8, *d1_free = bars + 9, *t_ready = bars + 10, *w_full = bars + 11;
  uint64_t *kd_full = bars + 12, *kd_free = bars + 14;                               // [2], [2]
  uint64_t *s_ready = bars + 16, *u_full = bars + 17, *u_ready = bars + 18, *s_done = bars + 19;
  uint64_t *o_done = bars + 20, *o_free = bars + 21, *kt_free = bars + 22, *drain = bars + 24;  // 1, 1, 1, [2]
  uint64_t *kt_full = bars + 26, *kms_free = bars + 27;                              // 1, [2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 30);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  float *Af = reinterpret_cast<float *>(sm + L.af);
  float *Tf = reinterpret_cast<float *>(sm + L.tf);
  auto stage = [&](int s) { return sm + (uint32_t)s * L.stage; };
  auto mslot = [&](int j) { return reinterpret_cast<float *>(sm + L.misc + (uint32_t)(j % kNM) * kSsBytes); };
  auto kslot = [&](int n) { return reinterpret_cast<float *>(sm + L.kms + (uint32_t)(n & 1) * kMsBytes); };
  auto pbuf = [&](int b) { return sm + L.p + (uint32_t)b * 8192u; };
  auto tpbuf = [&](int b) { return sm + L.tp + (uint32_t)b * 8192u; };
  auto wnbuf = [&](int b) { return sm + L.wn + (uint32_t)b * 16384u; };

  if (warp == 3) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&full[s], 2);   // TMA bytes + the producer's gate prefix
      mbar_init(&empty[s], 1);  // state-side MMA commit after the chunk's last MMA
    }
    for (int m = 0; m < kNM; ++m) mbar_init(&mfree[m], 1);
    mbar_init(d1_full, 1);
    mbar_init(d1_free, 1);
    mbar_init(t_ready, 1);
    mbar_init(w_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&kd_full[b], 1);  // own: the key group's arrive; other: arm + the bulk copies' bytes
      mbar_init(&kd_free[b], 2);  // (own buffer only) both CTAs have consumed the chunk's key data
      mbar_init(&drain[b], 1);
    }
    mbar_init(o_done, 1);
    mbar_init(o_free, 1);
    mbar_init(kt_free, 1);  // the key group has its scores and its K^T copy
    mbar_init(s_ready, 1);
    mbar_init(u_full, 1);
    mbar_init(u_ready, 1);
    mbar_init(s_done, 1);
    mbar_init(kt_full, 2);  // TMA bytes + the key producer's gate prefix
    mbar_init(&kms_free[0], 1);
    mbar_init(&kms_free[1], 1);
    *abort_flag = 0;
    // the other CTA's first chunk (chunk `peer`) arrives by bulk copy
    if ((int)peer < nchunks) mbar_arrive_expect_tx(&kd_full[peer], kKeyBytes);
    fence_mbar_init();
  }
  for (int i = tid; i < 512; i += kThreads) reinterpret_cast<uint4 *>(sm + L.zero)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async();
  tc_fence_before();
  // barriers of both CTAs exist before either sends anything
  cluster_sync_all();
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
    constexpr uint32_t bytes = 2u * DK * kC * 2u + NV * kC * 2u;
    int issued = 0;
    for (int j = 0; j < nchunks; ++j) {
      const int s = j % kNS, t0 = j * kC;
      int ok = 1;
      if (lane == 0) ok = wait_or_abort(&mfree[j % kNM], ((j / kNM) & 1) ^ 1, abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      {  // state-side scalars of chunk j: e^b (Qt), e^{b_last - b} (U for the state update), e^{b_last}
        float *ms = mslot(j);
        const int t = t0 + lane;
        const float g0 = (gated && t < T) ? __ldg(p.g + (size_t)bh * T + t) : 0.f;
        const float g1 = (gated && t + 32 < T) ? __ldg(p.g + (size_t)bh * T + t + 32) : 0.f;
        float v0 = g0 * kLog2e, v1 = g1 * kLog2e;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float a0 = __shfl_up_sync(0xffffffffu, v0, off);
          const float a1 = __shfl_up_sync(0xffffffffu, v1, off);
          if (lane >= off) { v0 += a0; v1 += a1; }
        }
        v1 += __shfl_sync(0xffffffffu, v0, 31);
        const float bl = __shfl_sync(0xffffffffu, v1, 31);
        ms[kSsEB + lane] = exp2f(v0);
        ms[kSsEB + lane + 32] = exp2f(v1);
        ms[kSsVS + lane] = exp2f(bl - v0);
        ms[kSsVS + lane + 32] = exp2f(bl - v1);
        if (lane == 0) ms[kSsDec] = exp2f(bl);
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
        }
        tma_load_3d(st + L.v, &tm_v, &full[s], v_base, t0, bh);
        mbar_arrive(&full[s]);
        // the load of chunk j + kNS waits for this chunk's last MMA; warm L2 now
        if (j + kNS < nchunks) {
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            tma_prefetch_3d(&tm_q, 64 * a, t0 + kNS * kC, bh);
            tma_prefetch_3d(&tm_k, 64 * a, t0 + kNS * kC, bh);
          }
          tma_prefetch_3d(&tm_v, v_base, t0 + kNS * kC, bh);
        }
      }
      issued = j + 1;
    }
    if (lane == 0)
      for (int j = (issued > kNS ? issued - kNS : 0); j < issued; ++j)
        (void)mbar_wait_bounded(&full[j % kNS], (j / kNS) & 1, kSpinLimit);
  } else if (warp == 3) {
    // ------------------------------------------- key producer (own chunks)
    // [Q; K] of this CTA's next chunk into its own buffer as soon as the key
    // group has the previous one's scores and K^T copy, and the key-side
    // scalars, so that the key side never waits for the state side to recycle
    // a stage.
    for (int j = (int)rank, n = 0; j < nchunks; j += 2, ++n) {
      const int t0 = j * kC;
      int ok = 1;
      if (lane == 0) ok = wait_or_abort(&kms_free[n & 1], ((n >> 1) & 1) ^ 1, abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      {
        float *ms = kslot(n);
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
        if (lane == 0) ms[kMsFast] = (-bl < kFastLimit) ? 1.f : 0.f;
        __syncwarp();
      }
      // the buffer is free once the previous own chunk's D1 MMA and K^T copy are done
      if (lane == 0 && n > 0) ok = wait_or_abort(kt_free, (n - 1) & 1, abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(kt_full, 32768u);
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          tma_load_3d(sm + L.kt + a * 16384, &tm_q, kt_full, 64 * a, t0, bh);
          tma_load_3d(sm + L.kt + a * 16384 + 8192, &tm_k, kt_full, 64 * a, t0, bh);
        }
        mbar_arrive(kt_full);
        // the next own chunk's load waits for this chunk's scores; warm L2 now
        if (j + 2 < nchunks) {
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            tma_prefetch_3d(&tm_q, 64 * a, t0 + 2 * kC, bh);
            tma_prefetch_3d(&tm_k, 64 * a, t0 + 2 * kC, bh);
          }
        }
      }
    }
    if (lane == 0) {  // no copy in flight when the CTA leaves
      const int nown = (nchunks - (int)rank + 1) / 2;
      if (nown > 0) (void)mbar_wait_bounded(kt_full, (nown - 1) & 1, kSpinLimit);
    }
  } else if (warp == 1) {
    // ------------------------------------ key-side MMAs of this CTA's chunks
    if (lane == 0) {
      constexpr uint32_t id_d1 = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t id_w = idesc_bf16_f32(128, 64, false, false);
      const uint32_t a_tpp = smem_u32(sm + L.af), a_qk = smem_u32(sm + L.kt);
      const uint64_t d_qk = desc_sw128(a_qk, 16, 1024), d_tpp = desc_sw128(a_tpp, 16, 1024);
      // D1 = [Q; K] K^T of own chunk n once the key group has read the previous one
      auto issue_d1 = [&](int n) -> bool {
        if (!wait_or_abort(kt_full, n & 1, abort_flag, p.status)) return false;
        if (!wait_or_abort(d1_free, (n & 1) ^ 1, abort_flag, p.status)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16(tbase + kColD1, desc_add(d_qk, ko), desc_add(d_qk, ko + 8192), id_d1, kk > 0);
        }
        mma_commit(d1_full);
        return true;
      };
      const int nown = (nchunks - (int)rank + 1) / 2;
      bool ok = nown > 0 && issue_d1(0);
      for (int n = 0; n < nown && ok; ++n) {
        // the next own chunk's scores, once the key group has consumed these
        if (n + 1 < nown && !issue_d1(n + 1)) break;
        // W^T = K^T T''^T: K^T from its TMEM copy (M = dk), T'' K-major
        if (!wait_or_abort(t_ready, n & 1, abort_flag, p.status)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16_ts(tbase + kColW, tbase + kColKT + kk * 8, desc_add(d_tpp, kk * 32), id_w, kk > 0);
        mma_commit(w_full);
      }
      mma_commit(&drain[0]);
      (void)mbar_wait_bounded(&drain[0], 0, kSpinLimit);
    }
  } else if (warp == 2) {
    // ------------------------------- state-side MMAs (every chunk): U, O, S
    if (lane == 0) {
      constexpr uint32_t id_ut = idesc_bf16_f32(128, 64, true, false);   // V^T T'^T
      constexpr uint32_t id_us = idesc_bf16_f32(128, 64, false, true);   // S^T (-W)^T, S^T from TMEM
      constexpr uint32_t id_o1 = idesc_bf16_f32(128, 64, false, false);  // S^T Qt^T
      constexpr uint32_t id_su = idesc_bf16_f32(128, DK, false, true);   // U^T Kt, from TMEM
      constexpr uint32_t id_o2 = idesc_bf16_f32(128, 64, false, false);  // U^T P^T
      const uint32_t a_zero = smem_u32(sm + L.zero);
      for (int i = 0; i < nchunks; ++i) {
        const int s = i % kNS, b = i & 1;
        if (!wait_or_abort_cluster(&kd_full[b], (i >> 1) & 1, abort_flag, p.status)) break;
        if (!wait_or_abort(s_ready, i & 1, abort_flag, p.status)) break;
        tc_fence_after();
        uint8_t *st = stage(s);
        const uint32_t a_v = smem_u32(st + L.v), a_qk = smem_u32(st + L.qk);
        const uint32_t a_tp = smem_u32(tpbuf(b)), a_wn = smem_u32(wnbuf(b)), a_p = smem_u32(pbuf(b));
        const uint32_t d_o = tbase + kColO;
        // base descriptors of this chunk's operands (constant offsets per K step below)
        const uint64_t dv = desc_sw128(a_v, a_zero - a_v, 1024), dtp = desc_sw128(a_tp, 16, 1024),
                       dwn = desc_sw128(a_wn, 8192, 1024), dqk = desc_sw128(a_qk, 16, 1024),
                       dp = desc_sw128(a_p, 16, 1024), dkmn = desc_sw128(a_qk + 8192, 16384, 1024);
        // V^T (value rows 64..127 from the zero atom: LBO spans the two MN blocks)
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tbase + kColU, desc_add(dv, kk * 2048), desc_add(dtp, kk * 32), id_ut, kk > 0);
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk)
          mma_bf16_ts(tbase + kColU, tbase + kColSC + kk * 8, desc_add(dwn, kk * 2048), id_us, 1);
        mma_commit(u_full);
        // O is single-buffered: the previous chunk's output epilogue runs during this U
        if (i > 0 && !wait_or_abort(o_free, (i - 1) & 1, abort_flag, p.status)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16_ts(d_o, tbase + kColSC + kk * 8, desc_add(dqk, ko), id_o1, kk > 0);
        }
        if (!wait_or_abort(u_ready, i & 1, abort_flag, p.status)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16_ts(d_o, tbase + kColU + kk * 8, desc_add(dp, kk * 32), id_o2, 1);
        // S^T += (U^T Diag(e^{b_last - b})) K: the decay to the chunk end rides on U, so K stays unscaled
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16_ts(tbase + kColS, tbase + kColU + 32 + kk * 8,
                      desc_add(dkmn, kk * 2048), id_su, 1);
        mma_commit(s_done);
        mma_commit(o_done);
        mma_commit(&empty[s]);
      }
      mma_commit(&drain[1]);
      (void)mbar_wait_bounded(&drain[1], 0, kSpinLimit);
    }
  } else if (tid >= kSG && tid < kKG) {
    // ------------------------------------------------------------ state group
    const int v = tid - kSG;
    const bool live = v < NV;  // warps 4-5: the value rows this CTA owns
    if (live) {
#pragma unroll 1
      for (int c0 = 0; c0 < DK; c0 += 32) {
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = p.S0 ? p.S0[((size_t)bh * DK + c0 + e) * DV + v_base + v] : 0.f;
        tmem_st32(tl + kColS + c0, x);
      }
    } else {  // rows 64..127 of S and of its bf16 copy stay zero
      float z[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) z[e] = 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < DK; c0 += 32) tmem_st32(tl + kColS + c0, z);
      tmem_st32(tl + kColSC, z);
      tmem_st32(tl + kColSC + 32, z);
    }
    tmem_wait_st();
    bool alive = true;
    for (int i = 0; i <= nchunks && alive; ++i) {
      if (i < nchunks) {
        const int s = i % kNS;
        const float *ms = mslot(i);
        // the tiles are in and the previous chunk's MMAs have finished (the key
        // side reads its own copy of [Q; K])
        bool ok = wait_or_abort(&full[s], (i / kNS) & 1, abort_flag, p.status);
        if (ok && i > 0) ok = wait_or_abort(s_done, (i - 1) & 1, abort_flag, p.status);
        if (!group_all(ok, kBarSG)) { alive = false; break; }
        if (i > 0 && v == 0) {
          // chunk i-1's key data is consumed here: tell its writer, and expect
          // the writer's next chunk (i+1) if it is the other CTA
          const int bp = (i - 1) & 1;
          mbar_arrive_cluster(mapa_shared(smem_u32(&kd_free[bp]), (uint32_t)bp));
          if ((uint32_t)bp != rank && i + 1 < nchunks) mbar_arrive_expect_tx(&kd_full[bp], kKeyBytes);
        }
        tc_fence_after();
        // Qt = Diag(e^b) Q in place: warps 6-7 (row v - 64), while warps 4-5 do the round trip
        if (gated && !live) {
          uint8_t *qk = stage(s) + L.qk;
          const int r = v - kC;
          const float rs = ms[kSsEB + r];
#pragma unroll 1
          for (int g0 = 0; g0 < 16; g0 += 4) {
            uint4 u[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
              u[q] = *reinterpret_cast<const uint4 *>(qk + ((g0 + q) >> 3) * 16384 + sw128_off(r, ((g0 + q) & 7) * 8));
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float f[8];
              unpack8(u[q], f);
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] *= rs;
              *reinterpret_cast<uint4 *>(qk + ((g0 + q) >> 3) * 16384 + sw128_off(r, ((g0 + q) & 7) * 8)) = pack8(f);
            }
          }
        }
        // state round trip: bf16 copy of S_prev into TMEM (packed pairs), decay in place
        if (live) {
          const float dec = ms[kSsDec];
#pragma unroll 1
          for (int c0 = 0; c0 < DK; c0 += 64) {
            float x[32], y[32], pk[16];
            tmem_ld32(tl + kColS + c0, x);
            tmem_ld32(tl + kColS + c0 + 32, y);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = __uint_as_float(pack_bf16(x[2 * e], x[2 * e + 1]));
            tmem_st16(tl + kColSC + c0 / 2, pk);
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = __uint_as_float(pack_bf16(y[2 * e], y[2 * e + 1]));
            tmem_st16(tl + kColSC + c0 / 2 + 16, pk);
            if (gated) {
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                x[e] *= dec;
                y[e] *= dec;
              }
              tmem_st32(tl + kColS + c0, x);
              tmem_st32(tl + kColS + c0 + 32, y);
            }
          }
          tmem_wait_st();
        }
        fence_proxy_async();
        tc_fence_before();
        group_sync(kBarSG);
        if (v == 0) mbar_arrive(s_ready);
      }
      if (i > 0) {
        // output epilogue of chunk c = i - 1: its MMAs completed before this chunk's round
        // trip, and it fills the wait for this chunk's U MMA
        const int c = i - 1, n = min(kC, T - c * kC);
        bool ok = wait_or_abort(o_done, c & 1, abort_flag, p.status);
        if (!group_all(ok, kBarSG)) { alive = false; break; }
        tc_fence_after();
        if (live) {
          __nv_bfloat16 *og =
              static_cast<__nv_bfloat16 *>(p.o) + ((size_t)bh * T + (size_t)c * kC) * DV + v_base;
          const bool odd = lane & 1;
#pragma unroll 1
          for (int r0 = 0; r0 < kC; r0 += 16) {
            float a[16];
            tmem_ld16(tl + kColO + r0, a);
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
        }
        tc_fence_before();
        group_sync(kBarSG);
        if (v == 0) {
          mbar_arrive(o_free);
          mbar_arrive(&mfree[c % kNM]);
        }
      }
      if (i < nchunks) {
        // U epilogue: U^T (fp32) -> bf16 pairs in place, the A operand of the O and state MMAs
        bool ok = wait_or_abort(u_full, i & 1, abort_flag, p.status);
        if (!group_all(ok, kBarSG)) { alive = false; break; }
        tc_fence_after();
        if (live) {
          const float *ms = mslot(i);
          float x[32], y[32], pk[32];
          tmem_ld32(tl + kColU, x);
          tmem_ld32(tl + kColU + 32, y);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            pk[e] = __uint_as_float(pack_bf16(x[2 * e], x[2 * e + 1]));
            pk[16 + e] = __uint_as_float(pack_bf16(y[2 * e], y[2 * e + 1]));
          }
          tmem_st32(tl + kColU, pk);  // U^T for the output MMA
          float f[32];
          load32(ms + kSsVS, f);
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = __uint_as_float(pack_bf16(x[2 * e] * f[2 * e], x[2 * e + 1] * f[2 * e + 1]));
          load32(ms + kSsVS + 32, f);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[16 + e] = __uint_as_float(pack_bf16(y[2 * e] * f[2 * e], y[2 * e + 1] * f[2 * e + 1]));
          tmem_st32(tl + kColU + 32, pk);  // U^T Diag(e^{b_last - b}) for the state update
          tmem_wait_st();
        }
        tc_fence_before();
        group_sync(kBarSG);
        if (v == 0) mbar_arrive(u_ready);
      }
    }
    if (alive && p.S_final) {
      bool ok = wait_or_abort(s_done, (nchunks - 1) & 1, abort_flag, p.status);
      if (group_all(ok, kBarSG) && live) {
        tc_fence_after();
        for (int c0 = 0; c0 < DK; c0 += 32) {
          float x[32];
          tmem_ld32(tl + kColS + c0, x);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) p.S_final[((size_t)bh * DK + c0 + e) * DV + v_base + v] = x[e];
        }
      }
    }
  } else if (tid >= kKG) {
    // ------------------------------------- key group: this CTA's chunks only
    const int kg = tid - kKG;
    const int b = (int)rank;
    uint8_t *pb = pbuf(b), *tpb = tpbuf(b), *wnb = wnbuf(b);
    // K^T of the own chunk into TMEM (lane = key channel kg, packed token pairs), the A
    // operand of the W MMA, so that the [Q; K] buffer can take the next own chunk
    auto kt_copy = [&]() {
      const uint8_t *kb = sm + L.kt + (uint32_t)(kg >> 6) * 16384u + 8192u;
      const uint32_t c = (uint32_t)kg & 63u;
      float pk[32];
#pragma unroll
      for (int r2 = 0; r2 < 32; ++r2) {
        const uint32_t lo = *reinterpret_cast<const uint16_t *>(kb + sw128_off(2 * r2, c));
        const uint32_t hi = *reinterpret_cast<const uint16_t *>(kb + sw128_off(2 * r2 + 1, c));
        pk[r2] = __uint_as_float(lo | (hi << 16));
      }
      tmem_st32(tl + kColKT, pk);
      tmem_wait_st();
      tc_fence_before();
    };
    for (int j = (int)rank, n = 0; j < nchunks; j += 2, ++n) {
      const int nrow = min(kC, T - j * kC);
      float *ms = kslot(n);
      // scalars and D1 in
      bool ok = wait_or_abort(kt_full, n & 1, abort_flag, p.status);
      if (ok) ok = wait_or_abort(d1_full, n & 1, abort_flag, p.status);
      if (!group_all(ok, kBarKG)) break;
      tc_fence_after();
      const bool fast = ms[kMsFast] != 0.f;
      // ---- A from D1 lanes 64..127 (K K^T rows) by warps 10-11: only private buffers until
      // the solve is done; warps 8-9 copy their half of K^T meanwhile, warps 10-11 after
      if (kg < kC) kt_copy();
      if (kg >= kC) {
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
            for (int e = 0; e < 32; ++e) d[e] = (s0 + e < r && r < nrow) ? round_tf32(d[e] * (ar * fs[e])) : 0.f;
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int sc = s0 + e;
              d[e] = (sc < r && r < nrow) ? round_tf32(d[e] * (br * exp2f(b2r - fs[e]))) : 0.f;
            }
          }
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4 *>(Af + r * kAp + s0 + 4 * q) =
                make_float4(d[4 * q], d[4 * q + 1], d[4 * q + 2], d[4 * q + 3]);
        }
        kt_copy();
      }
      group_sync(kBarKG);
      if (kg == 0) mbar_arrive(kt_free);  // the D1 MMA and the K^T copy are done with [Q; K]
      // ---- T = (I + A)^-1: 16x16 diagonal blocks, then three block levels
      if (kg < kC) diag_inverse_16(Af, Tf, kg >> 4, kg & 15);
      group_sync(kBarKG);
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
      // ---- P from D1 lanes 0..63 (Q K^T rows) into the exchange buffer, once both CTAs
      // have consumed this CTA's previous chunk (P, T' and -W buffers free)
      ok = true;
      if (kg == 0) ok = wait_or_abort_cluster(&kd_free[b], (n & 1) ^ 1, abort_flag, p.status);
      if (!group_all(ok, kBarKG)) break;
      if (kg < kC) {
        const int r = kg;
        const float b2r = ms[kMsB2 + r], fr = ms[kMsF + r];
#pragma unroll 1
        for (int s0 = 0; s0 < kC; s0 += 32) {
          float d[32], fs[32];
          load32(ms + (fast ? kMsVS : kMsB2) + s0, fs);
          tmem_ld32(tl + kColD1 + s0, d);
          tmem_wait_ld();
          if (fast) {
#pragma unroll
            for (int e = 0; e < 32; ++e) d[e] = (s0 + e <= r && r < nrow) ? d[e] * (fr * fs[e]) : 0.f;
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int sc = s0 + e;
              d[e] = (sc <= r && r < nrow) ? d[e] * exp2f(b2r - fs[e]) : 0.f;
            }
          }
          store_row32_bf16(pb, 8192, r, s0, d);
        }
      }
      tc_fence_before();
      group_sync(kBarKG);
      if (kg == 0) mbar_arrive(d1_free);
      // ---- T' (exchange buffer) and T'' (the dead A buffer), bf16
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
          *reinterpret_cast<uint4 *>(tpb + sw128_off(r, g8 * 8)) = pack8(f1);
          *reinterpret_cast<uint4 *>(sm + L.af + sw128_off(r, g8 * 8)) = pack8(f2);
        }
      }
      fence_proxy_async();
      group_sync(kBarKG);
      if (kg == 0) {
        mbar_arrive(t_ready);  // T'' for the W MMA
        mbar_arrive(&kms_free[n & 1]);
      }
      // ---- -W as the MN-major B operand [c][r] (TMEM lane = key channel c)
      ok = wait_or_abort(w_full, n & 1, abort_flag, p.status);
      if (!group_all(ok, kBarKG)) break;
      tc_fence_after();
#pragma unroll 1
      for (int r0 = 0; r0 < kC; r0 += 32) {
        float x[32];
        tmem_ld32(tl + kColW + r0, x);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = -x[e];
        store_row32_bf16(wnb, 16384, kg, r0, x);
      }
      fence_proxy_async();
      tc_fence_before();
      group_sync(kBarKG);
      if (kg == 0) {
        mbar_arrive(&kd_full[b]);  // this CTA's state side
        // the other CTA: P, T' and -W by bulk copy, completing its kd_full[b]
        const uint32_t rbar = mapa_shared(smem_u32(&kd_full[b]), peer);
        bulk_copy_to_cluster(mapa_shared(smem_u32(pb), peer), pb, 8192u, rbar);
        bulk_copy_to_cluster(mapa_shared(smem_u32(tpb), peer), tpb, 8192u, rbar);
        bulk_copy_to_cluster(mapa_shared(smem_u32(wnb), peer), wnb, 16384u, rbar);
      }
    }
  }

  tc_fence_before();
  // neither CTA leaves while the other may still address its shared memory
  cluster_sync_all();
  tc_fence_after();
  if (warp == 3) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

int launch_chunk_delta_pair(const ChunkParams &p, cudaStream_t stream) {
  if (p.dk != DK || p.dv != DV) {
    set_error("la_chunk_fwd: the paired delta-rule kernel takes dk = dv = 128");
    return LA_ERR_UNSUPPORTED;
  }
  if (!encode_fn()) {
    set_error("la_chunk_fwd: cuTensorMapEncodeTiled is unavailable");
    return LA_ERR_CUDA;
  }
  const PLayout L = p_layout();
  const size_t smem = L.total + 1024;
  if (smem > 232448) {
    set_error("la_chunk_fwd: paired delta-rule kernel needs %zu bytes of shared memory", smem);
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
      cudaFuncSetAttribute(chunk_delta_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) {
    chunk_delta_pair_kernel<<<(unsigned)(2 * BH), kThreads, smem, stream>>>(p, mq, mk, mv);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_error("la_chunk_fwd: paired delta-rule kernel launch failed: %s", cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  return LA_OK;
}

}  // namespace la
