// Warp-specialised chunk forward for the unit-write modes (plain linear
// attention, elu+1 with normaliser, RetNet decay, scalar decay, GLA gates) on
// tcgen05 + TMEM + TMA, bf16 inputs, fp32 state.
//
// One CTA owns one (b, h) for the whole sequence and keeps S^T in TMEM
// (lane = value column, columns = key axis). Per chunk of C = 64 tokens with
// inclusive log-gate prefix b ("Talk Linear Attention" sections 3.2 and 5.2):
//
//   P    = (Q K^T) ⊙ exp(b_r - b_s) ⊙ M        (scores from D1 = [Q; K] K^T)
//   S^T <- Diag(e^{b_last}) S^T + V^T Kt,   Kt = Diag(e^{b_last - b}) K
//   O^T  = Diag(e^{b}) (S_prev^T Q^T) + V^T P^T
//
// GLA factors the per-channel exp(b_r - b_s) around the chunk midpoint m:
// Q and K are scaled by e^{b - b_m} and e^{b_m - b}, the bf16 state copy by
// e^{b_m}. The state update then uses the same K (e^{b_m - b}), so TMEM holds
// X = S Diag(e^{b_m - b_last}) of the previous chunk: one per-channel factor
// e^{b_m} e^{b_last' - b_m'} (this chunk's midpoint, the previous chunk's
// midpoint-to-end decay) gives both the bf16 copy and the decayed state. elu+1 applies phi to q and k, splits phi(k) into bf16 high and low
// halves for the state update, and divides o by q.z + P 1 (kernel-attention
// notes, sections 13-14).
//
// The outer-product gate (alpha_t beta_t^T, "Talk Linear Attention" section
// 5.4) takes GLA's key-axis fold unchanged and adds the same fold on the
// value axis: V is scaled by e^{bv_m - bv} in place, o by e^{bv - bv_m} in
// the output epilogue (each state-group thread rescans its value column's
// gates, which stay in L2), and the per-column factor e^{bv_m} e^{bv_last' -
// bv_m'} rides on the state round trip next to the key-axis one.
//
// REV (every unit-write mode but elu+1) runs the same recurrence over the
// time-reversed sequence without copying it: chunk j is the 64-row window
// ending at row T-1-64j of the stored tensors (its TMA load may start above
// row 0, where the fill is zero), and its smem row m is reversed row 63-m.
// The per-row gate factors are written to the slots of the smem rows, the
// masks become s >= r, and o lands in stored order, so the anti-causal passes
// of the backward read and write q, k, v, dO, dk, dv where they are. With
// data-dependent gates (scalar, per key channel, per value column), position
// t of a reversed run decays by the gate of the stored token after it (index
// T - t; none at t = 0): the decay between stored tokens s < u is then the
// product of the gates of s+1 .. u, as the backward's anti-causal sums need.
// The per-channel prefixes then run from smem row 63 down to 0, with the
// midpoint at smem row 32 (reversed row 31).
//
// Roles (384 threads):
//   warp 0      TMA producer: q/k/v (and GLA gate) tiles into an ns-stage ring
//   warp 1      issues the score MMA of each chunk
//   warp 2      issues the state-update and output MMAs
//   warp 3      owns the TMEM allocation
//   warps 4-7   state group: per chunk, read S^T from TMEM once to build the
//               bf16 operand copy and apply the decay; then the output
//               epilogue of the previous chunk (overlapping the state MMA)
//   warps 8-11  key group, one chunk ahead: gate prefix, q/k transforms,
//               masked/decayed scores P, Kt in place, elu+1 normaliser
// Every wait is a bounded mbarrier poll; on expiry the CTA raises the device
// status word, every role leaves its loop, in-flight copies and MMAs are
// drained and TMEM is released.
#include "la_tc_common.cuh"

namespace la {
namespace {

using namespace sm100;
using namespace tc;

constexpr int kThreads = 384;
constexpr int kMid = kC / 2 - 1;
constexpr uint32_t kSpin = 1u << 24;  // polls before a wait gives up (well over 100 ms)
constexpr int kNM = 4;                // slots of the per-chunk scalar ring
constexpr uint32_t kTmemCols = 512;
// TMEM columns: state, two score buffers, two output buffers
// O: two 64-column buffers; scalar gates keep the inter-chunk part S^T Q^T in
// its own pair (O1) so that e^{b} is applied in the epilogue, not to Q in place
constexpr uint32_t kColS = 0, kColD1 = 128, kColO = 256, kColO1 = 384;
constexpr int kSG = 128, kKG = 256;    // first thread of each group
constexpr int kBarSG = 1, kBarKG = 2;  // named barriers of the groups
constexpr float kLog2e = 1.4426950408889634f;

// per-stage scalars (floats): log2-domain gate prefix b2, e^{b}, elu+1
// denominators, chunk decay, fast-path flag, per-row factors e^{b - b_last}
// (scores) and e^{b_last - b} (value or key rows), GLA per-channel factors
// (state factor e^{b_m} e^{b_last' - b_m'}, midpoint-to-end decay e^{b_last - b_m}),
// and for the outer-product gate the same two factors per value column
constexpr int kMsB2 = 0, kMsEB = 64, kMsDen = 128, kMsDec = 192, kMsB2L = 193, kMsFast = 194,
              kMsF = 256, kMsVS = 320, kMsBM = 384, kMsLM = 640, kMsBMV = 768, kMsLMV = 896;
// per-key-channel gates (GLA, outer-product gate): a gate tile per stage, midpoint fold
__host__ __device__ constexpr bool chan_gates(int kind) { return kind == kGla || kind == kOuter; }
// bytes of one scalar slot: the per-channel factors need the upper part
__host__ __device__ constexpr uint32_t ms_bytes(int kind) {
  return kind == kOuter ? 4096u : kind == kGla ? 3072u : 1536u;
}
// the 32 KB gate tiles leave no room for an output staging tile: o is stored directly
__host__ __device__ constexpr bool staged_out(int kind) { return !chan_gates(kind); }
// A chunk whose total decay is below 2^-kFastLimit takes the exact path.
constexpr float kFastLimit = 100.f;

__host__ __device__ inline uint32_t up1k(uint32_t x) { return (x + 1023u) & ~1023u; }

// Offsets inside one pipeline stage (released when the chunk's MMAs are
// done), and of the per-CTA buffers after the stages: the bf16 state copy,
// the output staging tile, the ring of per-chunk scalars (released after the
// chunk's output epilogue), elu+1 normaliser, barriers.
struct WsLayout {
  uint32_t qk, v, g, klo, p, stage;  // inside a stage
  uint32_t st, ot, misc, z, tmp, bar, total;
};

__host__ __device__ inline WsLayout ws_layout(int dk, int dv, int kind, int ns) {
  WsLayout L;
  const bool elu = kind == kElu1;
  // the tile holds the key gates; the outer-product gate reuses it for its value-axis prefix
  const int gw = kind == kOuter && dv > dk ? dv : dk;
  const uint32_t qk_bytes = (uint32_t)(dk / 64) * 16384u;
  uint32_t o = 0;
  L.qk = o; o += qk_bytes;
  L.v = o; o += 16384u;  // upper 8 KB is a zero pad when dv = 64
  L.g = o; o += chan_gates(kind) ? up1k((uint32_t)kC * gw * 4u) : 0u;
  L.klo = o; o += elu ? (uint32_t)(dk / 64) * 8192u : 0u;
  L.p = o; o += 8192u;
  L.stage = o;
  o = L.stage * ns;
  L.st = o; o += qk_bytes;
  L.ot = o; o += staged_out(kind) ? 16384u : 0u;
  L.misc = o; o += kNM * ms_bytes(kind);
  L.z = o; o += 512u;
  L.tmp = o; o += 256u;
  L.bar = o; o += 256u;
  L.total = o;
  return L;
}

template <int DK, int DV, int KIND, bool REV>
__global__ void __launch_bounds__(kThreads, 1)
chunk_ws_kernel(const ChunkParams p, int ns, const __grid_constant__ CUtensorMap tm_q,
                const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_o) {
  constexpr bool elu = KIND == kElu1, outer = KIND == kOuter;
  constexpr bool gla = chan_gates(KIND);  // key-axis channel gates (GLA and the outer-product gate)
  constexpr bool sgate = KIND == kRetnet || KIND == kScalar;
  static_assert(!REV || KIND != kElu1, "reversed runs: the unit-write modes without a normaliser");
  // smem rows of the chunk midpoint and of its last token (reversed runs: rows 32 and 0)
  constexpr int kMidRow = REV ? kC - 1 - kMid : kMid, kLastRow = REV ? 0 : kC - 1;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const WsLayout L = ws_layout(DK, DV, KIND, ns);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x, h = bh % p.H;
  const int T = p.T, nchunks = (T + kC - 1) / kC;
  constexpr int Wmem = DV + (elu ? 1 : 0);

  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.bar);
  uint64_t *full = bars, *empty = bars + 3, *qk_ready = bars + 6, *key_ready = bars + 9;
  uint64_t *s_ready = bars + 13, *s_done = bars + 14, *o1_done = bars + 15;
  uint64_t *o_done = bars + 16, *o_free = bars + 18, *drain = bars + 20;
  uint64_t *d1_full = bars + 22, *d1_free = bars + 24, *mfree = bars + 26;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 26 + kNM);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  float *zs = reinterpret_cast<float *>(sm + L.z);
  float *tmp = reinterpret_cast<float *>(sm + L.tmp);
  auto stage = [&](int s) { return sm + (uint32_t)s * L.stage; };
  auto mslot = [&](int j) {
    return reinterpret_cast<float *>(sm + L.misc + (uint32_t)(j % kNM) * ms_bytes(KIND));
  };

  if (warp == 3) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < 3; ++s) {
      mbar_init(&full[s], sgate ? 2 : 1);  // TMA bytes (+ the producer's gate prefix)
      mbar_init(&empty[s], 2);  // key group + state-side MMA commit
      mbar_init(&qk_ready[s], 1);
      mbar_init(&key_ready[s], 1);
    }
    mbar_init(s_ready, 1);
    mbar_init(s_done, 1);
    mbar_init(o1_done, 1);
    for (int m = 0; m < kNM; ++m) mbar_init(&mfree[m], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&d1_full[b], 1);
      mbar_init(&d1_free[b], 1);
      mbar_init(&o_done[b], 1);
      mbar_init(&o_free[b], 1);
      mbar_init(&drain[b], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (DV == 64) {  // zero rows 64..127 of the value operand in every stage
    for (int i = tid; i < ns * 512; i += kThreads)
      reinterpret_cast<uint4 *>(stage(i >> 9) + L.v + 8192)[i & 511] = make_uint4(0, 0, 0, 0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t tl = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Lane 0 streams the tiles; for the scalar-gate modes the whole warp
    // then forms the chunk's log-gate prefix and per-row factors.
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      if (gla) prefetch_tmap(&tm_g);
    }
    constexpr uint32_t bytes = 2u * DK * kC * 2u + DV * kC * 2u + (gla ? DK * kC * 4u : 0u);
    int issued = 0;
    for (int j = 0; j < nchunks; ++j) {
      const int s = j % ns;
      const int t0 = REV ? T - (j + 1) * kC : j * kC;  // first stored row of the tile
      int ok = 1;
      // per-chunk scalars first (their slot frees after the chunk kNM back has
      // been written out), so the gate loads overlap the wait for a stage
      if (lane == 0) ok = wait_or_abort(&mfree[j % kNM], ((j / kNM) & 1) ^ 1, abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (sgate) {
        float *ms = mslot(j);
        const int t = j * kC + lane;  // position in the (possibly reversed) sequence
        float g0, g1;
        if (KIND == kRetnet) {
          const float g = __ldg(p.g + h);
          g0 = (t < T) ? g : 0.f;
          g1 = (t + 32 < T) ? g : 0.f;
        } else if (REV) {  // the gate of the stored token after each position
          g0 = (t >= 1 && t < T) ? __ldg(p.g + (size_t)bh * T + (T - t)) : 0.f;
          g1 = (t + 32 < T) ? __ldg(p.g + (size_t)bh * T + (T - t - 32)) : 0.f;
        } else {
          g0 = (t < T) ? __ldg(p.g + (size_t)bh * T + t) : 0.f;
          g1 = (t + 32 < T) ? __ldg(p.g + (size_t)bh * T + t + 32) : 0.f;
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
        // slots are indexed by the tile's smem row (reversed: row 63 - r)
        const int m0 = REV ? kC - 1 - lane : lane, m1 = REV ? kC / 2 - 1 - lane : lane + 32;
        ms[kMsB2 + m0] = v0;
        ms[kMsB2 + m1] = v1;
        ms[kMsEB + m0] = exp2f(v0);
        ms[kMsEB + m1] = exp2f(v1);
        ms[kMsF + m0] = exp2f(v0 - bl);
        ms[kMsF + m1] = exp2f(v1 - bl);
        ms[kMsVS + m0] = exp2f(bl - v0);
        ms[kMsVS + m1] = exp2f(bl - v1);
        if (lane == 0) {
          ms[kMsDec] = exp2f(bl);
          ms[kMsB2L] = bl;
          ms[kMsFast] = (-bl < kFastLimit) ? 1.f : 0.f;
        }
        __syncwarp();
      }
      if (lane == 0) ok = wait_or_abort(&empty[s], ((j / ns) & 1) ^ 1, abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      uint8_t *st = stage(s);
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
        for (int a = 0; a < DK / 64; ++a) {
          tma_load_3d(st + L.qk + a * 16384, &tm_q, &full[s], 64 * a, t0, bh);
          tma_load_3d(st + L.qk + a * 16384 + 8192, &tm_k, &full[s], 64 * a, t0, bh);
        }
#pragma unroll
        for (int a = 0; a < DV / 64; ++a)
          tma_load_3d(st + L.v + a * 8192, &tm_v, &full[s], 64 * a, t0, bh);
        // (reversed runs: the gates of the stored tokens one row later; rows past T read zero)
        if (gla) tma_load_3d(st + L.g, &tm_g, &full[s], 0, REV ? t0 + 1 : t0, bh);
        if (outer) {  // the value-axis gates are read with plain loads by the key and state groups
          const int g0r = REV ? max(t0 + 1, 0) : t0, g1r = REV ? min(t0 + 1 + kC, T) : min(t0 + kC, T);
          if (g1r > g0r) bulk_prefetch_l2(p.beta + ((size_t)bh * T + g0r) * DV, (uint32_t)(g1r - g0r) * DV * 4u);
        }
        if (sgate) mbar_arrive(&full[s]);  // the gate prefix of this chunk is in place
        // the load of chunk j + ns waits for this chunk's last MMA; warm L2 now
        // (a prefetch is a hint: the reversed run skips a window that starts above row 0)
        if (j + ns < nchunks && (!REV || t0 - ns * kC >= 0)) {
          const int tp = REV ? t0 - ns * kC : t0 + ns * kC;
#pragma unroll
          for (int a = 0; a < DK / 64; ++a) {
            tma_prefetch_3d(&tm_q, 64 * a, tp, bh);
            tma_prefetch_3d(&tm_k, 64 * a, tp, bh);
          }
#pragma unroll
          for (int a = 0; a < DV / 64; ++a) tma_prefetch_3d(&tm_v, 64 * a, tp, bh);
          if (gla) tma_prefetch_3d(&tm_g, 0, REV ? tp + 1 : tp, bh);
        }
      }
      issued = j + 1;
    }
    // copies still in flight must land before the CTA's memory is released
    if (lane == 0)
      for (int j = (issued > ns ? issued - ns : 0); j < issued; ++j)
        (void)mbar_wait_bounded(&full[j % ns], (j / ns) & 1, kSpin);
  } else if (warp == 1) {
    // ---------------------------------------------- score MMA: D1 = [Q;K] K^T
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 64, false, false);
      for (int j = 0; j < nchunks; ++j) {
        const int s = j % ns;
        // tiles that need no elementwise transform are used as soon as they land
        if (!wait_or_abort((elu || gla) ? &qk_ready[s] : &full[s], (j / ns) & 1, abort_flag, p.status))
          break;
        if (!wait_or_abort(&d1_free[j & 1], ((j >> 1) & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t a_qk = smem_u32(stage(s) + L.qk);
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16(tbase + kColD1 + (uint32_t)(j & 1) * 64u, desc_sw128(a_qk + ko, 16, 1024),
                   desc_sw128(a_qk + ko + 8192, 16, 1024), idesc, kk > 0);
        }
        mma_commit(&d1_full[j & 1]);
      }
      mma_commit(&drain[0]);
      (void)mbar_wait_bounded(&drain[0], 0, kSpin);
    }
  } else if (warp == 2) {
    // ------------------------------------------ state update and output MMAs
    if (lane == 0) {
      constexpr uint32_t id_su = idesc_bf16_f32(128, DK, true, true);
      constexpr uint32_t id_o1 = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t id_o2 = idesc_bf16_f32(128, 64, true, false);
      const uint32_t a_st = smem_u32(sm + L.st);
      for (int i = 0; i < nchunks; ++i) {
        const int s = i % ns;
        if (!wait_or_abort(&key_ready[s], (i / ns) & 1, abort_flag, p.status)) break;
        if (!wait_or_abort(s_ready, i & 1, abort_flag, p.status)) break;
        if (!wait_or_abort(&o_free[i & 1], ((i >> 1) & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        uint8_t *st = stage(s);
        const uint32_t a_v = smem_u32(st + L.v), a_qk = smem_u32(st + L.qk), a_p = smem_u32(st + L.p);
        // S^T += V^T Kt (V as MN-major A; Kt rows of the k tile as MN-major B)
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk) {
          const uint64_t dv_ = desc_sw128(a_v + kk * 2048, 8192, 1024);
          mma_bf16(tbase + kColS, dv_, desc_sw128(a_qk + 8192 + kk * 2048, 16384, 1024), id_su, 1);
          if (elu)
            mma_bf16(tbase + kColS, dv_, desc_sw128(smem_u32(st + L.klo) + kk * 2048, 8192, 1024),
                     id_su, 1);
        }
        mma_commit(s_done);
        // O^T = S_prev^T Q^T (bf16 state copy; scalar gates: own buffer, times e^b in the epilogue) ...
        const uint32_t d_o2 = tbase + kColO + (uint32_t)(i & 1) * 64u;
        const uint32_t d_o1 = sgate ? tbase + kColO1 + (uint32_t)(i & 1) * 64u : d_o2;
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16(d_o1, desc_sw128(a_st + ko, 16, 1024), desc_sw128(a_qk + ko, 16, 1024), id_o1, kk > 0);
        }
        mma_commit(o1_done);
        // ... + V^T P^T
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(d_o2, desc_sw128(a_v + kk * 2048, 8192, 1024), desc_sw128(a_p + kk * 32, 16, 1024),
                   id_o2, sgate ? (kk > 0) : 1);
        mma_commit(&o_done[i & 1]);
        mma_commit(&empty[s]);
      }
      mma_commit(&drain[1]);
      (void)mbar_wait_bounded(&drain[1], 0, kSpin);
    }
  } else if (tid >= kSG && tid < kKG) {
    // ------------------------------------------------------------ state group
    const int v = tid - kSG;
    for (int c0 = 0; c0 < DK; c0 += 32) {
      float vals[32];
#pragma unroll
      for (int e = 0; e < 32; ++e)
        vals[e] = (p.S0 && v < DV) ? p.S0[((size_t)bh * DK + c0 + e) * Wmem + v] : 0.f;
      tmem_st32(tl + kColS + c0, vals);
    }
    tmem_wait_st();
    bool alive = true;
    for (int i = 0; i <= nchunks && alive; ++i) {
      if (i < nchunks) {
        const int s = i % ns;
        const float *ms = mslot(i);
        bool ok = wait_or_abort(&key_ready[s], (i / ns) & 1, abort_flag, p.status);
        if (ok && i > 0)
          ok = wait_or_abort(s_done, (i - 1) & 1, abort_flag, p.status) &&
               wait_or_abort(o1_done, (i - 1) & 1, abort_flag, p.status);
        if (!group_all(ok, kBarSG)) { alive = false; break; }
        tc_fence_after();
        // state round trip: bf16 operand copy of S_prev, decay in place
#pragma unroll 1
        for (int c0 = 0; c0 < DK; c0 += 32) {
          float x[32];
          tmem_ld32(tl + kColS + c0, x);
          tmem_wait_ld();
          if (gla) {  // one factor: the bf16 copy is the decayed state
            float fm[32];
            load32(ms + kMsBM + c0, fm);
            if (outer) {  // times this value column's factor
              const float fv = v < DV ? ms[kMsBMV + v] : 0.f;
#pragma unroll
              for (int e = 0; e < 32; ++e) fm[e] *= fv;
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] *= fm[e];
            store_row32_bf16(sm + L.st, 16384, v, c0, x);
            tmem_st32(tl + kColS + c0, x);
          } else {
            store_row32_bf16(sm + L.st, 16384, v, c0, x);
            if (sgate) {
              const float dec = ms[kMsDec];
#pragma unroll
              for (int e = 0; e < 32; ++e) x[e] *= dec;
              tmem_st32(tl + kColS + c0, x);
            }
          }
        }
        tmem_wait_st();
        fence_proxy_async();
        tc_fence_before();
        group_sync(kBarSG);
        if (v == 0) mbar_arrive(s_ready);
      }
      if (i > 0) {
        // output epilogue of chunk c = i - 1 (overlaps the state MMA of chunk i)
        const int c = i - 1, ob = c & 1, n = min(kC, T - c * kC);
        const float *ms = mslot(c);
        bool ok = wait_or_abort(&o_done[ob], (c >> 1) & 1, abort_flag, p.status);
        if (v == 0) bulk_wait_read<0>();  // the previous tile has left the staging buffer
        if (!group_all(ok, kBarSG)) { alive = false; break; }
        tc_fence_after();
        uint8_t *ot = sm + L.ot + (uint32_t)(v >> 6) * 8192u;
        // first stored row of the tile; a reversed window that starts above row 0
        // (the last one when 64 does not divide T) is written row by row, since a
        // TMA store may not start at a negative coordinate
        const int t0c = REV ? T - (c + 1) * kC : c * kC;
        const bool staged = staged_out(KIND) && (!REV || t0c >= 0);
        __nv_bfloat16 *obh = static_cast<__nv_bfloat16 *>(p.o) + (size_t)bh * T * DV;
        const bool odd = lane & 1;
        // outer-product gate: value column v's log2 prefix over the chunk (the key
        // group's scan, redone from L2), carried across the two halves
        float vcar = 0.f, vbm = 0.f;
        const int vrb = REV ? T - (c + 1) * kC + 1 : c * kC;  // stored row of smem row 0's gate
        const float *gvc = outer ? p.beta + (size_t)bh * T * DV + v : nullptr;
        auto vgate = [&](int m) {
          return (v < DV && vrb + m >= 0 && vrb + m < T && (!REV || m >= kC - n)) ? __ldg(gvc + (size_t)(vrb + m) * DV)
                                                                                  : 0.f;
        };
        if (outer && REV) {  // the scan runs from smem row 63: rows 32..63 first give the midpoint
          float x[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = vgate(32 + e);
#pragma unroll
          for (int e = 31; e >= 0; --e) vcar = fmaf(x[e], kLog2e, vcar);
          vbm = vcar;
        }
#pragma unroll 1
        for (int r0 = 0; r0 < kC; r0 += 32) {
          float a[32], gq[outer ? 32 : 1];
          if (outer) {
#pragma unroll
            for (int e = 0; e < 32; ++e) gq[e] = vgate(r0 + e);
          }
          tmem_ld32(tl + kColO + ob * 64 + r0, a);
          if (sgate) {  // O = e^{b_r} (S^T Q^T) + (local part)
            float b[32], f[32];
            tmem_ld32(tl + kColO1 + ob * 64 + r0, b);
            load32(ms + kMsEB + r0, f);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) a[e] = fmaf(f[e], b[e], a[e]);
          }
          tmem_wait_ld();
          if (outer) {  // o = e^{bv - bv_m} (midpoint-relative value-axis products)
            if (REV) {  // rows 0..31 continue from row 32; rows 32..63 start at row 63
              float car = r0 == 0 ? vbm : 0.f;
#pragma unroll
              for (int e = 31; e >= 0; --e) {
                car = fmaf(gq[e], kLog2e, car);
                gq[e] = car;
              }
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                vcar = fmaf(gq[e], kLog2e, vcar);
                gq[e] = vcar;
              }
              if (r0 == 0) vbm = gq[kMid];
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) a[e] *= ex2(gq[e] - vbm);
          }
          if (elu) {
            float den[32];
            load32(ms + kMsDen + r0, den);
#pragma unroll
            for (int e = 0; e < 32; ++e) a[e] = __fdividef(a[e], den[e]);
          }
          // rows (r, r+1) of neighbouring lanes are exchanged so that each
          // thread writes two adjacent bf16 of one row
          if (v < DV) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float send = odd ? a[e] : a[e + 1];
              const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
              const int r = r0 + e + (odd ? 1 : 0);
              const int col = v - (odd ? 1 : 0);
              const uint32_t w = odd ? pack_bf16(recv, a[e + 1]) : pack_bf16(a[e], recv);
              if (staged)
                *reinterpret_cast<uint32_t *>(ot + sw128_off(r, col & 63)) = w;
              else if (REV ? r >= kC - n : r < n)
                *reinterpret_cast<uint32_t *>(obh + (size_t)(t0c + r) * DV + col) = w;
            }
          }
        }
        if (staged) fence_proxy_async();
        tc_fence_before();
        group_sync(kBarSG);
        if (v == 0) {
          if (staged) {
#pragma unroll
            for (int a = 0; a < DV / 64; ++a)
              tma_store_3d(&tm_o, sm + L.ot + a * 8192, 64 * a, t0c, bh);
            bulk_commit();
          }
          mbar_arrive(&o_free[ob]);
          mbar_arrive(&mfree[c % kNM]);
        }
      }
    }
    if (v == 0) bulk_wait<0>();  // output tiles written before the CTA leaves
    if (alive && p.S_final) {
      bool ok = wait_or_abort(s_done, (nchunks - 1) & 1, abort_flag, p.status);
      if (group_all(ok, kBarSG)) {
        tc_fence_after();
        for (int c0 = 0; c0 < DK; c0 += 32) {
          float x[32];
          tmem_ld32(tl + kColS + c0, x);
          tmem_wait_ld();
          if (gla) {  // the last chunk's midpoint-to-end decay
            float fl[32];
            load32(mslot(nchunks - 1) + kMsLM + c0, fl);
            if (outer) {  // of both axes
              const float lv = v < DV ? mslot(nchunks - 1)[kMsLMV + v] : 0.f;
#pragma unroll
              for (int e = 0; e < 32; ++e) fl[e] *= lv;
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] *= fl[e];
          }
          if (v < DV) {
#pragma unroll
            for (int e = 0; e < 32; ++e) p.S_final[((size_t)bh * DK + c0 + e) * Wmem + v] = x[e];
          }
        }
      }
    }
  } else if (tid >= kKG) {
    // -------------------------------------------------------------- key group
    const int kg = tid - kKG;
    if (elu && kg < DK) zs[kg] = p.S0 ? p.S0[((size_t)bh * DK + kg) * Wmem + DV] : 0.f;
    float lm_prev = 1.f;  // GLA: the previous chunk's e^{b_last - b_m} of channel kg
    float lv_prev = 1.f;  // outer-product gate: the same for value column kg
    for (int j = 0; j < nchunks; ++j) {
      const int s = j % ns, n = min(kC, T - j * kC);
      uint8_t *st = stage(s);
      float *ms = mslot(j);
      uint8_t *qk = st + L.qk;
      float *gt = reinterpret_cast<float *>(st + L.g);
      bool ok = wait_or_abort(&full[s], (j / ns) & 1, abort_flag, p.status);
      if (!group_all(ok, kBarKG)) break;
      // ---- inclusive log-gate prefix
      float gvr[outer ? kC : 1];  // outer-product gate: this thread's value-axis gates
      if (gla) {
        if (kg < DK) {  // channel kg: all 64 loads first, then the scan (log2 units) in registers
          float b[kC];
          // (reversed runs: the padding rows above a short last window read the gate of the
          // stored row just below them, row 0's; they must not decay)
#pragma unroll
          for (int r = 0; r < kC; ++r) b[r] = (!REV || r >= kC - n) ? gt[r * DK + kg] : 0.f;
          if (REV) {  // the reversed sequence's order: smem row 63 first
            b[kC - 1] *= kLog2e;
#pragma unroll
            for (int r = kC - 2; r >= 0; --r) b[r] = fmaf(b[r], kLog2e, b[r + 1]);
          } else {
            b[0] *= kLog2e;
#pragma unroll
            for (int r = 1; r < kC; ++r) b[r] = fmaf(b[r], kLog2e, b[r - 1]);
          }
#pragma unroll
          for (int r = 0; r < kC; ++r) gt[r * DK + kg] = b[r];
          const float lm = ex2(b[kLastRow] - b[kMidRow]);
          ms[kMsBM + kg] = ex2(b[kMidRow]) * lm_prev;
          ms[kMsLM + kg] = lm;
          lm_prev = lm;
        }
        if (outer && kg < DV) {  // value column kg: the loads fly during the q/k transform
          const int rb = REV ? T - (j + 1) * kC + 1 : j * kC;  // stored row of smem row 0's gate
          const float *gp = p.beta + (size_t)bh * T * DV + kg;
#pragma unroll
          for (int r = 0; r < kC; ++r)
            gvr[r] = (rb + r >= 0 && rb + r < T && (!REV || r >= kC - n)) ? __ldg(gp + (size_t)(rb + r) * DV) : 0.f;
        }
        group_sync(kBarKG);
        // Q e^{b - b_mid}, K e^{b_mid - b} in place: thread kg owns 8-channel
        // group cg of rows r0 + kStep m (conflict-free tile and gate accesses)
        constexpr int kGroups = DK / 8, kStep = 128 / kGroups, kRows = kC / kStep;
        const int cg = kg % kGroups, r0 = kg / kGroups;
        float bm[8];
        {
          const float4 *mp = reinterpret_cast<const float4 *>(gt + kMidRow * DK + cg * 8);
          const float4 m0 = mp[0], m1 = mp[1];
          bm[0] = m0.x; bm[1] = m0.y; bm[2] = m0.z; bm[3] = m0.w;
          bm[4] = m1.x; bm[5] = m1.y; bm[6] = m1.z; bm[7] = m1.w;
        }
#pragma unroll 2
        for (int m = 0; m < kRows; ++m) {
          const int r = r0 + kStep * m;
          const float4 *gp = reinterpret_cast<const float4 *>(gt + r * DK + cg * 8);
          const float4 g0 = gp[0], g1 = gp[1];
          const float bv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
          uint4 *pq = reinterpret_cast<uint4 *>(qk + (cg >> 3) * 16384 + sw128_off(r, (cg & 7) * 8));
          uint4 *pk = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(pq) + 8192);
          float fq[8], fk[8];
          unpack8(*pq, fq);
          unpack8(*pk, fk);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float d = bv[e] - bm[e];  // log2 units
            fq[e] *= ex2(d);
            fk[e] *= ex2(-d);
          }
          *pq = pack8(fq);
          *pk = pack8(fk);
        }
        fence_proxy_async();
        group_sync(kBarKG);
      }
      // ---- elementwise transforms of the q/k tiles (elu+1)
      if (elu) {
        constexpr int kPer = 2 * kC * DK / 8 / 128;  // 16-byte groups per thread
        const int row = kg;                          // row of [Q; K]
        const int r = row & (kC - 1);
        const bool is_k = row >= kC;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int g8 = i;  // 8-column group within the row
          uint8_t *ptr = qk + (g8 >> 3) * 16384 + sw128_off(row, (g8 & 7) * 8);
          float f[8];
          unpack8(*reinterpret_cast<uint4 *>(ptr), f);
          if (elu) {
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = (r < n) ? (f[e] > 0.f ? f[e] + 1.f : __expf(f[e])) : 0.f;
            const uint4 hi = pack8(f);
            if (is_k) {
              float fh[8];
              unpack8(hi, fh);
#pragma unroll
              for (int e = 0; e < 8; ++e) fh[e] = f[e] - fh[e];
              *reinterpret_cast<uint4 *>(st + L.klo + (g8 >> 3) * 8192 + sw128_off(r, (g8 & 7) * 8)) =
                  pack8(fh);
            }
            *reinterpret_cast<uint4 *>(ptr) = hi;
          }
        }
        fence_proxy_async();
        group_sync(kBarKG);
      }
      if ((elu || gla) && kg == 0) mbar_arrive(&qk_ready[s]);
      // ---- outer-product gate, value axis (while the score MMA runs): prefix of
      // column kg, d = bv - bv_m into the dead gate tile, then V e^{-d} in place
      if (outer) {
        if (kg < DV) {
          if (REV) {
            gvr[kC - 1] *= kLog2e;
#pragma unroll
            for (int r = kC - 2; r >= 0; --r) gvr[r] = fmaf(gvr[r], kLog2e, gvr[r + 1]);
          } else {
            gvr[0] *= kLog2e;
#pragma unroll
            for (int r = 1; r < kC; ++r) gvr[r] = fmaf(gvr[r], kLog2e, gvr[r - 1]);
          }
          const float bm = gvr[kMidRow], lv = ex2(gvr[kLastRow] - bm);
#pragma unroll
          for (int r = 0; r < kC; ++r) gt[r * DV + kg] = gvr[r] - bm;
          ms[kMsBMV + kg] = ex2(bm) * lv_prev;
          ms[kMsLMV + kg] = lv;
          lv_prev = lv;
        }
        group_sync(kBarKG);
        const int cg = kg & 15, r0 = kg >> 4;  // 16-byte group cg of rows r0 + 8 m (as the row scalings)
        if (cg < DV / 8) {
          uint8_t *base = st + L.v + (cg >> 3) * 8192;
#pragma unroll 2
          for (int m = 0; m < 8; ++m) {
            const int r = r0 + 8 * m;
            const float4 *dp = reinterpret_cast<const float4 *>(gt + r * DV + cg * 8);
            const float4 d0 = dp[0], d1 = dp[1];
            const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
            uint4 *ptr = reinterpret_cast<uint4 *>(base + sw128_off(r, (cg & 7) * 8));
            float f[8];
            unpack8(*ptr, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] *= ex2(-dd[e]);
            *ptr = pack8(f);
          }
        }
      }
      ok = wait_or_abort(&d1_full[j & 1], (j >> 1) & 1, abort_flag, p.status);
      if (!group_all(ok, kBarKG)) break;
      tc_fence_after();
      const bool fast = sgate && ms[kMsFast] != 0.f;
      // ---- masked, decayed scores P (TMEM lanes 0..63 hold the Q K^T rows)
      if (kg < kC) {
        const int r = kg;
        const float b2r = sgate ? ms[kMsB2 + r] : 0.f;
        const float fr = fast ? ms[kMsF + r] : 1.f;
        float rowsum = 0.f;
#pragma unroll 1
        for (int s0 = 0; s0 < kC; s0 += 32) {
          float d[32], b2s[32];
          if (sgate) load32(ms + kMsB2 + s0, b2s);
          tmem_ld32(tl + kColD1 + (uint32_t)(j & 1) * 64u + s0, d);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int sc = s0 + e;
            // causal: s <= r and r a real row; reversed (smem rows): s >= r and r in the
            // last n rows of the window
            const bool keep = REV ? (sc >= r && r >= kC - n) : (sc <= r && r < n);
            float x = keep ? d[e] : 0.f;
            // fast path: P' = Q K^T e^{b_r - b_last} against e^{b_last - b_s} V;
            // exact path: P = Q K^T e^{b_r - b_s} against Kt = e^{b_last - b_s} K
            if (sgate) x *= fast ? fr : exp2f(keep ? b2r - b2s[e] : 0.f);
            if (elu) {
              x = __bfloat162float(__float2bfloat16_rn(x));
              rowsum += x;
            }
            d[e] = x;
          }
          store_row32_bf16(st + L.p, 8192, r, s0, d);
        }
        if (elu) ms[kMsDen + r] = rowsum;
      } else if (elu) {
        const int r = kg - kC;  // phi(q_r) . z with the rounded phi(q) the MMA used
        float acc = 0.f;
#pragma unroll
        for (int g8 = 0; g8 < DK / 8; ++g8) {
          float f[8];
          unpack8(*reinterpret_cast<const uint4 *>(qk + (g8 >> 3) * 16384 + sw128_off(r, (g8 & 7) * 8)), f);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc = fmaf(f[e], zs[g8 * 8 + e], acc);
        }
        tmp[r] = acc;
      }
      tc_fence_before();
      group_sync(kBarKG);
      if (kg == 0) mbar_arrive(&d1_free[j & 1]);
      // Row scalings in place. Thread kg owns 16-byte column group cg of rows
      // r0 + 8 m: a quarter warp covers one row's eight groups of one atom, so
      // every access is free of bank conflicts.
      {
        const int cg = kg & 15, r0 = kg >> 4;
        // ---- e^{b_last - b_s} V (fast) or Kt; elu+1: z, den
        if (fast) {
          if (cg < DV / 8) {
            uint8_t *base = st + L.v + (cg >> 3) * 8192;
#pragma unroll 2
            for (int m = 0; m < 8; ++m) {
              const int r = r0 + 8 * m;
              const float rs = ms[kMsVS + r];
              uint4 *ptr = reinterpret_cast<uint4 *>(base + sw128_off(r, (cg & 7) * 8));
              float f[8];
              unpack8(*ptr, f);
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] *= rs;
              *ptr = pack8(f);
            }
          }
        } else if (sgate) {
          if (cg < DK / 8) {
            uint8_t *base = qk + 8192 + (cg >> 3) * 16384;
#pragma unroll 2
            for (int m = 0; m < 8; ++m) {
              const int r = r0 + 8 * m;
              const float rs = ms[kMsVS + r];
              uint4 *ptr = reinterpret_cast<uint4 *>(base + sw128_off(r, (cg & 7) * 8));
              float f[8];
              unpack8(*ptr, f);
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] *= rs;
              *ptr = pack8(f);
            }
          }
        }
      }
      if (elu) {
        if (kg < kC) ms[kMsDen + kg] += tmp[kg];
        if (kg < DK) {
          float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
          const uint8_t *kh = qk + (kg >> 6) * 16384 + 8192;
          const uint8_t *kl = st + L.klo + (kg >> 6) * 8192;
#pragma unroll 4
          for (int r = 0; r < kC; r += 2) {
            a0 += bf16_at(kh, sw128_off(r, kg & 63));
            a1 += bf16_at(kl, sw128_off(r, kg & 63));
            a2 += bf16_at(kh, sw128_off(r + 1, kg & 63));
            a3 += bf16_at(kl, sw128_off(r + 1, kg & 63));
          }
          zs[kg] += (a0 + a2) + (a1 + a3);
        }
      }
      fence_proxy_async();
      group_sync(kBarKG);
      if (kg == 0) {
        mbar_arrive(&key_ready[s]);
        mbar_arrive(&empty[s]);
      }
    }
    if (elu && p.S_final && kg < DK && !*abort_flag)
      p.S_final[((size_t)bh * DK + kg) * Wmem + DV] = zs[kg];
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 3) tmem_dealloc(tbase, kTmemCols);
}

template <int DK, int DV, int KIND, bool REV>
int launch_typed(const ChunkParams &p, cudaStream_t stream) {
  int ns = 3;
  WsLayout L = ws_layout(DK, DV, KIND, ns);
  while (ns > 2 && L.total + 1024 > 232448) L = ws_layout(DK, DV, KIND, --ns);
  const size_t smem = L.total + 1024;
  if (smem > 232448) {
    set_error("la_chunk_fwd: pipelined kernel needs %zu bytes of shared memory", smem);
    return LA_ERR_UNSUPPORTED;
  }
  const int BH = p.B * p.H;
  CUtensorMap mq, mk, mv, mg, mo;
  bool ok = make_map(&mq, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DK, p.T, BH, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&mo, p.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, p.T, BH, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&mk, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DK, p.T, BH, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&mv, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, p.T, BH, 64,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  if (ok && chan_gates(KIND))
    ok = make_map(&mg, p.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, DK, p.T, BH, DK,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
  else
    mg = mq;
  if (!ok) {
    set_error("la_chunk_fwd: cuTensorMapEncodeTiled rejected a tensor map");
    return LA_ERR_CUDA;
  }
  auto kern = chunk_ws_kernel<DK, DV, KIND, REV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) {
    kern<<<BH, kThreads, smem, stream>>>(p, ns, mq, mk, mv, mg, mo);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_error("la_chunk_fwd: pipelined kernel launch failed: %s", cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  return LA_OK;
}

template <int KIND, bool REV = false>
int launch_kind(const ChunkParams &p, cudaStream_t stream) {
  if (p.dk == 128 && p.dv == 128) return launch_typed<128, 128, KIND, REV>(p, stream);
  if (p.dk == 128 && p.dv == 64) return launch_typed<128, 64, KIND, REV>(p, stream);
  if (p.dk == 64 && p.dv == 128) return launch_typed<64, 128, KIND, REV>(p, stream);
  return launch_typed<64, 64, KIND, REV>(p, stream);
}

}  // namespace

int launch_chunk_ws(const ChunkParams &p, cudaStream_t stream) {
  if (!encode_fn()) {
    set_error("la_chunk_fwd: cuTensorMapEncodeTiled is unavailable");
    return LA_ERR_CUDA;
  }
  if (p.rev) {
    if (p.kind == kLinear) return launch_kind<kLinear, true>(p, stream);
    if (p.kind == kRetnet) return launch_kind<kRetnet, true>(p, stream);
    if (p.kind == kScalar) return launch_kind<kScalar, true>(p, stream);
    if (p.kind == kGla) return launch_kind<kGla, true>(p, stream);
    if (p.kind == kOuter) return launch_kind<kOuter, true>(p, stream);
    set_error("la_chunk_fwd: no reversed run for mode %d", p.kind);
    return LA_ERR_UNSUPPORTED;
  }
  switch (p.kind) {
    case kLinear: return launch_kind<kLinear>(p, stream);
    case kElu1: return launch_kind<kElu1>(p, stream);
    case kRetnet: return launch_kind<kRetnet>(p, stream);
    case kScalar: return launch_kind<kScalar>(p, stream);
    case kGla: return launch_kind<kGla>(p, stream);
    case kOuter: return launch_kind<kOuter>(p, stream);
    default:
      set_error("la_chunk_fwd: mode %d is not handled by the pipelined kernel", p.kind);
      return LA_ERR_UNSUPPORTED;
  }
}

}  // namespace la
