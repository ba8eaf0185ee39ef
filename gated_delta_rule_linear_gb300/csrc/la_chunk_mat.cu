// Materialised chunk forward for the unit-write modes (plain linear, elu+1,
// RetNet, scalar decay, GLA), bf16 inputs: the two-phase variant "Talk Linear
// Attention" section 4.1.2 describes (a serial state pass that materialises
// the chunk-boundary states, then a fully parallel output pass).
//
//   state pass  one CTA per (b, h): S^T stays in TMEM; per chunk it writes the
//               incoming state S_{i-1} as a bf16 operand image (one bulk copy
//               of the 128B-swizzled shared-memory tile) and applies
//               S <- Diag(e^{b_last}) S + Kt^T V on the tensor core.
//   output pass one CTA per (b, h, chunk), all chunks in parallel:
//               O = Diag(e^{b}) Q S_{i-1} + P V with P the masked, decayed
//               local scores, S_{i-1} loaded straight into its operand layout.
//
// The workspace (one state image per chunk, plus z per chunk for elu+1) is
// provided by the caller of these launchers.
#include <algorithm>

#include "la_tc_common.cuh"

namespace la {
namespace {

using namespace sm100;
using namespace tc;

constexpr int kMid = kC / 2 - 1;
constexpr float kLog2e = 1.4426950408889634f;

__host__ __device__ inline uint32_t up1k(uint32_t x) { return (x + 1023u) & ~1023u; }
// bytes of one materialised state image: S^T as 128 rows (value axis, zero
// padded when dv = 64) x dk bf16 in 64-column 128B-swizzled atoms
__host__ __device__ constexpr uint32_t blob_bytes(int dk) { return (uint32_t)(dk / 64) * 16384u; }

// ============================================================ state pass
// For the unit-write modes every row of S (one key channel) evolves on its
// own, so a CTA owns one 64-channel key block of one head: it writes exactly
// one 64-column atom of each state image.
//
// The chunk-local update dS_i = V_i^T Kt_i (Kt = K e^{b_last - b}) has no
// dependency between chunks, so the tensor core computes it for chunks ahead
// into a ring of TMEM slots, and the state group keeps S^T in registers and
// runs the scan S_i = Diag(e^{b_last}) S_{i-1} + dS_i ("Talk Linear Attention"
// section 4.1.2: the states of the chunk boundaries, then the outputs).
//
// Roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer, warp 3 TMEM
// owner, warps 4..7 the state group (lane = value row of S^T: writes S_{i-1}
// as an image atom, adds dS_i), warps 8..11 the key group (gate prefix, Kt or
// phi(K) in place, the elu+1 normaliser z).
constexpr int kAThreads = 384;
constexpr int kASG = 128;  // first thread of the state group
constexpr int kAKG = 256;  // first thread of the key group
constexpr int kAKBar = 2;  // key-group named barrier
constexpr int kKB = 64;    // key channels per state-pass CTA
constexpr int kANB = 4;    // TMEM slots of dS (64 columns each)

// Stages in flight, so that loads run several chunks ahead of the scan.
template <int KIND>
__host__ __device__ constexpr int a_stages() {
  return KIND == kGla ? 4 : KIND == kElu1 ? 5 : 6;
}
constexpr int kAMaxStages = 6;

struct ALayout {
  uint32_t k, v, g, klo, stage, st, misc, tmp, bar, total;
};
__host__ __device__ inline ALayout a_layout(int kind, int ns) {
  ALayout L;
  const bool gla = kind == kGla, elu = kind == kElu1;
  uint32_t o = 0;
  L.k = o; o += 8192u;
  L.v = o; o += 16384u;
  L.g = o; o += gla ? (uint32_t)kC * kKB * 4u : 0u;
  L.klo = o; o += elu ? 8192u : 0u;
  L.stage = up1k(o);
  o = (uint32_t)ns * L.stage;
  L.st = o; o += 2u * 16384u;             // two image atoms (one bulk store may still be reading)
  L.misc = o; o += (uint32_t)ns * 1024u;  // per stage: [64..127] e^{b_last} (scalar gates), [128..191] per-channel decay
  L.tmp = o; o += 512u;                   // key-group exchange between row halves
  L.bar = o; o += 512u;
  L.total = o;
  return L;
}

template <int DK, int DV, int KIND>
__global__ void __launch_bounds__(kAThreads, 1)
chunk_state_kernel(const ChunkParams p, uint8_t *__restrict__ ws, float *__restrict__ zws, int istride,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_g) {
  constexpr bool elu = KIND == kElu1, gla = KIND == kGla;
  constexpr bool sgate = KIND == kRetnet || KIND == kScalar;
  constexpr int Wmem = DV + (elu ? 1 : 0);
  constexpr int nkb = DK / kKB;
  constexpr int NS = a_stages<KIND>();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const ALayout L = a_layout(KIND, NS);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x / nkb, kb = blockIdx.x % nkb, h = bh % p.H;
  const int c_base = kb * kKB;
  const int T = p.T, nch = (T + kC - 1) / kC;
  // one image every istride chunks (istride = 2 for the 128-token output pass)
  const int nimg = (nch + istride - 1) / istride;

  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.bar);
  uint64_t *full = bars, *empty = bars + kAMaxStages, *kready = bars + 2 * kAMaxStages;
  uint64_t *dfull = bars + 3 * kAMaxStages, *dfree = dfull + kANB, *drain = dfree + kANB;
  uint64_t *img_full = drain + 1, *img_free = img_full + 2;  // [2] each
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(img_free + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  float *tmp = reinterpret_cast<float *>(sm + L.tmp);
  auto stage = [&](int s) { return sm + (uint32_t)s * L.stage; };

  if (warp == 3) {
    tmem_alloc(tmem_slot, kANB * 64);
    tmem_relinquish();
  }
  if (tid == 0) {
    // a stage is refilled once the tensor core has read it and the state group
    // has read its decay factors, so the key group never laps the state group
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1 + 128);
      mbar_init(&kready[s], 1);
    }
    for (int b = 0; b < kANB; ++b) {
      mbar_init(&dfull[b], 1);
      mbar_init(&dfree[b], 128);
    }
    mbar_init(drain, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&img_full[b], 128);  // every state-group thread has written its row
      mbar_init(&img_free[b], 1);    // the bulk store has read the buffer
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (DV == 64) {  // rows 64..127 of the value operand stay zero in every stage
    for (int i = tid; i < NS * 512; i += kAThreads)
      reinterpret_cast<uint4 *>(stage(i >> 9) + L.v + 8192)[i & 511] = make_uint4(0, 0, 0, 0);
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {  // producer
      constexpr uint32_t bytes = kKB * kC * 2u + DV * kC * 2u + (gla ? kKB * kC * 4u : 0u);
      int issued = 0;
      for (int j = 0; j < nch; ++j) {
        const int s = j % NS;
        if (!wait_or_abort(&empty[s], ((j / NS) & 1) ^ 1, abort_flag, p.status)) break;
        uint8_t *st = stage(s);
        mbar_arrive_expect_tx(&full[s], bytes);
        tma_load_3d(st + L.k, &tm_k, &full[s], c_base, j * kC, bh);
#pragma unroll
        for (int a = 0; a < DV / 64; ++a) tma_load_3d(st + L.v + a * 8192, &tm_v, &full[s], 64 * a, j * kC, bh);
        if (gla) tma_load_3d(st + L.g, &tm_g, &full[s], c_base, j * kC, bh);
        issued = j + 1;
      }
      for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
        (void)mbar_wait_bounded(&full[j % NS], (j / NS) & 1, kSpinLimit);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // chunk-local updates dS_i = V^T Kt into the TMEM ring
      constexpr uint32_t id_su = idesc_bf16_f32(128, kKB, true, true);
      for (int i = 0; i < nch; ++i) {
        const int s = i % NS, b = i % kANB;
        if (!wait_or_abort(&kready[s], (i / NS) & 1, abort_flag, p.status)) break;
        if (!wait_or_abort(&dfree[b], ((i / kANB) & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        uint8_t *st = stage(s);
        const uint32_t a_v = smem_u32(st + L.v), a_k = smem_u32(st + L.k), d = tbase + (uint32_t)b * 64u;
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk) {
          const uint64_t dv_ = desc_sw128(a_v + kk * 2048, 8192, 1024);
          mma_bf16(d, dv_, desc_sw128(a_k + kk * 2048, 8192, 1024), id_su, kk > 0);
          if (elu) mma_bf16(d, dv_, desc_sw128(smem_u32(st + L.klo) + kk * 2048, 8192, 1024), id_su, 1);
        }
        mma_commit(&dfull[b]);
        mma_commit(&empty[s]);
      }
      mma_commit(drain);
      (void)mbar_wait_bounded(drain, 0, kSpinLimit);
    }
  } else if (warp == 2) {
    if (lane == 0) {  // ships each image atom with one bulk copy; one copy in flight
      int done = 0;
      for (int i = 0; i < nimg; ++i) {
        const int ib = i & 1;
        if (!wait_or_abort(&img_full[ib], (i >> 1) & 1, abort_flag, p.status)) break;
        bulk_store(ws + ((size_t)bh * nimg + i) * blob_bytes(DK) + (size_t)kb * 16384u,
                   sm + L.st + (uint32_t)ib * 16384u, 16384u);
        bulk_commit();
        if (i > 0) {
          bulk_wait_read<1>();  // the copy of chunk i - 1 has read its buffer
          mbar_arrive(&img_free[ib ^ 1]);
        }
        done = i + 1;
      }
      bulk_wait<0>();
      if (done > 0) mbar_arrive(&img_free[(done - 1) & 1]);
    }
  } else if (tid >= kAKG) {
    // ------------------------------------------------------------ key group
    const int kt = tid - kAKG;
    const int col = kt & 63, half = kt >> 6;  // GLA prefix / elu+1 z: channel and row half
    const int cg = kt & 7, r0 = kt >> 3;      // transform: 8-channel group, rows r0 + 16 j
    float z = 0.f;                            // elu+1 normaliser of channel c_base + col (half 0)
    if (elu && half == 0 && p.S0) z = p.S0[((size_t)bh * DK + c_base + col) * Wmem + DV];
    // scalar gates: every key warp scans the chunk's 64 gates itself, loaded one chunk ahead
    auto gate = [&](int t) -> float {
      if (t >= T) return 0.f;
      return KIND == kRetnet ? __ldg(p.g + h) : __ldg(p.g + (size_t)bh * T + t);
    };
    float gn0 = 0.f, gn1 = 0.f;
    if (sgate) {
      gn0 = gate(lane);
      gn1 = gate(lane + 32);
    }
    for (int i = 0; i < nch; ++i) {
      const int s = i % NS, n = min(kC, T - i * kC);
      uint8_t *st = stage(s);
      float *ms = reinterpret_cast<float *>(sm + L.misc + (uint32_t)s * 1024u);
      const float gc0 = gn0, gc1 = gn1;
      if (sgate && i + 1 < nch) {
        gn0 = gate((i + 1) * kC + lane);
        gn1 = gate((i + 1) * kC + lane + 32);
      }
      if (!group_wait(&full[s], (i / NS) & 1, kt, kAKBar, abort_flag, p.status)) break;
      if (elu && half == 0 && zws && i % istride == 0)  // z before chunk i, at image boundaries
        zws[((size_t)bh * nimg + i / istride) * DK + c_base + col] = z;
      float rs[4] = {1.f, 1.f, 1.f, 1.f};  // e^{b_last - b_r} of rows r0 + 16 j
      if (sgate) {
        float v0 = gc0 * kLog2e, v1 = gc1 * kLog2e;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float a0 = __shfl_up_sync(0xffffffffu, v0, off);
          const float a1 = __shfl_up_sync(0xffffffffu, v1, off);
          if (lane >= off) {
            v0 += a0;
            v1 += a1;
          }
        }
        v1 += __shfl_sync(0xffffffffu, v0, 31);
        const float bl = __shfl_sync(0xffffffffu, v1, 31);
        rs[0] = exp2f(bl - __shfl_sync(0xffffffffu, v0, r0));
        rs[1] = exp2f(bl - __shfl_sync(0xffffffffu, v0, r0 + 16));
        rs[2] = exp2f(bl - __shfl_sync(0xffffffffu, v1, r0));
        rs[3] = exp2f(bl - __shfl_sync(0xffffffffu, v1, r0 + 16));
        if (kt < 32) {
          ms[64 + lane] = exp2f(bl);
          ms[96 + lane] = exp2f(bl);
        }
      }
      if (gla) {  // channel col, rows 32*half .. +31: prefix, then e^{b_last - b_r}
        float *gt = reinterpret_cast<float *>(st + L.g);
        float b[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) b[e] = gt[(32 * half + e) * kKB + col];
#pragma unroll
        for (int e = 1; e < 32; ++e) b[e] += b[e - 1];
        if (half == 0) tmp[col] = b[31];
        group_sync(kAKBar);
        float bl;
        if (half == 1) {
          const float off = tmp[col];
#pragma unroll
          for (int e = 0; e < 32; ++e) b[e] += off;
          bl = b[31];
          tmp[64 + col] = bl;
          ms[128 + col] = __expf(bl);
        }
        group_sync(kAKBar);
        if (half == 0) bl = tmp[64 + col];
#pragma unroll
        for (int e = 0; e < 32; ++e) gt[(32 * half + e) * kKB + col] = __expf(bl - b[e]);
        group_sync(kAKBar);
      }
      if (KIND != kLinear) {
        // Kt (or phi(K) with its low half) in place; a quarter warp covers one row's 8 groups
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = r0 + 16 * j;
          const uint32_t off = sw128_off(r, cg * 8);
          float f[8];
          unpack8(*reinterpret_cast<const uint4 *>(st + L.k + off), f);
          if (elu) {
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = (r < n) ? (f[e] > 0.f ? f[e] + 1.f : __expf(f[e])) : 0.f;
            const uint4 hi = pack8(f);
            float fh[8];
            unpack8(hi, fh);
#pragma unroll
            for (int e = 0; e < 8; ++e) fh[e] = f[e] - fh[e];
            *reinterpret_cast<uint4 *>(st + L.klo + off) = pack8(fh);
            *reinterpret_cast<uint4 *>(st + L.k + off) = hi;
          } else {
            if (gla) {
              const float4 *gp = reinterpret_cast<const float4 *>(st + L.g + (r * kKB + cg * 8) * 4);
              const float4 ga = gp[0], gb = gp[1];
              f[0] *= ga.x; f[1] *= ga.y; f[2] *= ga.z; f[3] *= ga.w;
              f[4] *= gb.x; f[5] *= gb.y; f[6] *= gb.z; f[7] *= gb.w;
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] *= rs[j];
            }
            *reinterpret_cast<uint4 *>(st + L.k + off) = pack8(f);
          }
        }
        fence_proxy_async();
        group_sync(kAKBar);
      }
      if (elu) {  // z <- z + sum_s phi(k_s), from the hi and lo halves; rows split between halves
        float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const uint32_t off = sw128_off(32 * half + e, col);
          a[e & 3] += bf16_at(st + L.k, off) + bf16_at(st + L.klo, off);
        }
        const float part = (a[0] + a[1]) + (a[2] + a[3]);
        if (half == 1) tmp[col] = part;
        group_sync(kAKBar);
        if (half == 0) z += part + tmp[col];
      }
      if (kt == 0) mbar_arrive(&kready[s]);
    }
    if (elu && half == 0 && p.S_final)
      p.S_final[((size_t)bh * DK + c_base + col) * Wmem + DV] = z;
  } else if (tid >= kASG) {
    // ------------------------------------------------------------ state group
    const int v = tid - kASG;  // value row of S^T (TMEM lane of dS)
    const uint32_t tl = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    float S[kKB];              // S^T[v][c_base .. c_base + 63]
#pragma unroll
    for (int c = 0; c < kKB; ++c)
      S[c] = (p.S0 && v < DV) ? p.S0[((size_t)bh * DK + c_base + c) * Wmem + v] : 0.f;
    // Waits here are per thread (no group barrier in the loop), so a thread
    // that gives up cannot leave the others blocked on a named barrier.
    bool alive = true;
    for (int i = 0; i < nch; ++i) {
      const int s = i % NS, b = i % kANB;
      const float *ms = reinterpret_cast<const float *>(sm + L.misc + (uint32_t)s * 1024u);
      if (i % istride == 0) {  // S_{i-1} as a bf16 image atom (warp 2 ships it)
        const int j = i / istride, ib = j & 1;
        if (!wait_or_abort(&img_free[ib], ((j >> 1) & 1) ^ 1, abort_flag, p.status)) {
          alive = false;
          break;
        }
        uint8_t *img = sm + L.st + (uint32_t)ib * 16384u;
        store_row32_bf16(img, 16384, v, 0, S);
        store_row32_bf16(img, 16384, v, 32, S + 32);
        fence_proxy_async();
        mbar_arrive(&img_full[ib]);
      }
      // decay factors of chunk i (key group) and its local update (tensor core)
      if (!wait_or_abort(&kready[s], (i / NS) & 1, abort_flag, p.status) ||
          !wait_or_abort(&dfull[b], (i / kANB) & 1, abort_flag, p.status)) {
        alive = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < kKB; c0 += 32) {
        float d[32];
        tmem_ld32(tl + (uint32_t)b * 64u + c0, d);
        tmem_wait_ld();
        if (c0 + 32 == kKB) {
          tc_fence_before();
          mbar_arrive(&dfree[b]);
        }
        if (sgate || gla) {
          float dc[32];
          load32(ms + (gla ? 128 + c0 : 64), dc);
#pragma unroll
          for (int e = 0; e < 32; ++e) S[c0 + e] = fmaf(dc[e], S[c0 + e], d[e]);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) S[c0 + e] += d[e];
        }
      }
      mbar_arrive(&empty[s]);
    }
    if (alive && p.S_final && v < DV) {
#pragma unroll
      for (int c = 0; c < kKB; ++c) p.S_final[((size_t)bh * DK + c_base + c) * Wmem + v] = S[c];
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 3) tmem_dealloc(tbase, kANB * 64);
}

// ============================================================ output pass
constexpr int kBThreads = 128;

struct BLayout {
  uint32_t qk, v, g, s, p, ot, misc, bar, total;
};
__host__ __device__ inline BLayout b_layout(int dk, int kind) {
  BLayout L;
  const bool gla = kind == kGla;
  uint32_t o = 0;
  L.qk = o; o += (uint32_t)(dk / 64) * 16384u;
  L.v = o; o += 16384u;
  L.g = o; o += gla ? up1k((uint32_t)kC * dk * 4u) : 0u;
  L.s = o; o += blob_bytes(dk);
  L.p = o; o += 8192u;
  L.ot = o; o += 16384u;
  L.misc = o; o += 2048u;
  L.bar = o; o += 64u;
  L.total = o;
  return L;
}

template <int DK, int DV, int KIND>
__global__ void __launch_bounds__(kBThreads)
chunk_output_kernel(const ChunkParams p, const uint8_t *__restrict__ ws, const float *__restrict__ zws,
                    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                    const __grid_constant__ CUtensorMap tm_o) {
  constexpr bool elu = KIND == kElu1, gla = KIND == kGla;
  constexpr bool sgate = KIND == kRetnet || KIND == kScalar;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const BLayout L = b_layout(DK, KIND);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.T, nch = (T + kC - 1) / kC;
  const int bh = blockIdx.x / nch, i = blockIdx.x % nch, h = bh % p.H;
  const int t0 = i * kC, n = min(kC, T - t0);
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L.bar);
  uint64_t *mbar = bar + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 2);
  float *ms = reinterpret_cast<float *>(sm + L.misc);
  // ms: b2[64] | eb[64] | den[64] | qz[64] | bm[128] (e^{b_m}) ... GLA per channel
  float *b2 = ms, *eb = ms + 64, *den = ms + 128, *qz = ms + 192, *ebm = ms + 256;
  uint8_t *qk = sm + L.qk;
  float *gt = reinterpret_cast<float *>(sm + L.g);

  if (warp == 0) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(mbar, 1);
    fence_mbar_init();
    constexpr uint32_t bytes = 2u * DK * kC * 2u + DV * kC * 2u + (gla ? DK * kC * 4u : 0u) + blob_bytes(DK);
    mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
    for (int a = 0; a < DK / 64; ++a) {
      tma_load_3d(qk + a * 16384, &tm_q, bar, 64 * a, t0, bh);
      tma_load_3d(qk + a * 16384 + 8192, &tm_k, bar, 64 * a, t0, bh);
    }
#pragma unroll
    for (int a = 0; a < DV / 64; ++a) tma_load_3d(sm + L.v + a * 8192, &tm_v, bar, 64 * a, t0, bh);
    if (gla) tma_load_3d(sm + L.g, &tm_g, bar, 0, t0, bh);
    bulk_load(sm + L.s, ws + ((size_t)bh * nch + i) * blob_bytes(DK), blob_bytes(DK), bar);
  }
  if (DV == 64) {
    for (int q = tid; q < 512; q += kBThreads)
      reinterpret_cast<uint4 *>(sm + L.v + 8192)[q] = make_uint4(0, 0, 0, 0);
  }
  // scalar gates of this chunk (warp 0), while the tiles stream in
  if (sgate && warp == 0) {
    const int t = t0 + lane;
    float g0, g1;
    if (KIND == kRetnet) {
      const float g = __ldg(p.g + h);
      g0 = (t < T) ? g : 0.f;
      g1 = (t + 32 < T) ? g : 0.f;
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
    b2[lane] = v0;
    b2[lane + 32] = v1;
    eb[lane] = exp2f(v0);
    eb[lane + 32] = exp2f(v1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t tl = tbase + (static_cast<uint32_t>(warp * 32) << 16);
  // D1 is read out before the output MMAs are issued, so O1 reuses its columns
  constexpr uint32_t kD1 = 0, kO1 = 0, kO2 = 64;
  bool ok = mbar_wait_bounded(bar, 0, kSpinLimit);
  if (!__syncthreads_and(ok)) {
    if (tid == 0) atomicOr(p.status, kStatusTimeout);
  } else {
    // ---- GLA prefix per key channel; q/k transforms
    if (gla && tid < DK) {
      float acc = 0.f, bmid = 0.f;
      for (int r = 0; r < kC; ++r) {
        acc += gt[r * DK + tid];
        gt[r * DK + tid] = acc;
        if (r == kMid) bmid = acc;
      }
      ebm[tid] = __expf(bmid);
    }
    __syncthreads();
    if (elu || gla) {
      const int row = tid;  // row of [Q; K]
      const int r = row & (kC - 1);
      const bool is_k = row >= kC;
#pragma unroll 4
      for (int g8 = 0; g8 < DK / 8; ++g8) {
        uint8_t *ptr = qk + (g8 >> 3) * 16384 + sw128_off(row, (g8 & 7) * 8);
        float f[8];
        unpack8(*reinterpret_cast<uint4 *>(ptr), f);
        if (elu) {
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = (r < n) ? (f[e] > 0.f ? f[e] + 1.f : __expf(f[e])) : 0.f;
        } else {
          const float *brow = gt + r * DK + g8 * 8;
          const float *bmid = gt + kMid * DK + g8 * 8;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float d = (brow[e] - bmid[e]) * kLog2e;
            f[e] *= exp2f(is_k ? -d : d);
          }
        }
        *reinterpret_cast<uint4 *>(ptr) = pack8(f);
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t a_qk = smem_u32(qk);
      constexpr uint32_t idesc = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
      for (int kk = 0; kk < DK / 16; ++kk) {
        const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_bf16(tbase + kD1, desc_sw128(a_qk + ko, 16, 1024), desc_sw128(a_qk + ko + 8192, 16, 1024), idesc,
                 kk > 0);
      }
      mma_commit(mbar);
    }
    ok = mbar_wait_bounded(mbar, 0, kSpinLimit);
    if (!__syncthreads_and(ok)) {
      if (tid == 0) atomicOr(p.status, kStatusTimeout);
    } else {
      tc_fence_after();
      // ---- masked, decayed scores P (TMEM lanes 0..63); elu+1: q.z
      if (tid < kC) {
        const int r = tid;
        const float b2r = sgate ? b2[r] : 0.f;
        float rowsum = 0.f;
#pragma unroll 1
        for (int s0 = 0; s0 < kC; s0 += 32) {
          float d[32], fs[32];
          if (sgate) load32(b2 + s0, fs);
          tmem_ld32(tl + kD1 + s0, d);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int sc = s0 + e;
            float x = (sc <= r && r < n) ? d[e] : 0.f;
            if (sgate) x *= exp2f(sc <= r ? b2r - fs[e] : 0.f);
            if (elu) {
              x = __bfloat162float(__float2bfloat16_rn(x));
              rowsum += x;
            }
            d[e] = x;
          }
          store_row32_bf16(sm + L.p, 8192, r, s0, d);
        }
        if (elu) den[r] = rowsum;
      } else if (elu) {
        const int r = tid - kC;
        const float *zp = zws + ((size_t)bh * nch + i) * DK;
        float acc = 0.f;
        for (int g8 = 0; g8 < DK / 8; ++g8) {
          float f[8];
          unpack8(*reinterpret_cast<const uint4 *>(qk + (g8 >> 3) * 16384 + sw128_off(r, (g8 & 7) * 8)), f);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc = fmaf(f[e], __ldg(zp + g8 * 8 + e), acc);
        }
        qz[r] = acc;
      }
      tc_fence_before();
      __syncthreads();
      // ---- Qt for the inter-chunk term: GLA Q e^{b - b_m} -> Q e^{b}
      if (gla && tid < kC) {
        const int r = tid;
#pragma unroll 4
        for (int g8 = 0; g8 < DK / 8; ++g8) {
          uint8_t *ptr = qk + (g8 >> 3) * 16384 + sw128_off(r, (g8 & 7) * 8);
          float f[8];
          unpack8(*reinterpret_cast<uint4 *>(ptr), f);
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] *= ebm[g8 * 8 + e];
          *reinterpret_cast<uint4 *>(ptr) = pack8(f);
        }
      }
      if (elu && tid < kC) den[tid] += qz[tid];
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        const uint32_t a_s = smem_u32(sm + L.s), a_qk = smem_u32(qk), a_v = smem_u32(sm + L.v),
                       a_p = smem_u32(sm + L.p);
        constexpr uint32_t id_o1 = idesc_bf16_f32(128, 64, false, false);
        constexpr uint32_t id_o2 = idesc_bf16_f32(128, 64, true, false);
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16(tbase + kO1, desc_sw128(a_s + ko, 16, 1024), desc_sw128(a_qk + ko, 16, 1024), id_o1, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tbase + kO2, desc_sw128(a_v + kk * 2048, 8192, 1024), desc_sw128(a_p + kk * 32, 16, 1024),
                   id_o2, kk > 0);
        mma_commit(mbar);
      }
      ok = mbar_wait_bounded(mbar, 1, kSpinLimit);
      if (!__syncthreads_and(ok)) {
        if (tid == 0) atomicOr(p.status, kStatusTimeout);
      } else {
        tc_fence_after();
        const int v = tid;
        uint8_t *ot = sm + L.ot + (uint32_t)(v >> 6) * 8192u;
        const bool odd = lane & 1;
#pragma unroll 1
        for (int r0 = 0; r0 < kC; r0 += 32) {
          float a[32], b[32], f[32];
          tmem_ld32(tl + kO1 + r0, a);
          tmem_ld32(tl + kO2 + r0, b);
          if (sgate) load32(eb + r0, f);
          if (elu) load32(den + r0, f);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            float y = sgate ? fmaf(f[e], a[e], b[e]) : a[e] + b[e];
            if (elu) y = __fdividef(y, f[e]);
            a[e] = y;
          }
          if (v < DV) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float send = odd ? a[e] : a[e + 1];
              const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
              const int r = r0 + e + (odd ? 1 : 0);
              const uint32_t w = odd ? pack_bf16(recv, a[e + 1]) : pack_bf16(a[e], recv);
              *reinterpret_cast<uint32_t *>(ot + sw128_off(r, (v & 63) - (odd ? 1 : 0))) = w;
            }
          }
        }
        fence_proxy_async();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
          for (int a = 0; a < DV / 64; ++a) tma_store_3d(&tm_o, sm + L.ot + a * 8192, 64 * a, t0, bh);
          bulk_commit();
          bulk_wait_read<0>();  // the tile is read; the global writes complete with the grid
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, 128);
}

// ============================================= output pass, C = 128
// Chunk length 128 ("Talk Linear Attention" section 3.3: the chunk size trades
// the quadratic intra-chunk work against the number of materialised states)
// for the modes without per-channel gates. The state pass writes one image per
// 128 tokens, half the bytes of C = 64, and each output CTA computes one
// 128-token chunk for one 64-column half of the value axis, token-major:
//   D1 = Q K^T (M = N = 128), P = the masked, decayed scores (bf16, packed in
//   TMEM as the A operand), O1 = Q S_{i-1} (S^T image half as a K-major B),
//   O2 = P V (V half as an MN-major B), o = Diag(e^b) O1 + O2.
// The two value halves of a chunk are neighbouring CTAs: both compute D1 and P
// (the tensor core has room to spare) and share q and k through L2. 256
// threads, ~100 KB of shared memory and 256 TMEM columns let two CTAs share an
// SM, so one CTA's loads overlap the other's MMAs and epilogue.
constexpr int kC2 = 128;
constexpr int kB2Threads = 256;

struct B2Layout {
  uint32_t q, k, v, s, misc, bar, total;
};
__host__ __device__ inline B2Layout b2_layout(int dk) {
  B2Layout L;
  uint32_t o = 0;
  L.q = o; o += (uint32_t)(dk / 64) * 16384u;  // also the output staging tile once O1 is done
  L.k = o; o += (uint32_t)(dk / 64) * 16384u;
  L.v = o; o += 16384u;                       // 128 tokens x one 64-column half of V
  L.s = o; o += (uint32_t)(dk / 64) * 8192u;  // 64 value rows of the S^T image
  L.misc = o; o += 4096u;
  L.bar = o; o += 64u;
  L.total = o;
  return L;
}

// 3-D map over a [BH][T][d] bf16 tensor with 128-row boxes {64, 128, 1}, 128B swizzle
inline bool make_map128(CUtensorMap *m, const void *base, int d, int T, int BH) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * T};
  cuuint32_t box[3] = {64u, (cuuint32_t)kC2, 1u};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DK, int DV, int KIND>
__global__ void __launch_bounds__(kB2Threads, 2)
chunk_output128_kernel(const ChunkParams p, const uint8_t *__restrict__ ws, const float *__restrict__ zws,
                       const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o) {
  constexpr bool elu = KIND == kElu1;
  constexpr bool sgate = KIND == kRetnet || KIND == kScalar;
  constexpr int NVH = DV / 64;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const B2Layout L = b2_layout(DK);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.T, nimg = (T + kC2 - 1) / kC2;
  const int vh = blockIdx.x % NVH, ci = blockIdx.x / NVH;
  const int bh = ci / nimg, j = ci % nimg, h = bh % p.H;
  const int t0 = j * kC2, n = min(kC2, T - t0);
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L.bar);  // q and k landed
  uint64_t *mbar = bar + 1;                                   // MMA commits
  uint64_t *bar_vs = bar + 2;                                 // v and the state image landed
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 3);
  float *ms = reinterpret_cast<float *>(sm + L.misc);
  // b2[128] log2 prefix | eb[128] e^{b} | den[128] | part[2][128] row sums / q.z halves
  float *b2 = ms, *eb = ms + 128, *den = ms + 256, *part = ms + 384, *qzp = ms + 640;
  uint8_t *sq = sm + L.q, *sk = sm + L.k;

  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(mbar, 1);
    mbar_init(bar_vs, 1);
    fence_mbar_init();
    // q and k first (the score MMAs wait for them), then v and the state image
    mbar_arrive_expect_tx(bar, 2u * DK * kC2 * 2u);
#pragma unroll
    for (int a = 0; a < DK / 64; ++a) {
      tma_load_3d(sq + a * 16384, &tm_q, bar, 64 * a, t0, bh);
      tma_load_3d(sk + a * 16384, &tm_k, bar, 64 * a, t0, bh);
    }
    mbar_arrive_expect_tx(bar_vs, 64u * kC2 * 2u + (uint32_t)(DK / 64) * 8192u);
    tma_load_3d(sm + L.v, &tm_v, bar_vs, 64 * vh, t0, bh);
    const uint8_t *img = ws + ((size_t)bh * nimg + j) * blob_bytes(DK) + (size_t)vh * 8192u;
#pragma unroll
    for (int a = 0; a < DK / 64; ++a) bulk_load(sm + L.s + a * 8192, img + (size_t)a * 16384u, 8192u, bar_vs);
  }
  // scalar gates of this chunk (warp 1): 4 tokens per lane, then a warp scan
  if (sgate && warp == 1) {
    float gv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int t = t0 + 4 * lane + e;
      gv[e] = (t < T) ? (KIND == kRetnet ? __ldg(p.g + h) : __ldg(p.g + (size_t)bh * T + t)) * kLog2e : 0.f;
    }
    gv[1] += gv[0];
    gv[2] += gv[1];
    gv[3] += gv[2];
    float run = gv[3];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float a = __shfl_up_sync(0xffffffffu, run, off);
      if (lane >= off) run += a;
    }
    const float base = run - gv[3];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      b2[4 * lane + e] = base + gv[e];
      eb[4 * lane + e] = exp2f(base + gv[e]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const int row = 32 * (warp & 3) + lane, hc = warp >> 2;  // TMEM lane (token) and column half
  const uint32_t tl = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  // TMEM columns: D1 [0, 128); O1 [0, 64) and O2 [64, 128) once P is out of D1; P [128, 192)
  constexpr uint32_t kD1 = 0, kO1 = 0, kO2 = 64, kP = 128;
  bool ok = mbar_wait_bounded(bar, 0, kSpinLimit);
  if (!__syncthreads_and(ok)) {
    if (tid == 0) atomicOr(p.status, kStatusTimeout);
  } else {
    if (elu) {  // phi on the rows of [Q; K]; rows past the sequence end are zero
      const int r = tid & (kC2 - 1);
      uint8_t *base = tid < kC2 ? sq : sk;
#pragma unroll 4
      for (int g8 = 0; g8 < DK / 8; ++g8) {
        uint8_t *ptr = base + (g8 >> 3) * 16384 + sw128_off(r, (g8 & 7) * 8);
        float f[8];
        unpack8(*reinterpret_cast<uint4 *>(ptr), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = (r < n) ? (f[e] > 0.f ? f[e] + 1.f : __expf(f[e])) : 0.f;
        *reinterpret_cast<uint4 *>(ptr) = pack8(f);
      }
      fence_proxy_async();
      __syncthreads();
    }
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, false);
      const uint64_t dq = desc_sw128(smem_u32(sq), 16, 1024), dk_ = desc_sw128(smem_u32(sk), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < DK / 16; ++kk) {
        const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_bf16(tbase + kD1, desc_add(dq, ko), desc_add(dk_, ko), idesc, kk > 0);
      }
      mma_commit(mbar);
    }
    if (elu) {  // q.z for the normaliser, half of the key channels per thread, while D1 runs
      const float *zp = zws + ((size_t)bh * nimg + j) * DK + hc * (DK / 2);
      float acc = 0.f;
#pragma unroll 4
      for (int g8 = 0; g8 < DK / 16; ++g8) {
        const int c = hc * (DK / 2) + g8 * 8;
        float f[8];
        unpack8(*reinterpret_cast<const uint4 *>(sq + (c >> 6) * 16384 + sw128_off(row, c & 63)), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(f[e], __ldg(zp + g8 * 8 + e), acc);
      }
      qzp[hc * 128 + row] = acc;
    }
    ok = mbar_wait_bounded(mbar, 0, kSpinLimit);
    if (!__syncthreads_and(ok)) {
      if (tid == 0) atomicOr(p.status, kStatusTimeout);
    } else {
      tc_fence_after();
      // ---- P = masked, decayed scores of row `row`, columns [64 hc, 64 hc + 64), bf16 into TMEM
      const float b2r = sgate ? b2[row] : 0.f;
      float rowsum = 0.f;
#pragma unroll 1
      for (int s0 = 64 * hc; s0 < 64 * hc + 64; s0 += 32) {
        float d[32], fs[32];
        if (sgate) load32(b2 + s0, fs);
        tmem_ld32(tl + kD1 + s0, d);
        tmem_wait_ld();
        float pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float x0 = (s0 + e <= row && row < n) ? d[e] : 0.f;
          float x1 = (s0 + e + 1 <= row && row < n) ? d[e + 1] : 0.f;
          if (sgate) {
            x0 *= exp2f(s0 + e <= row ? b2r - fs[e] : 0.f);
            x1 *= exp2f(s0 + e + 1 <= row ? b2r - fs[e + 1] : 0.f);
          }
          const uint32_t w = pack_bf16(x0, x1);
          if (elu) rowsum += __uint_as_float(w << 16) + __uint_as_float(w & 0xffff0000u);
          pk[e >> 1] = __uint_as_float(w);
        }
        tmem_st16(tl + kP + (uint32_t)(s0 >> 1), pk);
      }
      if (elu) part[hc * 128 + row] = rowsum;
      tmem_wait_st();
      tc_fence_before();
      __syncthreads();
      // v and the state image (loaded while the scores ran); only the issuing thread waits,
      // so the MMAs are issued exactly when every thread goes on to wait for them
      ok = tid == 0 ? mbar_wait_bounded(bar_vs, 0, kSpinLimit) : true;
      if (tid == 0 && ok) {
        tc_fence_after();
        constexpr uint32_t id_o1 = idesc_bf16_f32(128, 64, false, false);
        constexpr uint32_t id_o2 = idesc_bf16_f32(128, 64, false, true);
        const uint64_t dq = desc_sw128(smem_u32(sq), 16, 1024), ds = desc_sw128(smem_u32(sm + L.s), 16, 1024);
        const uint64_t dv = desc_sw128(smem_u32(sm + L.v), 16384, 1024);
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk)
          mma_bf16(tbase + kO1, desc_add(dq, (kk >> 2) * 16384 + (kk & 3) * 32),
                   desc_add(ds, (kk >> 2) * 8192 + (kk & 3) * 32), id_o1, kk > 0);
#pragma unroll
        for (int kk = 0; kk < kC2 / 16; ++kk)
          mma_bf16_ts(tbase + kO2, tbase + kP + kk * 8, desc_add(dv, kk * 2048), id_o2, kk > 0);
        mma_commit(mbar);
      }
      if (elu && tid < kC2) den[tid] = (part[tid] + part[128 + tid]) + (qzp[tid] + qzp[128 + tid]);
      bool go = __syncthreads_and(ok);  // false: thread 0 gave up on bar_vs and issued nothing
      if (go) go = __syncthreads_and(mbar_wait_bounded(mbar, 1, kSpinLimit));
      if (!go) {
        if (tid == 0) atomicOr(p.status, kStatusTimeout);
      } else {
        tc_fence_after();
        // ---- o rows: value columns [32 hc, 32 hc + 32) of this half, staged token-major in the q tile
        float a[32], b[32];
        tmem_ld32(tl + kO1 + 32 * hc, a);
        tmem_ld32(tl + kO2 + 32 * hc, b);
        tmem_wait_ld();
        const float sc = sgate ? eb[row] : 1.f;
        const float dn = elu ? den[row] : 1.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float y = sgate ? fmaf(sc, a[e], b[e]) : a[e] + b[e];
          if (elu) y = __fdividef(y, dn);
          a[e] = y;
        }
        store_row32_bf16(sq, 16384, row, 32 * hc, a);
        fence_proxy_async();
        __syncthreads();
        if (tid == 0) {
          tma_store_3d(&tm_o, sq, 64 * vh, t0, bh);
          bulk_commit();
          bulk_wait_read<0>();  // the tile is read; the global writes complete with the grid
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, 256);
}

// ---------------------------------------------------------------- launch

// the parallel state pass of the modes without decay (defined with the non-causal kernels it reuses)
template <int DK, int DV, int KIND>
cudaError_t launch_scan_state(const ChunkParams &p, uint8_t *ws, float *zws, const CUtensorMap &mk,
                              const CUtensorMap &mv, cudaStream_t stream);

template <int DK, int DV, int KIND>
int launch_typed(const ChunkParams &p, uint8_t *ws, float *zws, bool scan, cudaStream_t stream) {
  const int BH = p.B * p.H, nch = (p.T + kC - 1) / kC;
  const ALayout La = a_layout(KIND, a_stages<KIND>());
  const BLayout Lb = b_layout(DK, KIND);
  const size_t sa = La.total + 1024, sb = Lb.total + 1024;
  if (sa > 232448 || sb > 232448) {
    set_error("la_chunk_fwd: materialised kernels need %zu / %zu bytes of shared memory", sa, sb);
    return LA_ERR_UNSUPPORTED;
  }
  CUtensorMap mq, mk, mv, mg, mgA, mo;
  bool ok = make_map(&mq, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DK, p.T, BH, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&mk, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DK, p.T, BH, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&mv, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, p.T, BH, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&mo, p.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, p.T, BH, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  if (ok && KIND == kGla) {
    ok = make_map(&mg, p.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, DK, p.T, BH, DK, CU_TENSOR_MAP_SWIZZLE_NONE) &&
         make_map(&mgA, p.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, DK, p.T, BH, kKB, CU_TENSOR_MAP_SWIZZLE_NONE);
  } else {
    mg = mq;
    mgA = mq;
  }
  if (!ok) {
    set_error("la_chunk_fwd: cuTensorMapEncodeTiled rejected a tensor map");
    return LA_ERR_CUDA;
  }
  auto ka = chunk_state_kernel<DK, DV, KIND>;
  cudaError_t e = cudaSuccess;
  const int istride = p.C == kC2 ? 2 : 1;
  if (scan && (KIND == kLinear || KIND == kElu1)) {
    e = launch_scan_state<DK, DV, KIND>(p, ws, zws, mk, mv, stream);
  } else {
    e = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sa);
    if (e == cudaSuccess) {
      ka<<<(unsigned)(BH * (DK / kKB)), kAThreads, sa, stream>>>(p, ws, zws, istride, mk, mv, mgA);
      e = cudaGetLastError();
    }
  }
  if constexpr (KIND != kGla) {
    if (e == cudaSuccess && p.C == kC2) {
      // the 128-token output pass: 128-row boxes, one CTA per (head, chunk, value half)
      CUtensorMap mq2, mk2, mv2, mo2;
      if (!(make_map128(&mq2, p.q, DK, p.T, BH) && make_map128(&mk2, p.k, DK, p.T, BH) &&
            make_map128(&mv2, p.v, DV, p.T, BH) && make_map128(&mo2, p.o, DV, p.T, BH))) {
        set_error("la_chunk_fwd: cuTensorMapEncodeTiled rejected a tensor map");
        return LA_ERR_CUDA;
      }
      auto kc = chunk_output128_kernel<DK, DV, KIND>;
      const size_t sc = b2_layout(DK).total + 1024;
      const size_t nimg = (size_t)(p.T + kC2 - 1) / kC2;
      e = cudaFuncSetAttribute(kc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sc);
      if (e == cudaSuccess) {
        kc<<<(unsigned)((size_t)BH * nimg * (DV / 64)), kB2Threads, sc, stream>>>(p, ws, zws, mq2, mk2, mv2, mo2);
        e = cudaGetLastError();
      }
      if (e != cudaSuccess) {
        set_error("la_chunk_fwd: materialised kernels failed to launch: %s", cudaGetErrorString(e));
        return LA_ERR_CUDA;
      }
      return LA_OK;
    }
  }
  auto kb = chunk_output_kernel<DK, DV, KIND>;
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kb, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sb);
  if (e == cudaSuccess) {
    kb<<<(unsigned)((size_t)BH * nch), kBThreads, sb, stream>>>(p, ws, zws, mq, mk, mv, mg, mo);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_error("la_chunk_fwd: materialised kernels failed to launch: %s", cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  return LA_OK;
}

template <int KIND>
int launch_kind(const ChunkParams &p, uint8_t *ws, float *zws, bool scan, cudaStream_t stream) {
  if (p.dk == 128 && p.dv == 128) return launch_typed<128, 128, KIND>(p, ws, zws, scan, stream);
  if (p.dk == 128 && p.dv == 64) return launch_typed<128, 64, KIND>(p, ws, zws, scan, stream);
  if (p.dk == 64 && p.dv == 128) return launch_typed<64, 128, KIND>(p, ws, zws, scan, stream);
  return launch_typed<64, 64, KIND>(p, ws, zws, scan, stream);
}

// ================================================= non-causal forward
// o_t = S_total^T q_t with S_total = S0 + sum_s k_s v_s^T over the whole
// sequence (elu+1: phi on q and k, divided by phi(q).z_total): the
// right-to-left product Q (K^T V) of the kernel-attention notes, section 3.
// Three launches: a split-T reduction of V^T K on the tensor cores (one CTA
// per head and T-range), a parallel finalize (S0 + partial sums -> S_final
// and a bf16 high/low image of the state), and an output pass whose persistent
// CTAs stream their run of query chunks through the image of each head.
constexpr int kNThreads = 128;

struct NLayout {
  uint32_t k, klo, v, stage, bar, total;
};
__host__ __device__ inline NLayout n_layout(int dk, bool elu) {
  NLayout L;
  uint32_t o = 0;
  L.k = o; o += (uint32_t)(dk / 64) * 8192u;
  L.klo = o; o += elu ? (uint32_t)(dk / 64) * 8192u : 0u;  // phi(k) - bf16(phi(k))
  L.v = o; o += 16384u;  // value rows 64..127 are a zero pad when dv = 64
  L.stage = up1k(o);
  o = 2u * L.stage;
  L.bar = o; o += 64u;
  L.total = o;
  return L;
}

template <int DK, int DV, bool ELU>
__global__ void __launch_bounds__(kNThreads)
nc_sum_kernel(const ChunkParams p, int nsplit, float *__restrict__ part, float *__restrict__ zpart,
              const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const NLayout L = n_layout(DK, ELU);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int T = p.T, nch = (T + kC - 1) / kC;
  const int bh = blockIdx.x / nsplit, sp = blockIdx.x % nsplit;
  const int c0 = (int)(((long long)sp * nch) / nsplit), c1 = (int)(((long long)(sp + 1) * nch) / nsplit);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.bar);
  uint64_t *full = bars, *empty = bars + 2, *drain = bars + 4;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 5);
  auto stage = [&](int s) { return sm + (uint32_t)s * L.stage; };
  constexpr uint32_t bytes = DK * kC * 2u + DV * kC * 2u;
  auto issue = [&](int j, int s) {
    uint8_t *st = stage(s);
    mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
    for (int a = 0; a < DK / 64; ++a) tma_load_3d(st + L.k + a * 8192, &tm_k, &full[s], 64 * a, j * kC, bh);
#pragma unroll
    for (int a = 0; a < DV / 64; ++a) tma_load_3d(st + L.v + a * 8192, &tm_v, &full[s], 64 * a, j * kC, bh);
  };
  if (warp == 0) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  if (DV == 64) {
    for (int q = tid; q < 2 * 512; q += kNThreads)
      reinterpret_cast<uint4 *>(stage(q >> 9) + L.v + 8192)[q & 511] = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async();
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&full[b], 1);
      mbar_init(&empty[b], 1);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    for (int j = c0; j < c0 + 2 && j < c1; ++j) issue(j, j - c0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t tl = tbase + (static_cast<uint32_t>(warp * 32) << 16);
  // elu+1: thread (cg, r0) owns key channels 8 cg .. 8 cg + 7 on rows r0, r0 + kStep, ...
  constexpr int kGroups = DK / 8, kStep = kNThreads / kGroups;
  const int cg = tid % kGroups, r0 = tid / kGroups;
  float zacc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  // thread 0 tracks failures (a wait that gave up) and the last chunk loaded into each stage
  bool ok = true;
  int last0 = c0, last1 = min(c0 + 1, c1 - 1);
  for (int j = c0; j < c1; ++j) {
    const int it = j - c0, s = it & 1, n = min(kC, T - j * kC);
    const uint32_t ph = (uint32_t)(it >> 1) & 1u;
    if (tid == 0 && ok) ok = mbar_wait_bounded(&full[s], ph, kSpinLimit);
    if (!__syncthreads_and(ok)) {  // every thread leaves together
      ok = false;
      break;
    }
    uint8_t *st = stage(s);
    if (ELU) {  // phi(k) = elu(k) + 1 on the rows in [0, n), zero beyond; bf16 high part in place, low part apart
#pragma unroll 2
      for (int r = r0; r < kC; r += kStep) {
        const uint32_t off = (uint32_t)(cg >> 3) * 8192u + sw128_off(r, (cg & 7) * 8);
        float f[8], fh[8];
        unpack8(*reinterpret_cast<const uint4 *>(st + L.k + off), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          f[e] = (r < n) ? (f[e] > 0.f ? f[e] + 1.f : __expf(f[e])) : 0.f;
          zacc[e] += f[e];
        }
        const uint4 hi = pack8(f);
        unpack8(hi, fh);
#pragma unroll
        for (int e = 0; e < 8; ++e) fh[e] = f[e] - fh[e];
        *reinterpret_cast<uint4 *>(st + L.k + off) = hi;
        *reinterpret_cast<uint4 *>(st + L.klo + off) = pack8(fh);
      }
      fence_proxy_async();
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      // S^T += V^T K: V as MN-major A (M = 128 value rows), K as MN-major B (N = dk)
      constexpr uint32_t id = idesc_bf16_f32(128, DK, true, true);
      const uint32_t a_v = smem_u32(st + L.v), a_k = smem_u32(st + L.k), a_kl = smem_u32(st + L.klo);
#pragma unroll
      for (int kk = 0; kk < kC / 16; ++kk) {
        const uint64_t dv_ = desc_sw128(a_v + kk * 2048, 8192, 1024);
        mma_bf16(tbase, dv_, desc_sw128(a_k + kk * 2048, 8192, 1024), id, (it > 0 || kk > 0) ? 1u : 0u);
        if (ELU) mma_bf16(tbase, dv_, desc_sw128(a_kl + kk * 2048, 8192, 1024), id, 1u);
      }
      mma_commit(&empty[s]);
      if (j + 2 < c1) {  // the stage takes chunk j + 2 once these MMAs have read it
        if (mbar_wait_bounded(&empty[s], ph, kSpinLimit)) {
          issue(j + 2, s);
          if (s == 0) last0 = j + 2; else last1 = j + 2;
        } else {
          ok = false;
        }
      }
    }
  }
  if (tid == 0) {
    mma_commit(drain);
    if (!mbar_wait_bounded(drain, 0, kSpinLimit)) ok = false;
    if (!ok) {
      atomicOr(p.status, kStatusTimeout);
      // loads still in flight land before the CTA leaves (bounded)
      (void)mbar_wait_bounded(&full[0], (uint32_t)((last0 - c0) >> 1) & 1u, 4096);
      if (c1 - c0 > 1) (void)mbar_wait_bounded(&full[1], (uint32_t)((last1 - c0) >> 1) & 1u, 4096);
    }
  }
  ok = __syncthreads_and(ok);
  tc_fence_after();
  if (ok) {
    // partial S of this T-range, key-major [c][v]: thread = TMEM lane = value row v, so
    // every store of one key channel is contiguous across the warp
    const int v = tid;
    float *dst = part + ((size_t)bh * nsplit + sp) * DV * DK + v;
#pragma unroll 1
    for (int cc = 0; cc < DK; cc += 32) {
      float x[32];
      tmem_ld32(tl + cc, x);
      tmem_wait_ld();
      if (v < DV) {
#pragma unroll
        for (int e = 0; e < 32; ++e) dst[(size_t)(cc + e) * DV] = x[e];
      }
    }
    if (ELU) {  // z partial: reduce the row-strided thread sums per channel
      float *zs = reinterpret_cast<float *>(stage(0));  // the stages are idle now
#pragma unroll
      for (int e = 0; e < 8; ++e) zs[r0 * DK + cg * 8 + e] = zacc[e];
      __syncthreads();
      if (tid < DK) {
        float z = 0.f;
        for (int r = 0; r < kStep; ++r) z += zs[r * DK + tid];
        zpart[((size_t)bh * nsplit + sp) * DK + tid] = z;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, 128);
}

// S_total = S0 + the partial sums of the key-major partials; S_final, and the
// bf16 image of S_total^T as a high/low pair (x = hi + lo to about 2^-16) in
// the output kernel's operand layout (value rows beyond dv zero). One CTA per
// (head, 16 value rows): the tile goes through shared memory so that both the
// [c][v] reads and writes and the image rows are contiguous. elu+1: z_total.
constexpr int kFRows = 16;

template <int DK, int DV, bool ELU>
__global__ void __launch_bounds__(256)
nc_finalize_kernel(const ChunkParams p, int nsplit, const float *__restrict__ part,
                   const float *__restrict__ zpart, uint8_t *__restrict__ img, float *__restrict__ zws) {
  constexpr int W = DV + (ELU ? 1 : 0);
  __shared__ float tile[DK][kFRows + 1];
  const int bh = blockIdx.x / (128 / kFRows), v0 = (blockIdx.x % (128 / kFRows)) * kFRows;
  const int tid = threadIdx.x;
  // sums: thread (c-slot, row) with the row fastest (16 contiguous floats of one channel)
  for (int i = tid; i < DK * kFRows; i += 256) {
    const int c = i / kFRows, r = i % kFRows, v = v0 + r;
    float x = 0.f;
    if (v < DV) {
      x = p.S0 ? p.S0[((size_t)bh * DK + c) * W + v] : 0.f;
      const float *pp = part + (size_t)bh * nsplit * DV * DK + (size_t)c * DV + v;
      for (int q = 0; q < nsplit; ++q) x += pp[(size_t)q * DV * DK];
      if (p.S_final) p.S_final[((size_t)bh * DK + c) * W + v] = x;
    }
    tile[c][r] = x;
  }
  __syncthreads();
  // image rows v0 .. v0+15: thread writes a 4-byte pair of keys of one row (rows contiguous)
  const size_t lo_off = (size_t)p.B * p.H * blob_bytes(DK);
  uint8_t *im = img + (size_t)bh * blob_bytes(DK);
  for (int i = tid; i < kFRows * (DK / 2); i += 256) {
    const int r = i / (DK / 2), c = 2 * (i % (DK / 2)), v = v0 + r;
    const float x0 = tile[c][r], x1 = tile[c + 1][r];
    const __nv_bfloat162 hi = __floats2bfloat162_rn(x0, x1);
    const __nv_bfloat162 lo = __floats2bfloat162_rn(x0 - __low2float(hi), x1 - __high2float(hi));
    const size_t off = (size_t)(c >> 6) * 16384u + sw128_off(v, c & 63);
    *reinterpret_cast<__nv_bfloat162 *>(im + off) = hi;
    *reinterpret_cast<__nv_bfloat162 *>(im + lo_off + off) = lo;
  }
  if (ELU && v0 == 0 && tid < DK) {
    float z = p.S0 ? p.S0[((size_t)bh * DK + tid) * W + DV] : 0.f;
    for (int q = 0; q < nsplit; ++q) z += zpart[((size_t)bh * nsplit + q) * DK + tid];
    zws[(size_t)bh * DK + tid] = z;
    if (p.S_final) p.S_final[((size_t)bh * DK + tid) * W + DV] = z;
  }
}

// Parallel state pass of the materialised variant for the modes without decay
// (linear, elu+1): the state entering chunk i is S0 plus the sum of the earlier
// chunks' K^T V (z: of their phi(k) sums), so nc_sum_kernel forms every 64-token
// chunk's partial at once (one split per chunk) and mat_scan_kernel walks a
// head's chunks for 16 value rows, writing the state at every image boundary as
// the output pass's bf16 image (the serial state pass's layout: S^T rows, value
// rows beyond dv zero), z there, and S_final. The partials' loads run
// kScanDepth chunks ahead of the running sums.
constexpr int kScanDepth = 4;

template <int DK, int DV, bool ELU>
__global__ void __launch_bounds__(256)
mat_scan_kernel(const ChunkParams p, int nch, int istride, const float *__restrict__ part,
                const float *__restrict__ zpart, uint8_t *__restrict__ ws, float *__restrict__ zws) {
  constexpr int W = DV + (ELU ? 1 : 0);
  constexpr int EPT = DK * kFRows / 256;  // running-sum elements per thread
  __shared__ float tile[DK][kFRows + 1];
  const int bh = blockIdx.x / (128 / kFRows), v0 = (blockIdx.x % (128 / kFRows)) * kFRows;
  const int tid = threadIdx.x;
  const int nimg = (nch + istride - 1) / istride;
  const bool zthr = ELU && v0 == 0 && tid < DK;  // the thread of key channel tid's z
  // element e of the thread: key channel (tid + 256 e) / 16, value row v0 + (tid + 256 e) % 16
  int ce[EPT], ve[EPT];
  float acc[EPT];
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int i = tid + 256 * e;
    ce[e] = i / kFRows;
    ve[e] = v0 + i % kFRows;
    acc[e] = (p.S0 && ve[e] < DV) ? p.S0[((size_t)bh * DK + ce[e]) * W + ve[e]] : 0.f;
  }
  float z = (zthr && p.S0) ? p.S0[((size_t)bh * DK + tid) * W + DV] : 0.f;
  const float *pp = part + (size_t)bh * nch * DV * DK;
  const float *zp = ELU ? zpart + (size_t)bh * nch * DK : nullptr;
  // the partials of chunks j .. j + kScanDepth - 1 in flight
  float buf[kScanDepth][EPT], zbuf[kScanDepth];
  auto load = [&](int j, float (&dst)[EPT], float &zdst) {
#pragma unroll
    for (int e = 0; e < EPT; ++e)
      dst[e] = (j < nch && ve[e] < DV) ? __ldg(pp + (size_t)j * DV * DK + (size_t)ce[e] * DV + ve[e]) : 0.f;
    zdst = (zthr && j < nch) ? __ldg(zp + (size_t)j * DK + tid) : 0.f;
  };
#pragma unroll
  for (int d = 0; d < kScanDepth; ++d) load(d, buf[d], zbuf[d]);
  for (int j0 = 0; j0 < nch; j0 += kScanDepth) {
#pragma unroll
    for (int d = 0; d < kScanDepth; ++d) {
      const int j = j0 + d;
      if (j >= nch) break;  // uniform across the CTA
      if (j % istride == 0) {  // the state entering image j / istride
        const int im_i = j / istride;
#pragma unroll
        for (int e = 0; e < EPT; ++e) tile[ce[e]][ve[e] - v0] = acc[e];
        if (zthr) zws[((size_t)bh * nimg + im_i) * DK + tid] = z;
        __syncthreads();
        uint8_t *im = ws + ((size_t)bh * nimg + im_i) * blob_bytes(DK);
        for (int i = tid; i < kFRows * (DK / 2); i += 256) {
          const int r = i / (DK / 2), c = 2 * (i % (DK / 2));
          *reinterpret_cast<__nv_bfloat162 *>(im + (size_t)(c >> 6) * 16384u + sw128_off(v0 + r, c & 63)) =
              __floats2bfloat162_rn(tile[c][r], tile[c + 1][r]);
        }
        __syncthreads();
      }
#pragma unroll
      for (int e = 0; e < EPT; ++e) acc[e] += buf[d][e];
      z += zbuf[d];
      load(j + kScanDepth, buf[d], zbuf[d]);
    }
  }
  if (p.S_final) {
#pragma unroll
    for (int e = 0; e < EPT; ++e)
      if (ve[e] < DV) p.S_final[((size_t)bh * DK + ce[e]) * W + ve[e]] = acc[e];
    if (zthr) p.S_final[((size_t)bh * DK + tid) * W + DV] = z;
  }
}

template <int DK, int DV, int KIND>
cudaError_t launch_scan_state(const ChunkParams &p, uint8_t *ws, float *zws, const CUtensorMap &mk,
                              const CUtensorMap &mv, cudaStream_t stream) {
  constexpr bool ELU = KIND == kElu1;
  const int BH = p.B * p.H, nch = (p.T + kC - 1) / kC, istride = p.C == kC2 ? 2 : 1;
  float *part = reinterpret_cast<float *>(ws + mat_workspace_bytes(p));  // [B*H][nch][dk][dv], after the images
  float *zpart = part + (size_t)BH * nch * DV * DK;                   // [B*H][nch][dk] (elu+1)
  const size_t sn = n_layout(DK, ELU).total + 1024;
  auto ka = nc_sum_kernel<DK, DV, ELU>;
  cudaError_t e = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sn);
  if (e == cudaSuccess) {
    ka<<<(unsigned)((size_t)BH * nch), kNThreads, sn, stream>>>(p, nch, part, zpart, mk, mv);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    mat_scan_kernel<DK, DV, ELU><<<(unsigned)(BH * (128 / kFRows)), 256, 0, stream>>>(p, nch, istride, part, zpart,
                                                                                      ws, zws);
    e = cudaGetLastError();
  }
  return e;
}

// Output of the non-causal form: persistent CTAs (two per SM) each walk a
// contiguous run of (head, chunk) pairs. At each new head a CTA takes the
// head's state image (high and low parts) and z by bulk copies, then per
// chunk: q tile by TMA (two stages), elu+1: phi(q) and phi(q).z,
// O^T = S_hi^T Q^T + S_lo^T Q^T on the tensor cores, and o stored straight
// from registers (pairs of rows exchanged between lanes: 4-byte stores).
constexpr int kOThreads = 128;

struct OLayout {
  uint32_t shi, slo, q, z, den, bar, total;
};
__host__ __device__ inline OLayout o_layout(int dk) {
  OLayout L;
  uint32_t o = 0;
  L.shi = o; o += blob_bytes(dk);
  L.slo = o; o += blob_bytes(dk);
  L.q = o; o += 2u * (uint32_t)(dk / 64) * 8192u;  // two stages of the q tile
  L.z = o; o += 512u;
  L.den = o; o += 256u;
  L.bar = o; o += 64u;
  L.total = o;
  return L;
}

template <int DK, int DV, bool ELU>
__global__ void __launch_bounds__(kOThreads, 2)
nc_out_kernel(const ChunkParams p, const uint8_t *__restrict__ img, const float *__restrict__ zws,
              const __grid_constant__ CUtensorMap tm_q) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const OLayout L = o_layout(DK);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.T, nch = (T + kC - 1) / kC;
  const long long total = (long long)p.B * p.H * nch;
  const long long g0 = (blockIdx.x * total) / gridDim.x, g1 = ((blockIdx.x + 1) * total) / gridDim.x;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.bar);
  uint64_t *qfull = bars, *mdone = bars + 2, *sfull = bars + 3;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 4);
  float *zs = reinterpret_cast<float *>(sm + L.z), *den = reinterpret_cast<float *>(sm + L.den);
  auto qstage = [&](int s) { return sm + L.q + (uint32_t)s * (DK / 64) * 8192u; };
  auto issue = [&](long long g, int s) {
    const int bh = (int)(g / nch), j = (int)(g % nch);
    mbar_arrive_expect_tx(&qfull[s], DK * kC * 2u);
#pragma unroll
    for (int a = 0; a < DK / 64; ++a) tma_load_3d(qstage(s) + a * 8192, &tm_q, &qfull[s], 64 * a, j * kC, bh);
  };
  if (warp == 0) {
    tmem_alloc(tmem_slot, 64);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&qfull[0], 1);
    mbar_init(&qfull[1], 1);
    mbar_init(mdone, 1);
    mbar_init(sfull, 1);
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    for (long long g = g0; g < g0 + 2 && g < g1; ++g) issue(g, (int)(g - g0));
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t tl = tbase + (static_cast<uint32_t>(warp * 32) << 16);
  bool ok = true;
  int cur_bh = -1, nloads = 0;
  long long last0 = g0, last1 = g0 + 1;  // thread 0: the last chunk loaded into each stage
  for (long long g = g0; g < g1; ++g) {
    const int it = (int)(g - g0), s = it & 1, bh = (int)(g / nch), j = (int)(g % nch);
    const uint32_t ph = (uint32_t)(it >> 1) & 1u;
    if (bh != cur_bh) {
      // the head's state image and z (the previous head's MMAs have completed: each chunk
      // waits for its own)
      if (tid == 0 && ok) {
        const size_t lo_off = (size_t)p.B * p.H * blob_bytes(DK);
        mbar_arrive_expect_tx(sfull, 2u * blob_bytes(DK) + (ELU ? DK * 4u : 0u));
        bulk_load(sm + L.shi, img + (size_t)bh * blob_bytes(DK), blob_bytes(DK), sfull);
        bulk_load(sm + L.slo, img + lo_off + (size_t)bh * blob_bytes(DK), blob_bytes(DK), sfull);
        if (ELU) bulk_load(zs, zws + (size_t)bh * DK, DK * 4u, sfull);
        ok = mbar_wait_bounded(sfull, (uint32_t)nloads & 1u, kSpinLimit);
      }
      ++nloads;
      cur_bh = bh;
    }
    if (tid == 0 && ok) ok = mbar_wait_bounded(&qfull[s], ph, kSpinLimit);
    if (!__syncthreads_and(ok)) {  // every thread leaves together
      ok = false;
      break;
    }
    uint8_t *qt = qstage(s);
    const int n = min(kC, T - j * kC);
    if (ELU) {  // phi(q) on rows in [0, n), zero beyond; then phi(q).z per row
      constexpr int kGroups = DK / 8, kStep = kOThreads / kGroups;
      const int cg = tid % kGroups;
#pragma unroll 2
      for (int r = tid / kGroups; r < kC; r += kStep) {
        uint4 *ptr = reinterpret_cast<uint4 *>(qt + (uint32_t)(cg >> 3) * 8192u + sw128_off(r, (cg & 7) * 8));
        float f[8];
        unpack8(*ptr, f);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = (r < n) ? (f[e] > 0.f ? f[e] + 1.f : __expf(f[e])) : 0.f;
        *ptr = pack8(f);
      }
      __syncthreads();
      if (tid < kC) {
        float acc = 0.f;
        for (int g8 = 0; g8 < DK / 8; ++g8) {
          float f[8];
          unpack8(*reinterpret_cast<const uint4 *>(qt + (uint32_t)(g8 >> 3) * 8192u + sw128_off(tid, (g8 & 7) * 8)), f);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc = fmaf(f[e], zs[g8 * 8 + e], acc);
        }
        den[tid] = acc;
      }
      fence_proxy_async();
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      // O^T = S_hi^T Q^T + S_lo^T Q^T: the image K-major (key blocks 16 KB apart), q K-major (8 KB apart)
      constexpr uint32_t id = idesc_bf16_f32(128, 64, false, false);
      const uint32_t a_hi = smem_u32(sm + L.shi), a_lo = smem_u32(sm + L.slo), a_q = smem_u32(qt);
#pragma unroll
      for (int kk = 0; kk < DK / 16; ++kk) {
        const uint32_t ka = (kk >> 2) * 16384 + (kk & 3) * 32, kb = (kk >> 2) * 8192 + (kk & 3) * 32;
        mma_bf16(tbase, desc_sw128(a_hi + ka, 16, 1024), desc_sw128(a_q + kb, 16, 1024), id, kk > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int kk = 0; kk < DK / 16; ++kk) {
        const uint32_t ka = (kk >> 2) * 16384 + (kk & 3) * 32, kb = (kk >> 2) * 8192 + (kk & 3) * 32;
        mma_bf16(tbase, desc_sw128(a_lo + ka, 16, 1024), desc_sw128(a_q + kb, 16, 1024), id, 1u);
      }
      mma_commit(mdone);
      ok = mbar_wait_bounded(mdone, (uint32_t)it & 1u, kSpinLimit);
      if (ok && g + 2 < g1) {  // the stage is free once the MMAs have read it
        issue(g + 2, s);
        if (s == 0) last0 = g + 2; else last1 = g + 2;
      }
    }
    if (!__syncthreads_and(ok)) {
      ok = false;
      break;
    }
    tc_fence_after();
    {  // epilogue: thread = TMEM lane = value row v; pairs of rows exchanged so each thread writes 4 bytes
      const int v = tid;
      const bool odd = lane & 1;
      __nv_bfloat16 *og = static_cast<__nv_bfloat16 *>(p.o) + ((size_t)bh * T + (size_t)j * kC) * DV;
#pragma unroll 1
      for (int r0 = 0; r0 < kC; r0 += 32) {
        float a[32];
        tmem_ld32(tl + r0, a);
        tmem_wait_ld();
        if (ELU) {
#pragma unroll
          for (int e = 0; e < 32; ++e) a[e] = __fdividef(a[e], den[r0 + e]);
        }
        if (v < DV) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float send = odd ? a[e] : a[e + 1];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
            const int r = r0 + e + (odd ? 1 : 0);
            const uint32_t w = odd ? pack_bf16(recv, a[e + 1]) : pack_bf16(a[e], recv);
            if (r < n) *reinterpret_cast<uint32_t *>(og + (size_t)r * DV + v - (odd ? 1 : 0)) = w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 2) (void)__shfl_xor_sync(0xffffffffu, a[e], 1);
        }
      }
    }
    tc_fence_before();  // the TMEM reads are done before the next chunk's MMAs overwrite it
  }
  if (tid == 0) {
    if (!ok) {
      atomicOr(p.status, kStatusTimeout);
      // loads still in flight land before the CTA leaves (bounded)
      (void)mbar_wait_bounded(&qfull[0], (uint32_t)((last0 - g0) >> 1) & 1u, 4096);
      if (g1 - g0 > 1) (void)mbar_wait_bounded(&qfull[1], (uint32_t)((last1 - g0) >> 1) & 1u, 4096);
      if (nloads > 0) (void)mbar_wait_bounded(sfull, (uint32_t)(nloads - 1) & 1u, 4096);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, 64);
}

int nc_splits(const ChunkParams &p) {
  const long long BH = (long long)p.B * p.H;
  const int nch = (p.T + kC - 1) / kC;
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 148;
  long long want = (2LL * sms + BH - 1) / BH;  // about two CTAs per SM
  want = std::min<long long>(want, std::max(1, nch / 4));  // at least four chunks each
  return (int)std::max<long long>(1, want);
}

template <int DK, int DV, int KIND>
int launch_nc_typed(const ChunkParams &p, uint8_t *ws, cudaStream_t stream) {
  constexpr bool ELU = KIND == kElu1;
  const int BH = p.B * p.H, nch = (p.T + kC - 1) / kC, ns = nc_splits(p);
  uint8_t *img = ws;  // B*H high images, then B*H low images
  float *zws = reinterpret_cast<float *>(img + 2 * (size_t)BH * blob_bytes(DK));  // [B*H][dk] z_total
  float *part = zws + (size_t)BH * DK;  // [B*H][splits][dk][dv] partial S
  float *zpart = part + (size_t)BH * ns * DV * DK;  // [B*H][splits][dk] partial z (elu+1)
  const NLayout Ln = n_layout(DK, ELU);
  const size_t sn = Ln.total + 1024;
  CUtensorMap mq, mk, mv, mo;
  const bool ok = make_map(&mq, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DK, p.T, BH, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
                  make_map(&mk, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DK, p.T, BH, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
                  make_map(&mv, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, p.T, BH, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
                  make_map(&mo, p.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, p.T, BH, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) {
    set_error("la_chunk_fwd: cuTensorMapEncodeTiled rejected a tensor map");
    return LA_ERR_CUDA;
  }
  auto ka = nc_sum_kernel<DK, DV, ELU>;
  auto kf = nc_finalize_kernel<DK, DV, ELU>;
  auto kb = nc_out_kernel<DK, DV, ELU>;
  const size_t so = o_layout(DK).total + 1024;
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 148;
  const long long nout = std::min<long long>((long long)BH * nch, 2LL * sms);
  cudaError_t e = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sn);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kb, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)so);
  if (e == cudaSuccess) {
    ka<<<(unsigned)(BH * ns), kNThreads, sn, stream>>>(p, ns, part, zpart, mk, mv);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    kf<<<(unsigned)(BH * (128 / kFRows)), 256, 0, stream>>>(p, ns, part, zpart, img, zws);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    kb<<<(unsigned)nout, kOThreads, so, stream>>>(p, img, zws, mq);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_error("la_chunk_fwd: non-causal kernels failed to launch: %s", cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  return LA_OK;
}

template <int KIND>
int launch_nc_kind(const ChunkParams &p, uint8_t *ws, cudaStream_t stream) {
  if (p.dk == 128 && p.dv == 128) return launch_nc_typed<128, 128, KIND>(p, ws, stream);
  if (p.dk == 128 && p.dv == 64) return launch_nc_typed<128, 64, KIND>(p, ws, stream);
  if (p.dk == 64 && p.dv == 128) return launch_nc_typed<64, 128, KIND>(p, ws, stream);
  return launch_nc_typed<64, 64, KIND>(p, ws, stream);
}

}  // namespace

size_t mat_workspace_bytes(const ChunkParams &p) {
  // one state image (and elu+1 normaliser) per chunk of p.C tokens
  const size_t c = p.C == kC2 ? kC2 : kC;
  const size_t nch = (size_t)(p.T + c - 1) / c, BH = (size_t)p.B * p.H;
  size_t b = BH * nch * blob_bytes(p.dk);
  if (p.kind == kElu1) b += BH * nch * p.dk * sizeof(float);
  return b;
}

size_t mat_scan_bytes(const ChunkParams &p) {
  if (p.kind != kLinear && p.kind != kElu1) return 0;
  const size_t nch = (size_t)(p.T + kC - 1) / kC, BH = (size_t)p.B * p.H;
  return BH * nch * (size_t)p.dv * p.dk * sizeof(float) + (p.kind == kElu1 ? BH * nch * p.dk * sizeof(float) : 0);
}

int launch_chunk_mat(const ChunkParams &p, void *workspace, cudaStream_t stream, bool scan) {
  if (!encode_fn()) {
    set_error("la_chunk_fwd: cuTensorMapEncodeTiled is unavailable");
    return LA_ERR_CUDA;
  }
  if (p.C == kC2 && (p.kind == kGla || p.kind == kOuter || p.kind == kGdn || p.kind == kKda)) {
    set_error("la_chunk_fwd: C=128 covers LA_LINEAR, LA_ELU1_NORM, LA_RETNET and LA_SCALAR_GATE");
    return LA_ERR_UNSUPPORTED;
  }
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  const size_t c = p.C == kC2 ? kC2 : kC;
  const size_t nch = (size_t)(p.T + c - 1) / c, BH = (size_t)p.B * p.H;
  float *zws = (p.kind == kElu1) ? reinterpret_cast<float *>(ws + BH * nch * blob_bytes(p.dk)) : nullptr;
  switch (p.kind) {
    case kLinear: return launch_kind<kLinear>(p, ws, zws, scan, stream);
    case kElu1: return launch_kind<kElu1>(p, ws, zws, scan, stream);
    case kRetnet: return launch_kind<kRetnet>(p, ws, zws, false, stream);
    case kScalar: return launch_kind<kScalar>(p, ws, zws, false, stream);
    case kGla: return launch_kind<kGla>(p, ws, zws, false, stream);
    default:
      set_error("la_chunk_fwd: the materialised variant covers the unit-write modes only");
      return LA_ERR_UNSUPPORTED;
  }
}

}  // namespace la

namespace la {

size_t nc_workspace_bytes(const ChunkParams &p) {
  const size_t BH = (size_t)p.B * p.H, ns = (size_t)nc_splits(p);
  return 2 * BH * blob_bytes(p.dk) + BH * p.dk * sizeof(float) + BH * ns * p.dv * p.dk * sizeof(float) +
         BH * ns * p.dk * sizeof(float);
}

int launch_chunk_noncausal(const ChunkParams &p, void *workspace, cudaStream_t stream) {
  if (!encode_fn()) {
    set_error("la_chunk_fwd: cuTensorMapEncodeTiled is unavailable");
    return LA_ERR_CUDA;
  }
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  if (p.kind == kLinear) return launch_nc_kind<kLinear>(p, ws, stream);
  if (p.kind == kElu1) return launch_nc_kind<kElu1>(p, ws, stream);
  set_error("la_chunk_fwd: LA_NONCAUSAL covers LA_LINEAR and LA_ELU1_NORM only");
  return LA_ERR_UNSUPPORTED;
}

}  // namespace la
