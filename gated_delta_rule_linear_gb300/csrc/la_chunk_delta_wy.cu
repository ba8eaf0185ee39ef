// Chunk forward for the gated delta rule in two kernels, bf16 inputs, fp32
// state, dk = dv = 128 ("Talk Linear Attention" section 6.2, WY/UT form;
// "LLM attention optimisation", Gated DeltaNet section):
//
//   b_r = sum_{t<=r} g_t (log-gate prefix inside the chunk)
//   A_rs = beta_r e^{b_r - b_s} k_r.k_s (s < r),  T = (I + A)^-1,  T' = T diag(beta)
//   W = T' diag(e^b) K,  U = T' V - W S_prev
//   O = Diag(e^b) Q S_prev + P U,  P_rs = e^{b_r - b_s} q_r.k_s (s <= r)
//   S <- e^{b_last} S_prev + K^T diag(e^{b_last - b}) U
//
// 1. wy_kernel: everything above that depends on neither S nor V nor Q, the
//    triangular solve, for every (head, chunk) at once: K K^T on the tensor
//    cores (warp MMAs), the gated A, T by 16x16 forward substitution and three
//    block levels, and T' written to a workspace as one 8 KB bf16 image per
//    chunk in the 128-byte-swizzled layout the second kernel's MMA reads.
// 2. chain_kernel: a pair of CTAs (a cluster of two) per head, CTA r owning
//    value columns 64r .. 64r + 63 of S, U and O. The S-dependent chain per
//    chunk is: S = e^{b_last} S + dS (fp32 in registers, a thread per
//    (value column, half of the key channels)), its bf16 copy into tensor
//    memory, U^T = V^T T'^T + S^T (-W)^T, the U epilogue, and dS^T = U'^T K
//    (a fresh accumulator every chunk, so the state never makes a round trip
//    through tensor memory). The S-independent side of a chunk (P and -W) is
//    computed by CTA (chunk mod 2) and copied into the other CTA's shared
//    memory; it reads the same staged q/k tiles and T' image as the chain.
//
// All waits are bounded (status word, then the CTA skips its remaining work).
#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "la_tc_common.cuh"
#include "la_wy.cuh"

namespace la {
namespace {

using namespace sm100;
using namespace tc;
using namespace wy;

constexpr int DK = 128, DV = 128, NV = 64;  // NV: value columns per CTA of the pair
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kImgBytes = 8192u;  // one bf16 64x64 T' image

// =====================================================================================
// 1. The triangular solve for every (head, chunk): T' images
// =====================================================================================

constexpr int kAThreads = 128;
constexpr int kAPerSM = 4;   // resident CTAs per SM (shared memory: two key tiles and A)
constexpr int kKp = DK + 8;  // bf16 pitch of the staged key rows: 272 B, ldmatrix rows on distinct banks

struct WyParams {
  const __nv_bfloat16 *k;
  const float *g, *beta;
  uint8_t *img;  // [B*H][nchunks][8192]
  int T, nchunks;
  long long items;  // B*H*nchunks
};

__device__ __forceinline__ void ldsm_x4(uint32_t *r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t *r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}
__device__ __forceinline__ void mma_16x8x16_bf16(float *d, const uint32_t *a, const uint32_t *b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// 16-byte asynchronous copy global -> shared; src_bytes = 0 fills zeros.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Shared memory: two key tiles (the next item's rows land while the current one
// is solved; T reuses the current tile once K K^T is formed), A, and per tile the
// log2 prefix of the gates and beta.
constexpr uint32_t kWyTile = 64u * kKp * 2u;  // 17408
// per tile: log2 prefix, beta, beta_r e^{b_r - b_last}, e^{b_last - b_s}, fast-path flag
constexpr int kWyB2 = 0, kWyBt = 64, kWyFr = 128, kWyFc = 192, kWyFast = 256, kWyScF = 260;
constexpr uint32_t kWyKs = 0, kWyAf = 2u * kWyTile, kWySc = kWyAf + 64u * kAp * 4u,
                   kWyBytes = kWySc + 2u * kWyScF * 4u;
constexpr float kWyFastLimit = 100.f;  // log2 units: -b_last below this -> factorised gate products
static_assert(kWyTile >= 64u * kAp * 4u, "T reuses a key tile's space");

// K K^T over the lower block triangle: the 20 (16-row block, 8-column tile) units
// with tile <= 2 block + 1, five per warp (the diagonal block's upper part is masked
// when A is formed). Unit u of warp w is entry 5w + u of this list.
__constant__ unsigned char kGUnits[20][2] = {{0, 0}, {0, 1}, {1, 0}, {1, 1}, {1, 2}, {1, 3}, {2, 0},
                                            {2, 1}, {2, 2}, {2, 3}, {2, 4}, {2, 5}, {3, 0}, {3, 1},
                                            {3, 2}, {3, 3}, {3, 4}, {3, 5}, {3, 6}, {3, 7}};

// Start the copies of one item's key rows: two threads per row, eight 16-byte
// pieces each, zeros past T.
__device__ __forceinline__ void wy_issue(const WyParams &p, long long item, uint8_t *tile, int tid) {
  const int bh = (int)(item / p.nchunks), j = (int)(item % p.nchunks), T = p.T, t0 = j * kC;
  const int nrow = min(kC, T - t0);
  const int r = tid >> 1, h = tid & 1;
  const __nv_bfloat16 *src = p.k + ((size_t)bh * T + t0 + (r < nrow ? r : 0)) * DK + h * 64;
  __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(tile) + r * kKp + h * 64;
#pragma unroll
  for (int i = 0; i < 8; ++i) cp_async16(dst + 8 * i, src + 8 * i, r < nrow ? 16u : 0u);
}
// One item's gates and beta for tokens lane and lane + 32 (zero gates and beta past T).
__device__ __forceinline__ void wy_scalars(const WyParams &p, long long item, int lane, float *gb) {
  const int bh = (int)(item / p.nchunks), j = (int)(item % p.nchunks), T = p.T, t = j * kC + lane;
  gb[0] = (p.g && t < T) ? __ldg(p.g + (size_t)bh * T + t) : 0.f;
  gb[1] = (p.g && t + 32 < T) ? __ldg(p.g + (size_t)bh * T + t + 32) : 0.f;
  gb[2] = t < T ? (p.beta ? __ldg(p.beta + (size_t)bh * T + t) : 1.f) : 0.f;
  gb[3] = t + 32 < T ? (p.beta ? __ldg(p.beta + (size_t)bh * T + t + 32) : 1.f) : 0.f;
}

__global__ void __launch_bounds__(kAThreads, kAPerSM) wy_kernel(const WyParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  float *Af = reinterpret_cast<float *>(smem + kWyAf);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.T;
  long long item = blockIdx.x;
  if (item >= p.items) return;
  float gb[4] = {0.f, 0.f, 0.f, 0.f};  // warp 0: this item's gates and beta (the next item's land meanwhile)
  wy_issue(p, item, smem + kWyKs, tid);
  cp_async_commit();
  if (warp == 0) wy_scalars(p, item, lane, gb);
  for (int buf = 0; item < p.items; item += gridDim.x, buf ^= 1) {
    uint8_t *tile = smem + kWyKs + (uint32_t)buf * kWyTile;
    float *raw = reinterpret_cast<float *>(smem + kWySc) + buf * kWyScF;
    const long long next = item + gridDim.x;
    if (next < p.items) wy_issue(p, next, smem + kWyKs + (uint32_t)(buf ^ 1) * kWyTile, tid);
    cp_async_commit();
    cp_async_wait<1>();  // this item's copies have landed (the next item's may still fly)
    __syncthreads();
    const int bh = (int)(item / p.nchunks), j = (int)(item % p.nchunks), t0 = j * kC;
    const int nrow = min(kC, T - t0);
    const __nv_bfloat16 *Ks = reinterpret_cast<const __nv_bfloat16 *>(tile);
    float *Tf = reinterpret_cast<float *>(tile);  // after K K^T
    // per-token log2 prefix of the gates (in place over the raw gates) and beta,
    // zero gates and beta past T
    if (warp == 0) {
      const float be0 = gb[2], be1 = gb[3];
      float v0 = gb[0] * kLog2e, v1 = gb[1] * kLog2e;
      if (next < p.items) wy_scalars(p, next, lane, gb);
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
      raw[kWyB2 + lane] = v0;
      raw[kWyB2 + lane + 32] = v1;
      raw[kWyBt + lane] = be0;
      raw[kWyBt + lane + 32] = be1;
      raw[kWyFr + lane] = be0 * exp2f(v0 - bl);
      raw[kWyFr + lane + 32] = be1 * exp2f(v1 - bl);
      raw[kWyFc + lane] = exp2f(bl - v0);
      raw[kWyFc + lane + 32] = exp2f(bl - v1);
      if (lane == 0) raw[kWyFast] = (-bl < kWyFastLimit) ? 1.f : 0.f;
    }
    const float *b2 = raw + kWyB2, *bt = raw + kWyBt, *fr = raw + kWyFr, *fc = raw + kWyFc;
    // K K^T: five (row block, column tile) units per warp, fp32 accumulators
    float acc[5][4];
    {
#pragma unroll
      for (int u = 0; u < 5; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
      const uint32_t ks = smem_u32(Ks);
      const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = ((lane >> 4) & 1) * 8;
      const int brow = lane & 7, bcol = ((lane >> 3) & 1) * 8;
      // a warp's units span at most two row blocks (the first and the last unit's)
      const int rb0 = kGUnits[5 * warp][0], rb1 = kGUnits[5 * warp + 4][0];
#pragma unroll
      for (int kk = 0; kk < DK / 16; ++kk) {
        uint32_t a0[4], a1[4];
        ldsm_x4(a0, ks + (uint32_t)((16 * rb0 + arow) * kKp + kk * 16 + acol) * 2u);
        ldsm_x4(a1, ks + (uint32_t)((16 * rb1 + arow) * kKp + kk * 16 + acol) * 2u);
#pragma unroll
        for (int u = 0; u < 5; ++u) {
          const int rb = kGUnits[5 * warp + u][0], n = kGUnits[5 * warp + u][1];
          uint32_t b[2];
          ldsm_x2(b, ks + (uint32_t)((8 * n + brow) * kKp + kk * 16 + bcol) * 2u);
          mma_16x8x16_bf16(acc[u], rb == rb0 ? a0 : a1, b);
        }
      }
    }
    __syncthreads();  // the prefix is in; the key rows are dead (T takes their space)
    // A_rs = beta_r e^{b_r - b_s} k_r.k_s for s < r (zero on and above the diagonal and
    // for padding rows), rounded to tf32 for the block MMAs of the solve
    {
      const int g = lane >> 2, t4 = lane & 3;
      const bool fast = raw[kWyFast] != 0.f;
#pragma unroll
      for (int u = 0; u < 5; ++u) {
        const int rb = kGUnits[5 * warp + u][0], n = kGUnits[5 * warp + u][1];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int r = 16 * rb + g + 8 * half, s = 8 * n + 2 * t4;
          float f0, f1;  // beta_r e^{b_r - b_s}, beta_r e^{b_r - b_{s+1}}
          if (fast) {
            const float2 c2 = *reinterpret_cast<const float2 *>(fc + s);
            f0 = fr[r] * c2.x;
            f1 = fr[r] * c2.y;
          } else {
            f0 = bt[r] * exp2f(b2[r] - b2[s]);
            f1 = bt[r] * exp2f(b2[r] - b2[s + 1]);
          }
          const float x0 = (s < r && r < nrow) ? round_tf32(acc[u][2 * half] * f0) : 0.f;
          const float x1 = (s + 1 < r && r < nrow) ? round_tf32(acc[u][2 * half + 1] * f1) : 0.f;
          *reinterpret_cast<float2 *>(Af + r * kAp + s) = make_float2(x0, x1);
        }
      }
    }
    __syncthreads();
    // T = (I + A)^-1: 16x16 diagonal blocks by forward substitution, then the
    // off-diagonal blocks in three levels, T_ij = -T_ii sum_{j<=k<i} A_ik T_kj
    if (tid < kC) diag_inverse_16(Af, Tf, tid >> 4, tid & 15);
    __syncthreads();
#pragma unroll 1
    for (int lvl = 1; lvl < 4; ++lvl) {
      if (warp < 4 - lvl) {
        const int ib = warp + lvl, jb = warp;
        float a2[2][4] = {};
        for (int kb = jb; kb < ib; ++kb)
          block_mma_16(a2, Af + ib * 16 * kAp + kb * 16, Tf + kb * 16 * kAp + jb * 16, lane);
        float *Tij = Tf + ib * 16 * kAp + jb * 16;
        block_store_16(Tij, a2, 1.f, lane);
        __syncwarp();
        float a3[2][4] = {};
        block_mma_16(a3, Tf + ib * 16 * kAp + ib * 16, Tij, lane);
        __syncwarp();
        block_store_16(Tij, a3, -1.f, lane);
      }
      __syncthreads();
    }
    // T' = T diag(beta) as bf16, straight into the swizzled image: thread tid owns
    // row tid / 2, columns 32 (tid % 2) .. + 31
    {
      const int r = tid >> 1, c0 = (tid & 1) * 32;
      uint8_t *img = p.img + ((size_t)bh * p.nchunks + j) * kImgBytes;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float f[8];
#pragma unroll
        for (int e4 = 0; e4 < 2; ++e4) {
          const int s = c0 + 8 * q + 4 * e4;
          const float4 t = *reinterpret_cast<const float4 *>(Tf + r * kAp + s);
          const float4 be = *reinterpret_cast<const float4 *>(bt + s);
          f[4 * e4 + 0] = s + 0 <= r ? t.x * be.x : 0.f;
          f[4 * e4 + 1] = s + 1 <= r ? t.y * be.y : 0.f;
          f[4 * e4 + 2] = s + 2 <= r ? t.z * be.z : 0.f;
          f[4 * e4 + 3] = s + 3 <= r ? t.w * be.w : 0.f;
        }
        *reinterpret_cast<uint4 *>(img + sw128_off(r, c0 + 8 * q)) = pack8(f);
      }
    }
    __syncthreads();  // T, A and this item's scalars are dead before the buffers are refilled
  }
}

// =====================================================================================
// 2. The state chain on a CTA pair per head
// =====================================================================================

constexpr int kThreads = 512;
constexpr int kNS = 2;  // state-side stages: [K; Q], this CTA's V columns and T' of one chunk
constexpr int kNM = 3;  // state-side scalar slots
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns: the S^T bf16 copy (packed pairs, key channels 64h .. 64h + 63 in
// columns 32h ..), dS^T (fp32, lane = value column, column = key channel), two U^T
// (chunk parity; fp32, then packed in place: U and U' = U Diag(e^{b_last - b}) for tokens
// 16m .. 16m + 15 in columns 16m .. 16m + 7 and 16m + 8 .. 16m + 15), O1^T = S^T Q^T,
// O2^T = U^T P^T, and, in the same columns one after the other, the key side's
// D1 = [K; Q] K^T (lanes 64 .. 127 hold Q K^T) and W^T (lane = key channel)
constexpr uint32_t kColSC = 0, kColDS = 64, kColU = 192, kColO1 = 320, kColO2 = 384, kColD1 = 448, kColW = 448;
constexpr float kFastLimit = 100.f;             // log2 units: -b_last below this -> factorised P
constexpr uint32_t kKeyBytes = 8192u + 16384u;  // P and -W of one chunk
constexpr uint32_t kStageBytes = 32768u + 8192u + kImgBytes;
constexpr uint32_t kKeyInBytes = 32768u + kImgBytes;
// per-chunk scalars (floats). State side: e^b, e^{b_last - b}, e^{b_last}. Key side:
// the log2 prefix, e^{b - b_last}, e^{b_last - b}, e^b, the fast-path flag.
constexpr int kSsEB = 0, kSsVS = 64, kSsDec = 128, kSsBytes = 1024;
constexpr int kKsB2 = 0, kKsF = 64, kKsVS = 128, kKsEB = 192, kKsFast = 256, kKsBytes = 1280;

struct CLayout {
  uint32_t kq, v, tp, stage;  // inside a stage (the key buffer: kq and tp only)
  uint32_t key, p, wn, tpp, ost, misc, kms, bar, total;
};

// Identical in both CTAs of a pair: the exchange addresses one buffer in the
// other CTA by its own offset.
__host__ __device__ inline CLayout c_layout() {
  CLayout L;
  uint32_t o = 0;
  L.kq = o; o += 32768u;  // per 64-channel atom a: K rows at a*16384, Q rows at a*16384 + 8192
  L.v = o; o += 8192u;    // this CTA's 64 value columns
  L.tp = o; o += kImgBytes;
  L.stage = o;
  o = L.stage * kNS;
  L.key = o; o += 32768u + kImgBytes;  // the key side's own chunk: [K; Q] and T'
  L.p = o; o += 2u * 8192u;            // P of chunks owned by CTA b: buffer b
  L.wn = o; o += 2u * 16384u;          // -W, MN-major [c][r]
  L.tpp = o; o += kImgBytes;           // T'' = T' diag(e^b) of the key side's chunk
  L.ost = o; o += 8u * 2048u;          // output staging: 2 per chain warp, 32 tokens x 32 value columns
  L.misc = o; o += kNM * kSsBytes;
  L.kms = o; o += 2u * kKsBytes;
  L.bar = o; o += 512u;
  L.total = o;
  return L;
}

struct ChainParams {
  const float *g;
  const float *S0;
  float *S_final;
  const uint8_t *img;
  unsigned *status;
  int T, nchunks;
};

// One chunk's gates for tokens lane and lane + 32 (zero past T or without gates).
__device__ __forceinline__ float2 load_gates(const float *g, size_t base, int t, int T) {
  return make_float2((g && t < T) ? __ldg(g + base + t) : 0.f, (g && t + 32 < T) ? __ldg(g + base + t + 32) : 0.f);
}
// Log2 prefix of one chunk's gates (as load_gates returns them) and its total.
__device__ __forceinline__ void gate_prefix(float2 gg, int lane, float &v0, float &v1, float &bl) {
  const float g0 = gg.x, g1 = gg.y;
  v0 = g0 * kLog2e;
  v1 = g1 * kLog2e;
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
  bl = __shfl_sync(0xffffffffu, v1, 31);
}

// Bounded wait that sleeps in hardware between polls (up to `ns` per poll): for
// roles off the state chain, so that their waits take no issue slots from it.
__device__ __forceinline__ bool wait_or_abort_sleep(uint64_t *bar, uint32_t parity, bool cluster,
                                                    volatile int *abort_flag, unsigned *status) {
#pragma unroll 1
  for (uint32_t i = 0; i < kSpinLimit / 16; ++i) {
    uint32_t ok;
    if (cluster)
      asm volatile(
          "{\n\t.reg .pred p;\n\t"
          "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(ok)
          : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
          : "memory");
    else
      asm volatile(
          "{\n\t.reg .pred p;\n\t"
          "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(ok)
          : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
          : "memory");
    if (ok) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  atomicOr(status, kStatusTimeout);
  return false;
}

// Roles (512 threads): warp 2 state-side MMAs, warp 3 TMEM owner and key-side MMAs,
// warps 4, 5, 8, 9 the chain and the output epilogue (value column = lane,
// key-channel half and token half = 4,5 -> 0, 8,9 -> 1), warps 0, 1, 6, 7, 14, 15 the
// key group (P from D1 lanes 64..127 by 6, 7 (tokens 0..31) and 14, 15 (32..63), then
// T'' by 6, 7; -W by 0, 1 (channels 0..63) and 14, 15 (64..127)), warp 10 state-side
// producer, warp 11 key-side producer; warps 12, 13 have no role.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
chain_kernel(const ChainParams p, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const CLayout L = c_layout();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int bh = blockIdx.x >> 1, v_base = (int)rank * NV;
  const int T = p.T, nchunks = p.nchunks;
  const size_t gbase = (size_t)bh * T;

  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.bar);
  uint64_t *full = bars, *empty = bars + 2, *mfree = bars + 4;  // [2], [2], [3]
  uint64_t *kd_full = bars + 7, *kd_free = bars + 9;             // [2] each
  uint64_t *kt_full = bars + 11, *kt_free = bars + 12, *kms_free = bars + 13;  // 1, 1, [2]
  uint64_t *d1_full = bars + 15, *d1_free = bars + 16, *t_ready = bars + 17, *w_full = bars + 18;
  uint64_t *s_ready = bars + 19, *u_full = bars + 20, *u_ready = bars + 21, *ds_full = bars + 22;
  uint64_t *o_full = bars + 23, *o_free = bars + 24, *drain = bars + 25;  // drain [2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 30);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  auto stage = [&](int j) { return sm + (uint32_t)(j % kNS) * L.stage; };
  auto mslot = [&](int j) { return reinterpret_cast<float *>(sm + L.misc + (uint32_t)(j % kNM) * kSsBytes); };
  auto kslot = [&](int n) { return reinterpret_cast<float *>(sm + L.kms + (uint32_t)(n & 1) * kKsBytes); };
  auto pbuf = [&](int b) { return sm + L.p + (uint32_t)b * 8192u; };
  auto wnbuf = [&](int b) { return sm + L.wn + (uint32_t)b * 16384u; };

  if (warp == 3) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&full[s], 2);   // stage bytes + the producer's scalars
      mbar_init(&empty[s], 1);  // state-side MMA commit after the chunk's last MMA
    }
    for (int m = 0; m < kNM; ++m) mbar_init(&mfree[m], 4);  // the four chain warps, after the output epilogue
    for (int b = 0; b < 2; ++b) {
      mbar_init(&kd_full[b], 1);  // own: the key group's arrive; other: arm + the bulk copies' bytes
      mbar_init(&kd_free[b], 2);  // (own buffer only) both CTAs have consumed the chunk's key data
      mbar_init(&drain[b], 1);
      mbar_init(&kms_free[b], 1);
    }
    mbar_init(kt_full, 2);  // key-buffer bytes + the key producer's scalars
    mbar_init(kt_free, 1);
    mbar_init(d1_full, 1);
    mbar_init(d1_free, 1);
    mbar_init(t_ready, 1);
    mbar_init(w_full, 1);
    mbar_init(s_ready, 4);
    mbar_init(u_full, 1);
    mbar_init(u_ready, 4);
    mbar_init(ds_full, 1);
    mbar_init(o_full, 1);
    mbar_init(o_free, 4);
    *abort_flag = 0;
    // the other CTA's first chunk (chunk `peer`) arrives by bulk copy
    if ((int)peer < nchunks) mbar_arrive_expect_tx(&kd_full[peer], kKeyBytes);
    fence_mbar_init();
  }
  fence_proxy_async();
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs exist before either sends anything
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t tl = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  if (warp == 6 || warp == 7) {  // lanes 64..127 of the S^T copy: the zero rows of the 128-row MMAs
    float z[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) z[e] = 0.f;
    tmem_st32(tl + kColSC, z);
    tmem_st32(tl + kColSC + 32, z);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 10) {
    // ------------------------------------------------ state-side producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_o);
    }
    int issued = 0;
    float2 gnext = load_gates(p.g, gbase, lane, T);  // gates one chunk ahead of their use
    for (int j = 0; j < nchunks; ++j) {
      const int t0 = j * kC;
      const float2 gcur = gnext;
      if (j + 1 < nchunks) gnext = load_gates(p.g, gbase, t0 + kC + lane, T);
      int ok = 1;
      if (lane == 0) ok = wait_or_abort_sleep(&empty[j % kNS], ((j / kNS) & 1) ^ 1, false, abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      uint8_t *st = stage(j);
      uint64_t *fb = &full[j % kNS];
      if (lane == 0) {
        mbar_arrive_expect_tx(fb, kStageBytes);
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          tma_load_3d(st + L.kq + a * 16384, &tm_k, fb, 64 * a, t0, bh);
          tma_load_3d(st + L.kq + a * 16384 + 8192, &tm_q, fb, 64 * a, t0, bh);
        }
        tma_load_3d(st + L.v, &tm_v, fb, v_base, t0, bh);
        bulk_load(st + L.tp, p.img + ((size_t)bh * nchunks + j) * kImgBytes, kImgBytes, fb);
      }
      issued = j + 1;
      // the chunk's scalars once its slot is free (the copies are already in flight)
      if (lane == 0) ok = wait_or_abort_sleep(&mfree[j % kNM], ((j / kNM) & 1) ^ 1, false, abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      {
        float *ms = mslot(j);
        float v0, v1, bl;
        gate_prefix(gcur, lane, v0, v1, bl);
        ms[kSsEB + lane] = exp2f(v0);
        ms[kSsEB + lane + 32] = exp2f(v1);
        ms[kSsVS + lane] = exp2f(bl - v0);
        ms[kSsVS + lane + 32] = exp2f(bl - v1);
        if (lane == 0) ms[kSsDec] = exp2f(bl);
        __syncwarp();
      }
      if (lane == 0) mbar_arrive(fb);
    }
    if (lane == 0)  // no copy in flight when the CTA leaves
      for (int j = (issued > kNS ? issued - kNS : 0); j < issued; ++j)
        (void)mbar_wait_bounded(&full[j % kNS], (j / kNS) & 1, kSpinLimit);
  } else if (warp == 11) {
    // -------------------------------------- key-side producer (own chunks)
    int n = 0;
    float2 gnext = load_gates(p.g, gbase, (int)rank * kC + lane, T);  // gates one own chunk ahead
    for (int j = (int)rank; j < nchunks; j += 2, ++n) {
      const int t0 = j * kC;
      const float2 gcur = gnext;
      if (j + 2 < nchunks) gnext = load_gates(p.g, gbase, t0 + 2 * kC + lane, T);
      int ok = 1;
      // the key buffer once the previous own chunk's MMAs are done with it
      if (lane == 0 && n > 0) ok = wait_or_abort_sleep(kt_free, (n - 1) & 1, false, abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(kt_full, kKeyInBytes);
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          tma_load_3d(sm + L.key + a * 16384, &tm_k, kt_full, 64 * a, t0, bh);
          tma_load_3d(sm + L.key + a * 16384 + 8192, &tm_q, kt_full, 64 * a, t0, bh);
        }
        bulk_load(sm + L.key + 32768u, p.img + ((size_t)bh * nchunks + j) * kImgBytes, kImgBytes, kt_full);
        // the next own chunk's tiles and image into L2
        if (j + 2 < nchunks) {
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            tma_prefetch_3d(&tm_q, 64 * a, t0 + 2 * kC, bh);
            tma_prefetch_3d(&tm_k, 64 * a, t0 + 2 * kC, bh);
          }
          bulk_prefetch_l2(p.img + ((size_t)bh * nchunks + j + 2) * kImgBytes, kImgBytes);
        }
      }
      if (lane == 0) ok = wait_or_abort_sleep(&kms_free[n & 1], ((n >> 1) & 1) ^ 1, false, abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      {
        float *ks = kslot(n);
        float v0, v1, bl;
        gate_prefix(gcur, lane, v0, v1, bl);
        ks[kKsB2 + lane] = v0;
        ks[kKsB2 + lane + 32] = v1;
        ks[kKsF + lane] = exp2f(v0 - bl);
        ks[kKsF + lane + 32] = exp2f(v1 - bl);
        ks[kKsVS + lane] = exp2f(bl - v0);
        ks[kKsVS + lane + 32] = exp2f(bl - v1);
        ks[kKsEB + lane] = exp2f(v0);
        ks[kKsEB + lane + 32] = exp2f(v1);
        if (lane == 0) ks[kKsFast] = (-bl < kFastLimit) ? 1.f : 0.f;
        __syncwarp();
      }
      if (lane == 0) mbar_arrive(kt_full);
    }
    if (lane == 0) {  // no copy in flight when the CTA leaves
      const int nown = (nchunks - (int)rank + 1) / 2;
      if (nown > 0) (void)mbar_wait_bounded(kt_full, (nown - 1) & 1, kSpinLimit);
    }
  } else if (warp == 3) {
    // ------------------------------------ key-side MMAs of this CTA's chunks
    if (lane == 0) {
      constexpr uint32_t id_d1 = idesc_bf16_f32(128, 64, false, false);  // [K; Q] K^T
      constexpr uint32_t id_w = idesc_bf16_f32(128, 64, true, false);    // W^T = K^T T''^T
      const uint32_t a_key = smem_u32(sm + L.key), a_tpp = smem_u32(sm + L.tpp);
      const uint64_t d_key = desc_sw128(a_key, 16, 1024), d_keymn = desc_sw128(a_key, 16384, 1024),
                     d_tpp = desc_sw128(a_tpp, 16, 1024);
      int n = 0;
      for (int j = (int)rank; j < nchunks; j += 2, ++n) {
        if (!wait_or_abort_sleep(kt_full, n & 1, false, abort_flag, p.status)) break;
        // D1 and W share their columns: the previous chunk's -W epilogue has read W
        if (!wait_or_abort_sleep(d1_free, (n & 1) ^ 1, false, abort_flag, p.status)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16(tbase + kColD1, desc_add(d_key, ko), desc_add(d_key, ko), id_d1, kk > 0);
        }
        mma_commit(d1_full);
        if (!wait_or_abort_sleep(t_ready, n & 1, false, abort_flag, p.status)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tbase + kColW, desc_add(d_keymn, kk * 2048), desc_add(d_tpp, kk * 32), id_w, kk > 0);
        mma_commit(w_full);
        mma_commit(kt_free);  // the key buffer and T'' are read
      }
      mma_commit(&drain[0]);
      (void)mbar_wait_bounded(&drain[0], 0, kSpinLimit);
    }
  } else if (warp == 2) {
    // ------------------------------- state-side MMAs (every chunk): U, dS, O
    if (lane == 0) {
      constexpr uint32_t id_ut = idesc_bf16_f32(128, 64, true, false);   // V^T T'^T
      constexpr uint32_t id_us = idesc_bf16_f32(128, 64, false, true);   // S^T (-W)^T, S^T from TMEM
      constexpr uint32_t id_o1 = idesc_bf16_f32(128, 64, false, false);  // S^T Q^T
      constexpr uint32_t id_ds = idesc_bf16_f32(128, DK, false, true);   // U'^T K
      constexpr uint32_t id_o2 = idesc_bf16_f32(128, 64, false, false);  // U^T P^T
      // base descriptors of stage 0 and exchange buffer 0 (the others: address offsets)
      const uint32_t a_st0 = smem_u32(sm);
      const uint64_t d_v0 = desc_sw128(a_st0 + L.v, 8192, 1024);  // V^T, MN-major; rows 64..127: the next block
      const uint64_t d_tp0 = desc_sw128(a_st0 + L.tp, 16, 1024);  // T'^T, K-major
      const uint64_t d_q0 = desc_sw128(a_st0 + 8192, 16, 1024);   // Q^T, K-major (Q rows of each atom)
      const uint64_t d_kmn0 = desc_sw128(a_st0, 16384, 1024);     // K, MN-major (both atoms)
      const uint64_t d_wn0 = desc_sw128(smem_u32(wnbuf(0)), 8192, 1024);  // (-W)^T, MN-major
      const uint64_t d_p0 = desc_sw128(smem_u32(pbuf(0)), 16, 1024);      // P^T, K-major
      // Issue order per chunk: U2(i), O1(i), dS(i), O2(i), U1(i + 1). O1 runs while the
      // chain forms U's bf16 copies and completes before dS (the pipe is in order), so the
      // chain may rewrite the S^T copy once dS is done; O2 and the next chunk's U1 run
      // while the chain forms the next state. U is double-buffered by chunk parity.
      auto issue_u1 = [&](int i) -> bool {  // U^T(i) = V^T T'^T (value rows 64..127: the MN
        const int s2 = i % kNS;               // block after V, whatever it holds; never read)
        if (!wait_or_abort(&full[s2], (i / kNS) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint32_t so = (uint32_t)s2 * L.stage;
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16(tbase + kColU + (uint32_t)(i & 1) * 64u, desc_add(d_v0, so + kk * 2048), desc_add(d_tp0, so + kk * 32),
                   id_ut, kk > 0);
        return true;
      };
      bool ok = nchunks > 0 && issue_u1(0);
      for (int i = 0; i < nchunks && ok; ++i) {
        const int b = i & 1, s2 = i % kNS;
        const uint32_t so = (uint32_t)s2 * L.stage, t_u = tbase + kColU + (uint32_t)(i & 1) * 64u;
        const uint64_t d_q = desc_add(d_q0, so), d_kmn = desc_add(d_kmn0, so);
        const uint64_t d_wn = desc_add(d_wn0, (uint32_t)b * 16384u), d_p = desc_add(d_p0, (uint32_t)b * 8192u);
        if (!wait_or_abort_cluster(&kd_full[b], (i >> 1) & 1, abort_flag, p.status)) break;
        // U^T += S^T (-W)^T once the state copy is in
        if (!wait_or_abort(s_ready, i & 1, abort_flag, p.status)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk)
          mma_bf16_ts(t_u, tbase + kColSC + kk * 8, desc_add(d_wn, kk * 2048), id_us, 1);
        mma_commit(u_full);
        // O1^T = S^T Q^T once the previous output epilogue has read O1 and O2
        if (i > 0 && !wait_or_abort(o_free, (i - 1) & 1, abort_flag, p.status)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk)
          mma_bf16_ts(tbase + kColO1, tbase + kColSC + kk * 8, desc_add(d_q, (kk >> 2) * 16384 + (kk & 3) * 32), id_o1,
                      kk > 0);
        // dS^T = U'^T K, a fresh accumulator (the chain)
        if (!wait_or_abort(u_ready, i & 1, abort_flag, p.status)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16_ts(tbase + kColDS, t_u + kk * 16 + 8, desc_add(d_kmn, kk * 2048), id_ds, kk > 0);
        mma_commit(ds_full);
        // O2^T = U^T P^T
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_bf16_ts(tbase + kColO2, t_u + kk * 16, desc_add(d_p, kk * 32), id_o2, kk > 0);
        mma_commit(o_full);
        mma_commit(&empty[s2]);
        if (i + 1 < nchunks) ok = issue_u1(i + 1);
      }
      mma_commit(&drain[1]);
      (void)mbar_wait_bounded(&drain[1], 0, kSpinLimit);
    }
  } else if (warp == 4 || warp == 5 || warp == 8 || warp == 9) {
    // --------------------------------------------------------- the chain
    // thread (value column v, key-channel half h): S[64h + e][v_base + v] in registers
    const int v = (warp & 1) * 32 + lane, h = warp >= 8 ? 1 : 0;
    const uint32_t tv = tl;  // lanes of this warp: value columns (warp & 1) * 32 ..
    float S[64];
#pragma unroll
    for (int e = 0; e < 64; ++e) S[e] = p.S0 ? p.S0[((size_t)bh * DK + 64 * h + e) * DV + v_base + v] : 0.f;
    bool alive = true;
    float dec = 1.f;
    auto warp_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      int ok = 1;
      if (lane == 0) ok = wait_or_abort(bar, parity, abort_flag, p.status);
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    auto warp_arrive = [&](uint64_t *bar) {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar);
    };
    for (int i = 0; i <= nchunks && alive; ++i) {
      // S_{i-1} = e^{b_last} S_{i-2} + dS_{i-1}, then its bf16 copy for chunk i
      if (i > 0) {
        if (!warp_wait(ds_full, (i - 1) & 1)) { alive = false; break; }
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          float d[32];
          tmem_ld32(tv + kColDS + 64 * h + 32 * q, d);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) S[32 * q + e] = fmaf(dec, S[32 * q + e], d[e]);
        }
      }
      if (i < nchunks) {
        // (the copy's last readers, U2 and O1 of chunk i - 1, completed before its dS)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          float pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = __uint_as_float(pack_bf16(S[32 * q + 2 * e], S[32 * q + 2 * e + 1]));
          tmem_st16(tv + kColSC + 32 * h + 16 * q, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(s_ready);
      }
      if (i > 0) {
        // output epilogue of chunk c = i - 1, in the wait for this chunk's U MMA:
        // o[t][v] = e^{b_t} O1[v][t] + O2[v][t] for tokens 32h .. 32h + 31 into this warp's
        // 32 x 32 staging tile (row = token, 64 bytes), then one TMA store of the tile
        const int c = i - 1;
        if (!warp_wait(o_full, c & 1)) { alive = false; break; }
        tc_fence_after();
        uint8_t *ob = sm + L.ost + (uint32_t)(((warp & 1) + 2 * h) * 2 + (c & 1)) * 2048u;
        if (lane == 0) bulk_wait_read<1>();  // the store of chunk c - 2 has read this tile
        __syncwarp();
        const float *eb = mslot(c) + kSsEB + 32 * h;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          float a[16], bb[16];
          tmem_ld16(tv + kColO1 + 32 * h + 16 * q, a);
          tmem_ld16(tv + kColO2 + 32 * h + 16 * q, bb);
          tmem_wait_ld();
          if (q == 1) {
            tc_fence_before();
            warp_arrive(o_free);
          }
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) {
            const float4 f = *reinterpret_cast<const float4 *>(eb + 16 * q + 4 * e4);
            const float fe[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              *reinterpret_cast<__nv_bfloat16 *>(ob + (16 * q + 4 * e4 + e) * 64 + 2 * lane) =
                  __float2bfloat16_rn(fmaf(fe[e], a[4 * e4 + e], bb[4 * e4 + e]));
          }
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tm_o, ob, v_base + 32 * (warp & 1), c * kC + 32 * h, bh);
          bulk_commit();
        }
        warp_arrive(&mfree[c % kNM]);
        if (warp == 4 && lane == 0) {
          // chunk c's key data is consumed (its last MMAs completed): tell its writer,
          // and expect the writer's next chunk (c + 2) if it is the other CTA
          const int bp = c & 1;
          mbar_arrive_cluster(mapa_shared(smem_u32(&kd_free[bp]), (uint32_t)bp));
          if ((uint32_t)bp != rank && c + 2 < nchunks) mbar_arrive_expect_tx(&kd_full[bp], kKeyBytes);
        }
      }
      if (i == nchunks) break;
      // U epilogue of chunk i (tokens 32h .. 32h + 31): packed U for the output MMA and
      // packed U Diag(e^{b_last - b}) for the state update, in this thread's own columns
      // (the scalars of chunk i: its stage's barrier orders the producer's writes before
      // these reads; the stage cannot be refilled before this chunk's last MMA)
      if (!warp_wait(&full[i % kNS], (i / kNS) & 1) || !warp_wait(u_full, i & 1)) { alive = false; break; }
      tc_fence_after();
      const float *ms = mslot(i);
      dec = ms[kSsDec];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int m = 2 * h + q;
        const float *f = ms + kSsVS + 16 * m;
        const uint32_t tu = tv + kColU + (uint32_t)(i & 1) * 64u + 16 * m;
        float x[16], pk[8];
        tmem_ld16(tu, x);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 8; ++e) pk[e] = __uint_as_float(pack_bf16(x[2 * e], x[2 * e + 1]));
        tmem_st8(tu, pk);
#pragma unroll
        for (int e = 0; e < 8; ++e) pk[e] = __uint_as_float(pack_bf16(x[2 * e] * f[2 * e], x[2 * e + 1] * f[2 * e + 1]));
        tmem_st8(tu + 8, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(u_ready);
    }
    if (alive && p.S_final) {
#pragma unroll
      for (int e = 0; e < 64; ++e) p.S_final[((size_t)bh * DK + 64 * h + e) * DV + v_base + v] = S[e];
    }
    if (lane == 0) bulk_wait<0>();  // every output store has completed before the CTA leaves
  } else if (warp <= 1 || warp == 6 || warp == 7 || warp >= 14) {
    // ------------------------------------- key group: this CTA's chunks only
    constexpr int kBarKG = 1, kKG = 192;
    const int b = (int)rank;
    uint8_t *pb = pbuf(b), *wnb = wnbuf(b);
    const int lane128 = (warp & 3) * 32 + lane;  // tensor-memory lane
    const bool leader = warp == 6 && lane == 0;
    auto kg_all = [&](bool ok) -> bool {
      uint32_t r;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\t"
          "setp.ne.u32 p, %1, 0;\n\t"
          "bar.red.and.pred q, %2, %3, p;\n\t"
          "selp.u32 %0, 1, 0, q;\n\t}"
          : "=r"(r)
          : "r"((uint32_t)ok), "r"(kBarKG), "r"(kKG)
          : "memory");
      return r != 0;
    };
    int n = 0;
    for (int j = (int)rank; j < nchunks; j += 2, ++n) {
      const int nrow = min(kC, T - j * kC);
      const float *ks = kslot(n);
      bool ok = true;
      if (leader) ok = wait_or_abort_sleep(kt_full, n & 1, false, abort_flag, p.status) &&
                       wait_or_abort_sleep(d1_full, n & 1, false, abort_flag, p.status);
      if (!kg_all(ok)) break;
      tc_fence_after();
      const bool pwarp = warp >= 6;  // 6, 7, 14, 15
      const int r = lane128 - 64, s0 = warp >= 14 ? 32 : 0;
      float d[32];
      if (pwarp) {
        // P from D1 lanes 64..127 (Q K^T rows), masked and decayed: tokens s0 .. s0 + 31,
        // kept in registers until the exchange buffer is free
        const bool fast = ks[kKsFast] != 0.f;
        const float b2r = ks[kKsB2 + r], fr = ks[kKsF + r];
        float fs[32];
        load32(ks + (fast ? kKsVS : kKsB2) + s0, fs);
        tmem_ld32(tl + kColD1 + s0, d);
        tmem_wait_ld();
        if (fast) {
#pragma unroll
          for (int e = 0; e < 32; ++e) d[e] = (s0 + e <= r && r < nrow) ? d[e] * (fr * fs[e]) : 0.f;
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) d[e] = (s0 + e <= r && r < nrow) ? d[e] * exp2f(b2r - fs[e]) : 0.f;
        }
      }
      if (warp == 6 || warp == 7) {
        // T'' = T' diag(e^b) from the key buffer's image (row r, same swizzled layout)
        const uint8_t *src = sm + L.key + 32768u;
        uint8_t *dst = sm + L.tpp;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          float eb[32];
          load32(ks + kKsEB + 32 * half, eb);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t off = sw128_off(r, 32 * half + 8 * q);
            float f[8];
            unpack8(*reinterpret_cast<const uint4 *>(src + off), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] *= eb[8 * q + e];
            *reinterpret_cast<uint4 *>(dst + off) = pack8(f);
          }
        }
      }
      fence_proxy_async();
      tc_fence_before();
      kg_all(true);
      if (leader) {
        mbar_arrive(t_ready);  // P has read D1; W may take its columns
        mbar_arrive(&kms_free[n & 1]);
      }
      // P and -W go into buffer b once both CTAs consumed this CTA's previous chunk
      ok = true;
      if (leader) ok = wait_or_abort_sleep(&kd_free[b], (n & 1) ^ 1, true, abort_flag, p.status) &&
                       wait_or_abort_sleep(w_full, n & 1, false, abort_flag, p.status);
      if (!kg_all(ok)) break;
      tc_fence_after();
      if (pwarp) store_row32_bf16(pb, 8192, r, s0, d);
      if (warp <= 1 || warp >= 14) {
        // -W as the MN-major B operand [c][r] (tensor-memory lane = key channel c)
#pragma unroll 1
        for (int r0 = 0; r0 < kC; r0 += 32) {
          float x[32];
          tmem_ld32(tl + kColW + r0, x);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = -x[e];
          store_row32_bf16(wnb, 16384, lane128, r0, x);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      kg_all(true);
      if (leader) {
        mbar_arrive(d1_free);      // W is read: the next D1 may take its columns
        mbar_arrive(&kd_full[b]);  // this CTA's state side
        // the other CTA: P and -W by bulk copy, completing its kd_full[b]
        const uint32_t rbar = mapa_shared(smem_u32(&kd_full[b]), peer);
        bulk_copy_to_cluster(mapa_shared(smem_u32(pb), peer), pb, 8192u, rbar);
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

namespace {
// 3-D map over o [BH][T][DV] bf16 with a 32 x 32 box, unswizzled: the chain warps'
// staging tiles (row = token, 64 bytes).
bool make_out_map(CUtensorMap *m, const void *base, int T, int BH) {
  cuuint64_t dims[3] = {(cuuint64_t)DV, (cuuint64_t)T, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)DV * 2, (cuuint64_t)DV * 2 * T};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

size_t delta_wy_workspace_bytes(const ChunkParams &p) {
  const size_t nchunks = (size_t)(p.T + kC - 1) / kC;
  return (size_t)p.B * p.H * nchunks * kImgBytes;
}

int launch_chunk_delta_wy(const ChunkParams &p, void *workspace, cudaStream_t stream) {
  if (p.dk != DK || p.dv != DV) {
    set_error("la_chunk_fwd: the two-kernel delta-rule path takes dk = dv = 128");
    return LA_ERR_UNSUPPORTED;
  }
  if (!encode_fn()) {
    set_error("la_chunk_fwd: cuTensorMapEncodeTiled is unavailable");
    return LA_ERR_CUDA;
  }
  const int BH = p.B * p.H, nchunks = (p.T + kC - 1) / kC;
  if (BH > 65535) {
    set_error("la_chunk_fwd: the two-kernel delta-rule path takes B*H <= 65535");
    return LA_ERR_UNSUPPORTED;
  }
  const CLayout L = c_layout();
  const size_t smem = L.total + 1024;
  if (smem > 232448) {
    set_error("la_chunk_fwd: delta-rule chain kernel needs %zu bytes of shared memory", smem);
    return LA_ERR_UNSUPPORTED;
  }
  CUtensorMap mq, mk, mv, mo;
  const bool ok = make_map(&mq, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DK, p.T, BH, 64,
                           CU_TENSOR_MAP_SWIZZLE_128B) &&
                  make_map(&mk, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DK, p.T, BH, 64,
                           CU_TENSOR_MAP_SWIZZLE_128B) &&
                  make_map(&mv, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, p.T, BH, 64,
                           CU_TENSOR_MAP_SWIZZLE_128B) &&
                  make_out_map(&mo, p.o, p.T, BH);
  if (!ok) {
    set_error("la_chunk_fwd: cuTensorMapEncodeTiled rejected a tensor map");
    return LA_ERR_CUDA;
  }
  const long long items = (long long)BH * nchunks;
  WyParams wp{static_cast<const __nv_bfloat16 *>(p.k), p.g, p.beta, static_cast<uint8_t *>(workspace), p.T, nchunks,
              items};
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 148;
  const long long grid = std::min<long long>(items, (long long)kAPerSM * sms);
  cudaError_t e = cudaFuncSetAttribute(wy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWyBytes);
  if (e == cudaSuccess) {
    wy_kernel<<<(unsigned)grid, kAThreads, kWyBytes, stream>>>(wp);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_error("la_chunk_fwd: delta-rule solve kernel launch failed: %s", cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  ChainParams cp{p.g, p.S0, p.S_final, static_cast<const uint8_t *>(workspace), p.status, p.T, nchunks};
  e = cudaFuncSetAttribute(chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) {
    chain_kernel<<<(unsigned)(2 * BH), kThreads, smem, stream>>>(cp, mq, mk, mv, mo);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_error("la_chunk_fwd: delta-rule chain kernel launch failed: %s", cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  return LA_OK;
}

}  // namespace la
