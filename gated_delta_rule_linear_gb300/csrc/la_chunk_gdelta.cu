// la_chunk_fwd_gdelta: chunkwise forward of the generalised delta rule
// ("Talk Linear Attention", section 7.1: an identity-plus-rank-one
// transition between linear-attention steps), in this library's key-major
// orientation
//
//   S_t = (I - b_t a_t^T) S_{t-1} + k_t v_t^T,   o_t = S_t^T q_t
//
// (the page writes the value-major S_{t-1}(I - a_t b_t^T) + v_t k_t^T; the
// state here is its transpose). Per chunk of C = 64 tokens with incoming
// state S and rows q_r, k_r, v_r, a_r, b_r, the retrieved values
// u_r = S_{r-1}^T a_r solve a unit lower-triangular system (the WY form of
// section 6.2 with separate retrieve and erase vectors):
//
//   U = (I + L_ab)^{-1} (A S + L_ak V),  L_ab[r,s] = a_r.b_s, L_ak[r,s] = a_r.k_s (s < r)
//   O = Q S + M(Q K^T) V - M(Q B^T) U    (M: inclusive causal mask)
//   S <- S + K^T V - B^T U
//
// This file holds the CUDA-core kernel, which runs float32 inputs (and
// bfloat16 ones when LA_GDELTA=simt; the default for bfloat16 is the
// two-phase tensor-core path of la_chunk_gdelta_wy.cu): float32 arithmetic,
// one CTA per (b, h) and 16-column tile of the value axis, the state slice in shared
// memory for the whole sequence. The four C x C products come from one
// register-tiled pass (a 4 x 4 block of (r, s) per thread, 16 shared-memory
// loads per 64 FMAs); the retrieved values U are found by forward
// substitution straight from (I + L_ab) U = R, one value column per half
// warp (the 16 lanes split the sum and reduce by shuffles), so no inverse
// is formed.
#include <cuda_bf16.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "la_internal.h"

namespace la {
namespace {

constexpr int kC = 64;
constexpr int kThreads = 256;
constexpr int kTile = 16;  // value columns per CTA

template <typename T> __device__ __forceinline__ float ld(const T *p);
template <> __device__ __forceinline__ float ld<float>(const float *p) { return __ldg(p); }
template <> __device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
// 16 bytes of input -> floats (8 bfloat16 or 4 float32)
template <typename T> __device__ __forceinline__ void unpack16(uint4 u, float *f);
template <> __device__ __forceinline__ void unpack16<float>(uint4 u, float *f) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y); f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
template <> __device__ __forceinline__ void unpack16<__nv_bfloat16>(uint4 u, float *f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
template <typename T> __device__ __forceinline__ void st(T *p, float x);
template <> __device__ __forceinline__ void st<float>(float *p, float x) { *p = x; }
template <> __device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

struct GdLayout {
  int pk, pw, pc;  // row pitches (floats): key rows dk + 1, value rows kTile + 1, C x C rows C + 1
  int q, k, a, b, v, s, r, u, p, lab, y, x, total;
};

__host__ __device__ inline GdLayout gd_layout(int dk) {
  GdLayout L;
  L.pk = dk + 1;
  L.pw = kTile + 1;
  L.pc = kC + 1;
  int o = 0;
  L.q = o; o += kC * L.pk;
  L.k = o; o += kC * L.pk;
  L.a = o; o += kC * L.pk;
  L.b = o; o += kC * L.pk;
  L.v = o; o += kC * L.pw;
  L.s = o; o += dk * L.pw;
  L.r = o; o += kC * L.pw;   // A S + L_ak V, later O
  L.u = o; o += kC * L.pw;
  L.p = o; o += kC * L.pc;   // M(Q K^T)
  L.lab = o; o += kC * L.pc; // L_ab
  L.y = o; o += kC * L.pc;   // M(Q B^T)
  L.x = o; o += kC * L.pc;   // L_ak
  L.total = o;
  return L;
}

struct GdParams {
  const void *q, *k, *v, *a, *b;
  void *o;
  const float *S0;
  float *S_final;
  int B, H, T, dk, dv;
};

template <typename Tin>
__global__ void __launch_bounds__(kThreads) chunk_gdelta_kernel(const GdParams p) {
  extern __shared__ float sm[];
  const int tid = threadIdx.x, bh = blockIdx.x, j0 = blockIdx.y * kTile;
  const int dk = p.dk, dv = p.dv, T = p.T;
  const int wv = min(kTile, dv - j0);
  const GdLayout L = gd_layout(dk);
  float *Q = sm + L.q, *K = sm + L.k, *A = sm + L.a, *Bm = sm + L.b, *V = sm + L.v, *S = sm + L.s;
  float *R = sm + L.r, *U = sm + L.u, *P = sm + L.p, *Lab = sm + L.lab, *Y = sm + L.y, *X = sm + L.x;
  const int warp = tid >> 5, lane = tid & 31;
  const size_t kbase = (size_t)bh * T * dk, vbase = (size_t)bh * T * dv;
  const Tin *q = static_cast<const Tin *>(p.q) + kbase, *k = static_cast<const Tin *>(p.k) + kbase;
  const Tin *a = static_cast<const Tin *>(p.a) + kbase, *b = static_cast<const Tin *>(p.b) + kbase;
  const Tin *v = static_cast<const Tin *>(p.v) + vbase;
  Tin *o = static_cast<Tin *>(p.o) + vbase;

  for (int i = tid; i < dk * kTile; i += kThreads) {
    const int c = i / kTile, j = i % kTile;
    S[c * L.pw + j] = (p.S0 && j < wv) ? p.S0[((size_t)bh * dk + c) * dv + j0 + j] : 0.f;
  }
  for (int t0 = 0; t0 < T; t0 += kC) {
    const int n = min(kC, T - t0);
    __syncthreads();
    // ---- stage the chunk (rows past the end are zero), 16-byte loads all in flight ----
    {
      constexpr int kVec = 16 / (int)sizeof(Tin);
      const int gpr = dk / kVec;
      for (int i = tid; i < kC * gpr; i += kThreads) {
        const int r = i / gpr, c0 = (i % gpr) * kVec;
        uint4 u[4] = {};
        if (r < n) {
          const size_t g = ((size_t)(t0 + r) * dk + c0) / kVec;
          u[0] = __ldg(reinterpret_cast<const uint4 *>(q) + g);
          u[1] = __ldg(reinterpret_cast<const uint4 *>(k) + g);
          u[2] = __ldg(reinterpret_cast<const uint4 *>(a) + g);
          u[3] = __ldg(reinterpret_cast<const uint4 *>(b) + g);
        }
        float *dst[4] = {Q, K, A, Bm};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          float f[kVec];
          unpack16<Tin>(u[m], f);
#pragma unroll
          for (int e = 0; e < kVec; ++e) dst[m][r * L.pk + c0 + e] = f[e];
        }
      }
    }
    for (int i = tid; i < kC * kTile; i += kThreads) {
      const int r = i / kTile, j = i % kTile;
      V[r * L.pw + j] = (r < n && j < wv) ? ld(v + (size_t)(t0 + r) * dv + j0 + j) : 0.f;
    }
    __syncthreads();
    // ---- M(Q K^T), L_ab, L_ak, M(Q B^T): rows tr + 16 i, columns ts + 16 j of one thread ----
    {
      const int tr = tid >> 4, ts = tid & 15;
      float qk[4][4] = {}, ab[4][4] = {}, ak[4][4] = {}, qb[4][4] = {};
      for (int c = 0; c < dk; ++c) {
        float qv[4], av[4], kv[4], bv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          qv[i] = Q[(tr + 16 * i) * L.pk + c];
          av[i] = A[(tr + 16 * i) * L.pk + c];
          kv[i] = K[(ts + 16 * i) * L.pk + c];
          bv[i] = Bm[(ts + 16 * i) * L.pk + c];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            qk[i][j] = fmaf(qv[i], kv[j], qk[i][j]);
            ab[i][j] = fmaf(av[i], bv[j], ab[i][j]);
            ak[i][j] = fmaf(av[i], kv[j], ak[i][j]);
            qb[i][j] = fmaf(qv[i], bv[j], qb[i][j]);
          }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = tr + 16 * i, sc = ts + 16 * j;
          const bool incl = sc <= r && r < n, strict = sc < r && r < n;
          P[r * L.pc + sc] = incl ? qk[i][j] : 0.f;
          Y[r * L.pc + sc] = incl ? qb[i][j] : 0.f;
          Lab[r * L.pc + sc] = strict ? ab[i][j] : 0.f;
          X[r * L.pc + sc] = strict ? ak[i][j] : 0.f;
        }
    }
    __syncthreads();
    // value column jt = tid % 16 and rows rt + 16 i of one thread (four independent sums)
    const int jt = tid & 15, rt = tid >> 4;
    // ---- R = A S + L_ak V (L_ak is zero on and above the diagonal) ----
    {
      float acc[4] = {};
      for (int c = 0; c < dk; ++c) {
        const float sv = S[c * L.pw + jt];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = fmaf(A[(rt + 16 * i) * L.pk + c], sv, acc[i]);
      }
      for (int sc = 0; sc < kC; ++sc) {
        const float vv = V[sc * L.pw + jt];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = fmaf(X[(rt + 16 * i) * L.pc + sc], vv, acc[i]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) R[(rt + 16 * i) * L.pw + jt] = acc[i];
    }
    __syncthreads();
    // ---- (I + L_ab) U = R by forward substitution: value column 2 warp + (lane >= 16) ----
    {
      const int jw = 2 * warp + (lane >> 4), l16 = lane & 15;
      for (int r = 0; r < kC; ++r) {
        float part = 0.f;
        for (int sc = l16; sc < r; sc += 16) part = fmaf(Lab[r * L.pc + sc], U[sc * L.pw + jw], part);
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (l16 == 0) U[r * L.pw + jw] = R[r * L.pw + jw] - part;
        __syncwarp();
      }
    }
    __syncthreads();
    // ---- O = Q S + M(Q K^T) V - M(Q B^T) U (into R; the masked products are zero above the diagonal) ----
    {
      float acc[4] = {};
      for (int c = 0; c < dk; ++c) {
        const float sv = S[c * L.pw + jt];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = fmaf(Q[(rt + 16 * i) * L.pk + c], sv, acc[i]);
      }
      for (int sc = 0; sc < kC; ++sc) {
        const float vv = V[sc * L.pw + jt], uu = U[sc * L.pw + jt];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[i] = fmaf(P[(rt + 16 * i) * L.pc + sc], vv, acc[i]);
          acc[i] = fmaf(-Y[(rt + 16 * i) * L.pc + sc], uu, acc[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) R[(rt + 16 * i) * L.pw + jt] = acc[i];
    }
    __syncthreads();
    for (int i = tid; i < kC * kTile; i += kThreads) {
      const int r = i / kTile, j = i % kTile;
      if (r < n && j < wv) st(o + (size_t)(t0 + r) * dv + j0 + j, R[r * L.pw + j]);
    }
    // ---- S <- S + K^T V - B^T U: key rows rt + 16 i (i < dk / 16) of column jt ----
    {
      const int nc = dk / 16;
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = (i < nc) ? S[(rt + 16 * i) * L.pw + jt] : 0.f;
      for (int sc = 0; sc < kC; ++sc) {
        const float vv = V[sc * L.pw + jt], uu = U[sc * L.pw + jt];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i < nc) {
            acc[i] = fmaf(K[sc * L.pk + rt + 16 * i], vv, acc[i]);
            acc[i] = fmaf(-Bm[sc * L.pk + rt + 16 * i], uu, acc[i]);
          }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (i < nc) S[(rt + 16 * i) * L.pw + jt] = acc[i];
    }
  }
  __syncthreads();
  if (p.S_final) {
    for (int i = tid; i < dk * kTile; i += kThreads) {
      const int c = i / kTile, j = i % kTile;
      if (j < wv) p.S_final[((size_t)bh * dk + c) * dv + j0 + j] = S[c * L.pw + j];
    }
  }
}

bool al16(const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; }

}  // namespace
}  // namespace la

using namespace la;

extern "C" int la_chunk_fwd_gdelta(const void *q, const void *k, const void *v, const void *a, const void *b,
                                   void *o, const float *S0, float *S_final, int B, int H, int T, int dk, int dv,
                                   int C, int mode, la_stream_t stream) {
  la::NvtxRange nvtx_range("la_chunk_fwd_gdelta");
  const char *fn = "la_chunk_fwd_gdelta";
  set_error("%s", "");
  if (!q || !k || !v || !a || !b || !o) {
    set_error("%s: q, k, v, a, b and o are required", fn);
    return LA_ERR_INVALID_ARG;
  }
  if (B < 1 || H < 1 || T < 1 || (long long)B * H > 0x7fffffffLL) {
    set_error("%s: B, H and T must be >= 1 (got %d, %d, %d)", fn, B, H, T);
    return LA_ERR_INVALID_ARG;
  }
  if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128)) {
    set_error("%s: dk and dv must be 64 or 128 (got %d, %d)", fn, dk, dv);
    return LA_ERR_UNSUPPORTED;
  }
  if (mode != 0 && mode != LA_F32) {
    set_error("%s: mode 0x%x: only 0 (bfloat16 inputs) or LA_F32 (float32 inputs)", fn, mode);
    return LA_ERR_INVALID_ARG;
  }
  if (C != 0 && C != 64) {
    set_error("%s: chunk length C=%d is not implemented in this build (use 0 or 64)", fn, C);
    return LA_ERR_UNSUPPORTED;
  }
  const void *p16[] = {q, k, v, a, b, o};
  for (const void *ptr : p16)
    if (!al16(ptr)) {
      set_error("%s: q, k, v, a, b and o must be 16-byte aligned", fn);
      return LA_ERR_INVALID_ARG;
    }
  if ((S0 && !al16(S0)) || (S_final && !al16(S_final))) {
    set_error("%s: S0 and S_final must be 16-byte aligned", fn);
    return LA_ERR_INVALID_ARG;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const char *env = getenv("LA_GDELTA");
  if (mode == 0 && !(env && strcmp(env, "simt") == 0)) {
    // bfloat16: the two-phase path on the tensor cores (per-chunk key side, then the
    // state chain), workspace from the library's pool on the caller's stream
    const GdeltaArgs x{q, k, v, a, b, o, S0, S_final, B, H, T, dk, dv};
    if ((long long)B * H > 65535) {
      set_error("%s: B*H must be <= 65535 for bfloat16 inputs (got %lld)", fn, (long long)B * H);
      return LA_ERR_UNSUPPORTED;
    }
    const size_t bytes = gdelta_wy_workspace_bytes(B * H, T, dk);
    cudaMemPool_t pool = library_pool();
    if (!pool) {
      set_error("%s: could not create the workspace pool: %s", fn, cudaGetErrorString(cudaGetLastError()));
      return LA_ERR_CUDA;
    }
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, bytes, pool, s);
    if (e != cudaSuccess) {
      set_error("%s: workspace allocation of %zu bytes failed: %s", fn, bytes, cudaGetErrorString(e));
      return LA_ERR_CUDA;
    }
    const int rc = launch_gdelta_wy(x, ws, s);
    e = cudaFreeAsync(ws, s);
    if (rc == LA_OK && e != cudaSuccess) {
      set_error("%s: workspace release failed: %s", fn, cudaGetErrorString(e));
      return LA_ERR_CUDA;
    }
    return rc;
  }
  const GdParams p{q, k, v, a, b, o, S0, S_final, B, H, T, dk, dv};
  const GdLayout L = gd_layout(dk);
  const size_t smem = sizeof(float) * (size_t)L.total;
  const dim3 grid((unsigned)(B * H), (unsigned)((dv + kTile - 1) / kTile));
  cudaError_t e;
  if (mode == LA_F32) {
    e = cudaFuncSetAttribute(chunk_gdelta_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) chunk_gdelta_kernel<float><<<grid, kThreads, smem, s>>>(p);
  } else {
    e = cudaFuncSetAttribute(chunk_gdelta_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e == cudaSuccess) chunk_gdelta_kernel<__nv_bfloat16><<<grid, kThreads, smem, s>>>(p);
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("%s: launch failed: %s", fn, cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  return LA_OK;
}
