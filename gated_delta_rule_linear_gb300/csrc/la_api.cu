// Host side of the C ABI declared in include/la.h: argument validation, the
// per-shape choice of kernel, the thread-local error message and the device
// status word. Every step of the computation runs in the CUDA kernels; this
// file only checks arguments and launches them on the caller's stream.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "la_internal.h"

namespace la {

namespace {
thread_local char g_err[512] = "";

// Written by kernels only when a bounded device-side wait gives up.
__device__ unsigned g_status_word;

constexpr int kMaxDevices = 64;

// Stream-ordered pool for the materialised variant's workspace, one per
// device, owned by the library. It keeps freed memory for the next call
// (release threshold = max) instead of unmapping it at every synchronisation.
cudaMemPool_t g_pool[kMaxDevices] = {};
std::mutex g_pool_mu;

cudaMemPool_t workspace_pool() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_pool_mu);
  if (!g_pool[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
    uint64_t keep = ~0ull;
    if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
      cudaMemPoolDestroy(pool);
      return nullptr;
    }
    g_pool[dev] = pool;
  }
  return g_pool[dev];
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
}  // namespace

cudaMemPool_t library_pool() { return workspace_pool(); }

void set_error(const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

// Looked up in the current context on every call (no synchronisation once
// the module is loaded): a cached address would go stale if the context were
// destroyed and created again.
unsigned *status_word() {
  void *ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return nullptr;
  return static_cast<unsigned *>(ptr);
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

// Host-side kernel choice. float32 inputs go to the CUDA-core kernel. bf16
// inputs go to the fused (non-materialised) tensor-core kernel, which runs
// one CTA per head, or, for the unit-write modes when B*H is at most half the
// SM count (the fused grid would leave most of the GPU idle) and the sequence
// spans at least 8 chunks, to the materialised two-phase variant, whose
// output pass uses every SM. LA_VARIANT (auto | tc | nonmat | mat | simt)
// overrides the choice for measurement sweeps.
int select_variant(const ChunkParams &p, int *chunk_out) {
  const char *env = getenv("LA_VARIANT");
  int want = -1;
  if (env && (strcmp(env, "tc") == 0 || strcmp(env, "nonmat") == 0)) want = kVariantTc;
  if (env && strcmp(env, "mat") == 0) want = kVariantMat;
  if (env && strcmp(env, "simt") == 0) want = kVariantSimt;
  if (p.C == 128) {  // the 128-token output pass of the materialised variant (modes checked by the caller)
    if (want == kVariantTc || want == kVariantSimt) {
      set_error("la_chunk_fwd: C=128 runs on the materialised variant only");
      return -1;
    }
    *chunk_out = 128;
    return kVariantMat;
  }
  *chunk_out = 64;
  if (p.f32 && (p.kind == kKda || p.kind == kOuter)) {
    set_error("la_chunk_fwd: LA_KDA and LA_OUTER_GATE take bfloat16 inputs only");
    return -1;
  }
  if (p.f32) return (want == kVariantTc || want == kVariantMat) ? -2 : kVariantSimt;
  if (p.kind == kKda) {
    // the two-phase path (every chunk's key side in parallel, then the state chain per
    // head and 64 value columns; la_chunk_kda_wy.cu), measured faster on GB300 than the
    // fused sequential-phase kernel, which LA_VARIANT=tc or LA_KDA=tc selects
    if (want == kVariantMat || want == kVariantSimt) {
      set_error("la_chunk_fwd: LA_KDA runs on its two-phase path or the fused tensor-core kernel");
      return -1;
    }
    const char *kd = getenv("LA_KDA");
    return (want == kVariantTc || (kd && strcmp(kd, "tc") == 0)) ? kVariantTc : kVariantKdaWy;
  }
  if ((want == kVariantMat || want == kVariantSimt) && p.kind == kOuter) {
    set_error("la_chunk_fwd: LA_OUTER_GATE runs on the pipelined tensor-core kernel only");
    return -1;
  }
  if (p.kind == kGdn) {
    // the delta rule: the fused kernels (a CTA pair per head while 2*B*H fits the GPU,
    // else one CTA per head; la_chunk_tc.cu), measured faster on GB300 than the
    // two-phase path (the solve for every chunk in parallel into T' images, then the
    // state chain on a CTA pair: dk = dv = 128), which LA_DELTA=wy or LA_VARIANT=mat
    // selects
    const bool big = p.dk == 128 && p.dv == 128;
    const char *d = getenv("LA_DELTA");
    const bool two_phase = (d && strcmp(d, "wy") == 0) || want == kVariantMat;
    if (two_phase && !big) {
      set_error("la_chunk_fwd: the two-phase delta-rule path takes dk = dv = 128");
      return -1;
    }
    if (want == kVariantSimt) return kVariantSimt;
    return two_phase ? kVariantDeltaWy : kVariantTc;
  }
  if (want >= 0) return want;
  // Materialised when its DRAM time stays below the fused kernel's serial time:
  // the fused kernel takes ~T/64 chunk periods whatever B*H (up to one CTA per SM);
  // the materialised one moves ~2.4x the bytes at C = 64 (GLA ~3.5 KB per
  // token-head, the others ~2.5 KB, measured by ncu) through a fully parallel
  // output pass. The measured crossover lies between B*H = 64 and 128 for RetNet,
  // the scalar decay and plain linear attention (SMs / 2), and below 64 for GLA,
  // whose fused chunk is the longest and whose materialised pass moves the most
  // (SMs / 4). elu+1's fused chunk is slow (~5 us) and its materialised pass at
  // C = 128 was faster at every B*H measured (up to 256): materialised from 8
  // chunks on.
  // Chunk length of the materialised pass: 128 (one state image per 128 tokens,
  // ~20% fewer DRAM bytes, measured faster or equal) for the modes without
  // per-channel gates, except RetNet and the scalar decay below 2048 tokens where
  // the two measured within a few percent either way; 64 for GLA.
  const long long BH = (long long)p.B * p.H, sms = sm_count();
  const bool small = p.kind == kGla ? 4 * BH <= sms : p.kind == kElu1 ? true : 2 * BH <= sms;
  if (p.kind != kGdn && p.kind != kOuter && p.T >= 8 * 64 && small) {
    if (p.C == 0 && p.kind != kGla && (p.kind == kLinear || p.kind == kElu1 || p.T >= 2048)) *chunk_out = 128;
    return kVariantMat;
  }
  return kVariantTc;
}

}  // namespace la

using namespace la;

extern "C" {

const char *la_last_error(void) { return g_err; }

int la_version(void) { return 1 * 10000 + 0 * 100 + 0; }

int la_stream_status(la_stream_t stream) {
  g_err[0] = '\0';
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    set_error("la_stream_status: stream synchronisation failed: %s", cudaGetErrorString(e));
    return LA_ERR_CUDA;
  }
  unsigned *w = status_word();
  if (!w) {
    set_error("la_stream_status: device status word unavailable");
    return LA_ERR_CUDA;
  }
  unsigned v = 0;
  if (cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(w, 0, sizeof(v)) != cudaSuccess) {
    set_error("la_stream_status: reading the status word failed");
    return LA_ERR_CUDA;
  }
  if (v & kStatusTimeout) {
    set_error("a kernel gave up on a bounded device-side wait (status 0x%x)", v);
    return LA_ERR_TIMEOUT;
  }
  return LA_OK;
}

static int check_mode(int mode, const float *g, const float *beta, const char *fn, bool allow_nc = false) {
  const int kind = mode & 0xff;
  const int flags = allow_nc ? (LA_F32 | LA_NONCAUSAL) : LA_F32;
  if ((mode & ~(0xff | flags)) != 0 || kind < LA_LINEAR || kind > LA_OUTER_GATE) {
    set_error("%s: unknown mode 0x%x", fn, mode);
    return LA_ERR_INVALID_ARG;
  }
  if ((mode & LA_NONCAUSAL) && kind != LA_LINEAR && kind != LA_ELU1_NORM) {
    set_error("%s: LA_NONCAUSAL goes with LA_LINEAR or LA_ELU1_NORM only", fn);
    return LA_ERR_INVALID_ARG;
  }
  const bool needs_g = kind == LA_RETNET || kind == LA_GLA || kind == LA_SCALAR_GATE || kind == LA_KDA ||
                       kind == LA_OUTER_GATE;
  const bool takes_g = needs_g || kind == LA_GDN;
  if (needs_g && !g) {
    set_error("%s: mode %d needs log-gates g", fn, kind);
    return LA_ERR_INVALID_ARG;
  }
  if (!takes_g && g) {
    set_error("%s: mode %d takes no gates (g must be NULL)", fn, kind);
    return LA_ERR_INVALID_ARG;
  }
  if (kind == LA_OUTER_GATE && !beta) {
    set_error("%s: LA_OUTER_GATE needs the value-axis log-gates in beta", fn);
    return LA_ERR_INVALID_ARG;
  }
  if (kind != LA_GDN && kind != LA_KDA && kind != LA_OUTER_GATE && beta) {
    set_error("%s: beta is only used by LA_GDN, LA_KDA and LA_OUTER_GATE (must be NULL for mode %d)", fn, kind);
    return LA_ERR_INVALID_ARG;
  }
  return LA_OK;
}

int la_chunk_fwd(const void *q, const void *k, const void *v, const float *g, const float *beta,
                 void *o, const float *S0, float *S_final, int B, int H, int T, int dk, int dv,
                 int C, int mode, la_stream_t stream) {
  la::NvtxRange nvtx_range("la_chunk_fwd");
  g_err[0] = '\0';
  const char *fn = "la_chunk_fwd";
  if (!q || !k || !v || !o) {
    set_error("%s: q, k, v and o are required", fn);
    return LA_ERR_INVALID_ARG;
  }
  if (B < 1 || H < 1 || T < 1) {
    set_error("%s: B, H and T must be >= 1 (got %d, %d, %d)", fn, B, H, T);
    return LA_ERR_INVALID_ARG;
  }
  if ((long long)B * H > 0x7fffffffLL) {
    set_error("%s: B*H too large", fn);
    return LA_ERR_INVALID_ARG;
  }
  if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128)) {
    set_error("%s: dk and dv must be 64 or 128 (got %d, %d)", fn, dk, dv);
    return LA_ERR_UNSUPPORTED;
  }
  if (C != 0 && C != 64 && C != 128) {
    set_error("%s: C must be 0, 64 or 128 (got %d)", fn, C);
    return LA_ERR_INVALID_ARG;
  }
  int rc = check_mode(mode, g, beta, fn, true);
  if (rc) return rc;
  const int kind = mode & 0xff;
  if (C == 128 && !c128_mode(mode)) {
    set_error("%s: C=128 is implemented for the materialised variant of LA_LINEAR, LA_ELU1_NORM, LA_RETNET "
              "and LA_SCALAR_GATE (bfloat16, causal)", fn);
    return LA_ERR_UNSUPPORTED;
  }
  if ((mode & LA_NONCAUSAL) && (mode & LA_F32)) {
    set_error("%s: LA_NONCAUSAL takes bfloat16 inputs only", fn);
    return LA_ERR_UNSUPPORTED;
  }
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16)) {
    set_error("%s: q, k, v and o must be 16-byte aligned", fn);
    return LA_ERR_INVALID_ARG;
  }
  const bool chan = kind == LA_GLA || kind == LA_KDA || kind == LA_OUTER_GATE;
  if ((g && !aligned(g, chan ? 16 : 4)) || (beta && !aligned(beta, kind == LA_OUTER_GATE ? 16 : 4)) ||
      (S0 && !aligned(S0, 4)) || (S_final && !aligned(S_final, 4))) {
    set_error("%s: g (16 bytes for LA_GLA, LA_KDA, LA_OUTER_GATE), beta (16 bytes for LA_OUTER_GATE), S0 and "
              "S_final must be aligned", fn);
    return LA_ERR_INVALID_ARG;
  }

  ChunkParams p{q, k, v, g, beta, o, S0, S_final, B, H, T, dk, dv, C, kind,
                (mode & LA_F32) ? 1 : 0, status_word()};
  if (!p.status) {
    set_error("%s: no CUDA device available (%s)", fn, cudaGetErrorString(cudaGetLastError()));
    return LA_ERR_CUDA;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (mode & LA_NONCAUSAL) {
    p.C = 64;
    void *ws = nullptr;
    const size_t bytes = nc_workspace_bytes(p);
    cudaMemPool_t pool = workspace_pool();
    if (!pool) {
      set_error("%s: could not create the workspace pool: %s", fn, cudaGetErrorString(cudaGetLastError()));
      return LA_ERR_CUDA;
    }
    cudaError_t e = cudaMallocFromPoolAsync(&ws, bytes, pool, s);
    if (e != cudaSuccess) {
      set_error("%s: workspace allocation of %zu bytes failed: %s", fn, bytes, cudaGetErrorString(e));
      return LA_ERR_CUDA;
    }
    rc = launch_chunk_noncausal(p, ws, s);
    e = cudaFreeAsync(ws, s);
    if (rc == LA_OK && e != cudaSuccess) {
      set_error("%s: workspace release failed: %s", fn, cudaGetErrorString(e));
      return LA_ERR_CUDA;
    }
    return rc;
  }
  int chunk = 64;
  const int variant = select_variant(p, &chunk);
  if (variant == -2) {
    set_error("%s: the tensor-core kernel takes bfloat16 inputs only", fn);
    return LA_ERR_UNSUPPORTED;
  }
  if (variant < 0) return LA_ERR_UNSUPPORTED;
  p.C = chunk;
  if (variant == kVariantMat) {
    // stream-ordered workspace: allocated and released on the caller's stream
    void *ws = nullptr;
    // linear and elu+1: the parallel state pass while its float32 chunk partials take
    // at most 2 GiB (LA_MAT_STATE=serial keeps the serial one)
    const char *ms = getenv("LA_MAT_STATE");
    const size_t sb = mat_scan_bytes(p);
    const bool scan = sb > 0 && sb <= (size_t(2) << 30) && !(ms && strcmp(ms, "serial") == 0);
    const size_t bytes = mat_workspace_bytes(p) + (scan ? mat_scan_bytes(p) : 0);
    cudaMemPool_t pool = workspace_pool();
    if (!pool) {
      set_error("%s: could not create the workspace pool: %s", fn, cudaGetErrorString(cudaGetLastError()));
      return LA_ERR_CUDA;
    }
    cudaError_t e = cudaMallocFromPoolAsync(&ws, bytes, pool, s);
    if (e != cudaSuccess) {
      set_error("%s: workspace allocation of %zu bytes failed: %s", fn, bytes, cudaGetErrorString(e));
      return LA_ERR_CUDA;
    }
    rc = launch_chunk_mat(p, ws, s, scan);
    e = cudaFreeAsync(ws, s);
    if (rc == LA_OK && e != cudaSuccess) {
      set_error("%s: workspace release failed: %s", fn, cudaGetErrorString(e));
      return LA_ERR_CUDA;
    }
    return rc;
  }
  if (variant == kVariantDeltaWy || variant == kVariantKdaWy) {
    // stream-ordered workspace for the per-chunk key-side images, from the library's pool
    void *ws = nullptr;
    const size_t bytes = variant == kVariantKdaWy ? kda_wy_workspace_bytes(p) : delta_wy_workspace_bytes(p);
    cudaMemPool_t pool = workspace_pool();
    if (!pool) {
      set_error("%s: could not create the workspace pool: %s", fn, cudaGetErrorString(cudaGetLastError()));
      return LA_ERR_CUDA;
    }
    cudaError_t e = cudaMallocFromPoolAsync(&ws, bytes, pool, s);
    if (e != cudaSuccess) {
      set_error("%s: workspace allocation of %zu bytes failed: %s", fn, bytes, cudaGetErrorString(e));
      return LA_ERR_CUDA;
    }
    rc = variant == kVariantKdaWy ? launch_kda_wy(p, ws, s) : launch_chunk_delta_wy(p, ws, s);
    e = cudaFreeAsync(ws, s);
    if (rc == LA_OK && e != cudaSuccess) {
      set_error("%s: workspace release failed: %s", fn, cudaGetErrorString(e));
      return LA_ERR_CUDA;
    }
    return rc;
  }
  return variant == kVariantTc ? launch_chunk_tc(p, s) : launch_chunk_simt(p, s);
}

int la_recurrent_step(const void *q, const void *k, const void *v, const float *g,
                      const float *beta, void *o, float *S, int B, int H, int dk, int dv, int mode,
                      la_stream_t stream) {
  la::NvtxRange nvtx_range("la_recurrent_step");
  g_err[0] = '\0';
  const char *fn = "la_recurrent_step";
  if (!q || !k || !v || !o || !S) {
    set_error("%s: q, k, v, o and S are required", fn);
    return LA_ERR_INVALID_ARG;
  }
  if (B < 1 || H < 1 || (long long)B * H > 0x7fffffffLL) {
    set_error("%s: B and H must be >= 1 (got %d, %d)", fn, B, H);
    return LA_ERR_INVALID_ARG;
  }
  if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128)) {
    set_error("%s: dk and dv must be 64 or 128 (got %d, %d)", fn, dk, dv);
    return LA_ERR_UNSUPPORTED;
  }
  int rc = check_mode(mode, g, beta, fn);
  if (rc) return rc;
  const size_t el = (mode & LA_F32) ? 4 : 2;
  if (!aligned(q, el) || !aligned(k, el) || !aligned(v, el) || !aligned(o, el) ||
      !aligned(S, 4) || (g && !aligned(g, 4)) || (beta && !aligned(beta, 4))) {
    set_error("%s: pointers must be aligned to their element size", fn);
    return LA_ERR_INVALID_ARG;
  }
  StepParams p{q, k, v, g, beta, o, S, B, H, dk, dv, mode & 0xff, (mode & LA_F32) ? 1 : 0};
  return launch_step(p, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
