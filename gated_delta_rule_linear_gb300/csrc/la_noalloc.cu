// la_chunk_fwd_noalloc: the materialised chunk forward with its workspace in
// a fixed static device array, for callers that cannot allocate device
// memory. The kernels are the materialised variant's (la_chunk_mat.cu); only
// the origin of the workspace differs. Nothing here allocates: the array is
// part of this translation unit's device image, and its address is looked up
// on every call, so that a context that was destroyed and created again (the
// module then loads anew, possibly elsewhere) never receives a stale address.
#include <cstddef>

#include "la_internal.h"

// Workspace of every la_chunk_fwd_noalloc call on a device (shared by all
// calls: calls that overlap on the GPU race on it). Nothing in it needs to
// start at zero: the state pass writes every entry the output pass reads.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LA_NOALLOC_SCRATCH_BYTES];

namespace la {
namespace {

// Device address of the scratch array in the current context. The lookup
// does not synchronise once the module is loaded; the first call on a device
// may load this module's image, so that first call belongs before any stream
// capture.
void *scratch_address(const char *fn) {
  void *ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress((void **)&ptr, g_noalloc_scratch);
  if (e != cudaSuccess || !ptr) {
    set_error("%s: cudaGetSymbolAddress of the static scratch failed: %s", fn, cudaGetErrorString(e));
    return nullptr;
  }
  return ptr;
}

bool is_aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace la

using namespace la;

extern "C" int la_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *g,
                                    const float *beta, void *o, const float *S0, float *S_final, int B,
                                    int H, int T, int dk, int dv, int C, int mode, la_stream_t stream) {
  la::NvtxRange nvtx_range("la_chunk_fwd_noalloc");
  const char *fn = "la_chunk_fwd_noalloc";
  set_error("%s", "");
  if (!q || !k || !v || !o) {
    set_error("%s: q, k, v and o are required", fn);
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
  if (C != 0 && C != 64 && C != 128) {
    set_error("%s: C must be 0, 64 or 128 (got %d)", fn, C);
    return LA_ERR_INVALID_ARG;
  }
  const int kind = mode & 0xff;
  if ((mode & ~0xff) != 0 || kind < LA_LINEAR || kind > LA_OUTER_GATE) {
    set_error("%s: unknown mode 0x%x, or LA_F32 (bfloat16 inputs only)", fn, mode);
    return (mode & ~0xff) == LA_F32 ? LA_ERR_UNSUPPORTED : LA_ERR_INVALID_ARG;
  }
  if (kind == LA_GDN || kind == LA_KDA || kind == LA_OUTER_GATE) {
    set_error("%s: covers the unit-write modes with key-axis gates only (not LA_GDN, LA_KDA or LA_OUTER_GATE)", fn);
    return LA_ERR_UNSUPPORTED;
  }
  if (C == 128 && !c128_mode(mode)) {
    set_error("%s: C=128 covers LA_LINEAR, LA_ELU1_NORM, LA_RETNET and LA_SCALAR_GATE (not LA_GLA)", fn);
    return LA_ERR_UNSUPPORTED;
  }
  const bool needs_g = kind == LA_RETNET || kind == LA_GLA || kind == LA_SCALAR_GATE;
  if (needs_g != (g != nullptr) || beta) {
    set_error("%s: mode %d %s log-gates g and takes no beta", fn, kind, needs_g ? "needs" : "takes no");
    return LA_ERR_INVALID_ARG;
  }
  if (!is_aligned(q, 16) || !is_aligned(k, 16) || !is_aligned(v, 16) || !is_aligned(o, 16) ||
      (g && !is_aligned(g, kind == LA_GLA ? 16 : 4)) || (S0 && !is_aligned(S0, 4)) ||
      (S_final && !is_aligned(S_final, 4))) {
    set_error("%s: q, k, v, o (and g for LA_GLA) must be 16-byte aligned, S0 and S_final 4-byte", fn);
    return LA_ERR_INVALID_ARG;
  }
  ChunkParams p{q, k, v, g, beta, o, S0, S_final, B, H, T, dk, dv, C == 128 ? 128 : 64, kind, 0, nullptr};
  const size_t need = mat_workspace_bytes(p);
  if (need > (size_t)LA_NOALLOC_SCRATCH_BYTES) {
    set_error("%s: this shape needs %zu bytes of scratch (B*H*ceil(T/C)*dk*256, plus dk*4 per chunk for "
              "LA_ELU1_NORM); the static scratch holds %zu",
              fn, need, (size_t)LA_NOALLOC_SCRATCH_BYTES);
    return LA_ERR_INVALID_ARG;
  }
  p.status = status_word();
  if (!p.status) {
    set_error("%s: no CUDA device available (%s)", fn, cudaGetErrorString(cudaGetLastError()));
    return LA_ERR_CUDA;
  }
  void *ws = scratch_address(fn);
  if (!ws) return LA_ERR_CUDA;
  return launch_chunk_mat(p, ws, reinterpret_cast<cudaStream_t>(stream));
}
