// Internal declarations shared by the host entry points and the kernels of
// libla.so. Nothing here is part of the public ABI (include/la.h is).
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdint>

#include "../../include/la.h"

namespace la {

enum Kind : int {
  kLinear = LA_LINEAR,
  kElu1 = LA_ELU1_NORM,
  kRetnet = LA_RETNET,
  kGla = LA_GLA,
  kScalar = LA_SCALAR_GATE,
  kGdn = LA_GDN,
  kKda = LA_KDA,
  kOuter = LA_OUTER_GATE,
};

// Bits of the device status word (one per device, see la_status.cu).
enum StatusBits : unsigned {
  kStatusTimeout = 1u,
};

// Arguments of the generalised delta rule's forward (la_chunk_fwd_gdelta).
struct GdeltaArgs {
  const void *q, *k, *v, *a, *b;
  void *o;
  const float *S0;
  float *S_final;
  int B, H, T, dk, dv;
};
// The two-phase bf16 path: per-chunk key-side matrices into `workspace`
// (gdelta_wy_workspace_bytes), then the state chain (la_chunk_gdelta_wy.cu).
size_t gdelta_wy_workspace_bytes(int BH, int T, int dk);
int launch_gdelta_wy(const GdeltaArgs &x, void *workspace, cudaStream_t stream);

// Whether a mode word may request the 128-token chunk: the materialised
// variant's output pass for the modes without per-channel gates, bfloat16,
// causal (no flag bits).
inline bool c128_mode(int mode) {
  const int kind = mode & 0xff;
  return (mode & ~0xff) == 0 &&
         (kind == LA_LINEAR || kind == LA_ELU1_NORM || kind == LA_RETNET || kind == LA_SCALAR_GATE);
}

// Everything a chunk-forward kernel needs, by value.
struct ChunkParams {
  const void *q, *k, *v;
  const float *g, *beta;
  void *o;
  const float *S0;
  float *S_final;
  int B, H, T, dk, dv, C;
  int kind;
  int f32;          // 1: q/k/v/o are float32, 0: bfloat16
  unsigned *status; // device status word
  int rev;          // 1: run on the time-reversed sequence (row t of q, k, v, o is token T-1-t);
                    // the unit-write kernels (linear and RetNet) and the float32 kernel only
};

struct StepParams {
  const void *q, *k, *v;
  const float *g, *beta;
  void *o;
  float *S;
  int B, H, dk, dv;
  int kind;
  int f32;
};

// The library's stream-ordered workspace pool on the current device (keeps
// freed memory for the next call), or null if it cannot be created.
cudaMemPool_t library_pool();

// An NVTX range around an entry point's host work and launches (header-only
// NVTX; a no-op unless a profiler attaches to the process).
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange &) = delete;
  NvtxRange &operator=(const NvtxRange &) = delete;
};

// Thread-local error message for la_last_error().
void set_error(const char *fmt, ...);

// Device status word of the current device (a __device__ variable).
unsigned *status_word();
// multiprocessors of the current device (0 when the query fails)
int sm_count();

// Launchers: return LA_OK or an LA_ERR_* code (message already set).
int launch_chunk_simt(const ChunkParams &p, cudaStream_t stream);
int launch_chunk_tc(const ChunkParams &p, cudaStream_t stream);
int launch_chunk_ws(const ChunkParams &p, cudaStream_t stream);
int launch_chunk_delta(const ChunkParams &p, cudaStream_t stream);
int launch_chunk_delta_pair(const ChunkParams &p, cudaStream_t stream);
int launch_step(const StepParams &p, cudaStream_t stream);
// Materialised (two-phase) variant: chunk-state pass then a parallel output
// pass, through a caller-provided workspace of mat_workspace_bytes(p) bytes;
// with scan set (linear and elu+1 only; the workspace then has
// mat_scan_bytes(p) more) the state pass runs as every chunk's partial at once
// plus a prefix scan instead of one serial walk per head.
size_t mat_workspace_bytes(const ChunkParams &p);
size_t mat_scan_bytes(const ChunkParams &p);
int launch_chunk_mat(const ChunkParams &p, void *workspace, cudaStream_t stream, bool scan = false);
// Non-causal forward (LA_NONCAUSAL; linear and elu+1, bf16): split-T state
// reduction, finalize, parallel output pass, through a caller-provided
// workspace of nc_workspace_bytes(p) bytes.
size_t nc_workspace_bytes(const ChunkParams &p);
int launch_chunk_noncausal(const ChunkParams &p, void *workspace, cudaStream_t stream);

// Gated delta rule (dk = dv = 128, bf16) in two kernels: the triangular solve for
// every (head, chunk) into a workspace of delta_wy_workspace_bytes(p) bytes (one
// bf16 T' image per chunk), then the state chain on a CTA pair per head.
size_t delta_wy_workspace_bytes(const ChunkParams &p);
// Kimi Delta Attention's two-phase path (la_chunk_kda_wy.cu): the key side of
// every chunk into `workspace` (kda_wy_workspace_bytes), then the state chain.
size_t kda_wy_workspace_bytes(const ChunkParams &p);
int launch_kda_wy(const ChunkParams &p, void *workspace, cudaStream_t stream);
int launch_chunk_delta_wy(const ChunkParams &p, void *workspace, cudaStream_t stream);

// Which chunk-forward kernel a shape goes to (host-side selection).
enum Variant : int { kVariantSimt = 0, kVariantTc = 1, kVariantMat = 2, kVariantDeltaWy = 3, kVariantKdaWy = 4 };
int select_variant(const ChunkParams &p, int *chunk_out);

}  // namespace la
