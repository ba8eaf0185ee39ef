// Placeholder until the tensor-core kernel is in.
#include "la_internal.h"

namespace la {
int launch_chunk_tc(const ChunkParams &, cudaStream_t) {
  set_error("la_chunk_fwd: tensor-core kernel not built");
  return LA_ERR_UNSUPPORTED;
}
}  // namespace la
