// MLA absorbed decode over an NVFP4 latent cache (placeholder until the
// kernel lands).
#include "kvq_internal.h"

namespace kvq {
cudaError_t launch_mla_partial(const CUtensorMap&, const PartialArgs&, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace kvq
