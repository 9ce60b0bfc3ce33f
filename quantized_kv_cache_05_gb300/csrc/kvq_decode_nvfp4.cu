// Split-KV decode: NVFP4-cache instantiations of the partial kernel
// (head_dim 64, 128 and 256), in a translation unit of their own so that the
// library's sources compile in parallel.  The kernel is in kvq_decode.cuh.

#include "kvq_decode.cuh"

namespace kvq {
using namespace decode_impl;

cudaError_t launch_partial_nvfp4(int D, bool probq, const TensorMaps& m, const PartialArgs& a,
                                 cudaStream_t st) {
  if (D == 128) return dispatch_q<kFmtNvfp4, 128>(probq, m, a, st);
  if (D == 64) return dispatch_q<kFmtNvfp4, 64>(probq, m, a, st);
  if (D == 256) return dispatch_q<kFmtNvfp4, 256>(probq, m, a, st);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
