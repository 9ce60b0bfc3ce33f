// Split-KV decode: FP8-cache instantiations of the partial kernel, the
// combine kernel and the format dispatch (sm_103a).  The kernel itself is in
// kvq_decode.cuh.

#include "kvq_decode.cuh"

namespace kvq {
using namespace decode_impl;
namespace {

// ---------------------------------------------------------------------------
// Combine: one CTA merges kCombineRows consecutive (request, query head) rows.
// ---------------------------------------------------------------------------
constexpr int kCombineRows = 4;

__global__ void __launch_bounds__(128) combine_kernel(const CombineArgs a) {
  __shared__ float w[kCombineRows * kMaxFusedSplits];
  __shared__ float winv[kCombineRows];
  griddep_wait();
  const size_t row0 = (size_t)blockIdx.x * kCombineRows;
  const int rows = (int)min((size_t)kCombineRows, (size_t)a.rows - row0);
  merge_rows(a.part_o, a.part_lse, row0, rows, a.num_splits, a.Dv, w, winv, a.out, a.out_dtype,
             a.out_scale);
}

}  // namespace

cudaError_t launch_partial(int fmt, int D, bool probq, const TensorMaps& m, const PartialArgs& a,
                           cudaStream_t st) {
  if (fmt == kFmtFp8 && D == 128) return dispatch_q<kFmtFp8, 128>(probq, m, a, st);
  if (fmt == kFmtFp8 && D == 64) return dispatch_q<kFmtFp8, 64>(probq, m, a, st);
  if (fmt == kFmtNvfp4) return launch_partial_nvfp4(D, probq, m, a, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st) {
  if (a.num_splits > kMaxFusedSplits) return cudaErrorInvalidValue;
  return launch_pdl(combine_kernel, dim3((a.rows + kCombineRows - 1) / kCombineRows), dim3(128),
                    0, st, a);
}

}  // namespace kvq
