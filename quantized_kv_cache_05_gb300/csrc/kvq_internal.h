// Internal launcher interface between the C-ABI layer (kvq_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <utility>

namespace kvq {

constexpr int kFmtFp8 = 1;
constexpr int kFmtNvfp4 = 2;

// Decode pipeline geometry shared by host and device code.
constexpr int kBoxTokens = 16;    // tokens per TMA box (one 16-token page) = one MMA k-tile
constexpr int kDecodeWarps = 4;   // warps of a four-warp CTA; each streams and consumes its own boxes
// Wide CTAs: six decode warps, two CTAs per SM, for the common decode (no
// FP8 probabilities, up to 8 query heads per kv head, head_dim <= 128): the
// same twelve warps per SM as three four-warp CTAs, but a third fewer split
// partials, so that the fused merge of long sequences stages them in shared
// memory with one copy.
constexpr bool kWideCta = true;
constexpr int kWideWarps = 6;
inline bool wide_cta(int D, bool probq, int G) { return kWideCta && !probq && G <= 8 && D <= 128; }
constexpr int kStages = 3;        // boxes in flight per warp of a four-warp CTA (3 measured equal or faster than 4)
constexpr int kMaxGroup = 16;     // query heads per kv head (two 8-head MMA tiles)
constexpr int kScoreCapacity = 16384;  // fp32 scores per CTA in FP8-prob mode
constexpr int kPageCache = 512;   // block-table entries of a chunk kept in shared memory
constexpr int kMaxFusedSplits = 64;  // splits the fused decode merges in one CTA

struct AppendArgs {
  int fmt, D, Hkv, ps, max_pages, batch, T, rope, num_pages;
  const uint16_t* k_new;
  const uint16_t* v_new;
  const uint16_t* kpe_new;
  const int32_t* start_pos;
  const int32_t* block_table;
  uint8_t* k_codes;
  uint8_t* v_codes;
  uint8_t* k_bscale;
  uint8_t* v_bscale;
  uint16_t* k_pe;
  float k_scale, v_scale;
  float k_recip, v_recip;     // RN(1 / scale) of the FP8 scales
  const float* k_hs;          // per-kv-head scales (replace k_scale, v_scale) or null
  const float* v_hs;
  int has_v;
};

struct PartialArgs {
  const void* q;              // [B][Hq][Dqk] bf16, or E4M3 codes when q_fp8
  const uint8_t* k_bscale;    // NVFP4 block scales (1-D bulk copies)
  const uint8_t* v_bscale;
  const uint16_t* k_pe;       // MLA rope keys
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* part_o;
  float* part_lse;
  int32_t* error_flag;
  int batch, Hq, Hkv, G, ps, max_pages, num_splits, max_kv_len, num_pages;
  int Dv;                     // value dim (the partials' row length)
  int score_floats;           // FP8-prob mode: scores one chunk needs (<= kScoreCapacity)
  float qk_scale_log2;        // sm_scale * k_scale * log2(e)
  float sm_scale;             // with per-kv-head scales: the kernel forms the above per head
  int q_fp8;                  // 1: q holds E4M3 codes (FP8 query)
  float q_scale;              // FP8 query: dequantized q = code * q_scale
  const float* q_hs;          // FP8 query: per-query-head scales (replace q_scale) or null
  const float* k_hs;          // per-kv-head scales (replace k_scale, v_scale) or null
  const float* v_hs;
  float pe_scale_log2;        // MLA rope part: sm_scale * log2(e)
  float out_mult;             // v_scale (times prob_scale with FP8 probabilities)
  float prob_scale;           // > 0: FP8 probabilities
  float prob_recip;           // RN(1 / prob_scale), used when prob_fast
  int prob_fast;              // 1: p / prob_scale by the reciprocal and one correction
  int fresh;                  // > 0: only the last `fresh` positions wait for the append
  int q_len;                  // prefill: new query tokens per request
  // fused combine (kvq_decode): arrival counters [B * Hkv] and the output
  uint32_t* counters;         // null: partials only
  void* out;
  int out_dtype;
  float out_scale;
  // MLA fused decode launched as clusters of the s splits of a request: the
  // partials merge through distributed shared memory (no counters used)
  int cluster_merge;
};

struct CombineArgs {
  const float* part_o;
  const float* part_lse;
  void* out;
  int rows, num_splits, Dv, out_dtype;
  float out_scale;
};

// Launch with programmatic stream serialization (the kernel calls
// griddep_wait() before reading its inputs).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same, as clusters of cy CTAs along the grid's y dimension.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               int cy, cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = (unsigned)cy;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t st);
cudaError_t launch_amax_bf16(const uint16_t* x, size_t n, float* out, cudaStream_t st);
cudaError_t launch_encode(int kind, const float* x, uint8_t* out, size_t n, cudaStream_t st);
// E4M3(fl32(x / s)) of bf16 x, s per tensor (recip = RN(1/s)) or per head
cudaError_t launch_quantize_fp8(const uint16_t* x, size_t n, float scale, float recip,
                                const float* head_scale, int head_len, int num_heads,
                                uint8_t* out, cudaStream_t st);
// E4M3(fl32(p / prob_scale)) per element, through the decode kernel's division
cudaError_t launch_encode_prob(const float* p, uint8_t* out, size_t n, float prob_scale,
                               float prob_recip, int prob_fast, cudaStream_t st);
// TMA descriptors of the K and V code tensors (16-row boxes).
struct TensorMaps {
  CUtensorMap k16, v16;
};

cudaError_t launch_partial(int fmt, int D, bool probq, const TensorMaps& m, const PartialArgs& a,
                           cudaStream_t st);
cudaError_t launch_partial_nvfp4(int D, bool probq, const TensorMaps& m, const PartialArgs& a,
                                 cudaStream_t st);
cudaError_t launch_mla_partial(const CUtensorMap& tcodes, const CUtensorMap& tpe,
                               const CUtensorMap& tcodes64, const CUtensorMap& tpe64,
                               const PartialArgs& a, cudaStream_t st);
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st);
cudaError_t launch_prefill(int fmt, int D, const TensorMaps& m, const PartialArgs& a,
                           cudaStream_t st);

}  // namespace kvq
