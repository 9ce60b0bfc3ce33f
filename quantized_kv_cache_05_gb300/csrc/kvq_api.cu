// The extern "C" entry points of include/kvq.h: argument validation (before
// any launch), TMA descriptor setup and kernel dispatch.  Host code only.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cudaTypedefs.h>

#include "kvq.h"
#include "kvq_internal.h"

using namespace kvq;

namespace {

bool finite_pos(float x) { return std::isfinite(x) && x > 0.f; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  // The CUDA driver API entry point is looked up once per process.
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D byte view [rows][row_bytes] of a cache tensor, box_rows-row boxes, with the
// widest hardware swizzle the row allows.
bool make_row_map(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows,
                  uint32_t box_rows = kBoxTokens) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)row_bytes, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUtensorMapSwizzle sw = row_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                          : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                            : CU_TENSOR_MAP_SWIZZLE_NONE;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D byte view [rows][n_slices][slice_bytes] of a row-major tensor whose rows
// are n_slices * slice_bytes wide; boxes of one slice x box_rows rows.
bool make_slice_map(CUtensorMap* m, const void* base, uint64_t slice_bytes, uint64_t n_slices,
                    uint64_t rows, CUtensorMapSwizzle sw, uint32_t box_rows = kBoxTokens) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {slice_bytes, n_slices, rows};
  cuuint64_t strides[2] = {slice_bytes, slice_bytes * n_slices};
  cuuint32_t box[3] = {(cuuint32_t)slice_bytes, 1, box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool is_mla(const kvq_cache* c) { return c->rope_dim > 0; }

// Checks shared by append and decode.
kvq_status check_cache(const kvq_cache* c) {
  if (!c) return KVQ_ERR_INVALID;
  if (c->fmt != KVQ_FP8_E4M3 && c->fmt != KVQ_NVFP4) return KVQ_ERR_INVALID;
  if (c->num_pages < 1 || c->num_kv_heads < 1 || c->max_pages_per_seq < 1) return KVQ_ERR_INVALID;
  if (c->page_size < 16 || c->page_size % 16 != 0) return KVQ_ERR_INVALID;
  if (c->head_dim < 16 || c->head_dim % 16 != 0 || c->head_dim > 1024) return KVQ_ERR_INVALID;
  if ((long long)c->num_pages * c->num_kv_heads * c->page_size >= (1LL << 31))
    return KVQ_ERR_UNSUPPORTED;
  if (!c->block_table || !c->k_codes || !aligned16(c->k_codes)) return KVQ_ERR_INVALID;
  if (!c->k_head_scale && !finite_pos(c->k_scale)) return KVQ_ERR_INVALID;
  if (c->fmt == KVQ_NVFP4 && (!c->k_bscale || !aligned16(c->k_bscale))) return KVQ_ERR_INVALID;
  if (is_mla(c)) {
    if (c->rope_dim % 8 != 0 || !c->k_pe || !aligned16(c->k_pe)) return KVQ_ERR_INVALID;
    if (c->v_codes || !c->v_is_k_latent) return KVQ_ERR_INVALID;
    if (c->k_head_scale || c->v_head_scale) return KVQ_ERR_INVALID;
    if (c->num_kv_heads != 1) return KVQ_ERR_INVALID;
    if (c->fmt != KVQ_NVFP4) return KVQ_ERR_UNSUPPORTED;
  } else {
    if (c->rope_dim != 0 || c->k_pe || c->v_is_k_latent) return KVQ_ERR_INVALID;
    if (!c->v_codes || !aligned16(c->v_codes)) return KVQ_ERR_INVALID;
    if (!c->v_head_scale && !finite_pos(c->v_scale)) return KVQ_ERR_INVALID;
    if (c->fmt == KVQ_NVFP4 && (!c->v_bscale || !aligned16(c->v_bscale))) return KVQ_ERR_INVALID;
  }
  return KVQ_OK;
}

kvq_status check_params(const kvq_decode_params* p) {
  if (!p) return KVQ_ERR_INVALID;
  if (p->batch < 0 || p->num_q_heads < 1 || p->qk_dim < 1 || p->v_dim < 1) return KVQ_ERR_INVALID;
  if (p->num_splits < 1) return KVQ_ERR_INVALID;
  if (p->num_splits > kMaxFusedSplits) return KVQ_ERR_UNSUPPORTED;
  if (p->max_kv_len < 0) return KVQ_ERR_INVALID;
  if (p->batch > 0 && !p->seq_lens) return KVQ_ERR_INVALID;
  if (!finite_pos(p->sm_scale)) return KVQ_ERR_INVALID;
  if (!std::isfinite(p->prob_scale) || p->prob_scale < 0.f) return KVQ_ERR_INVALID;
  if (p->out_dtype < KVQ_OUT_F32 || p->out_dtype > KVQ_OUT_E4M3) return KVQ_ERR_INVALID;
  if (p->out_dtype == KVQ_OUT_E4M3 && !finite_pos(p->out_scale)) return KVQ_ERR_INVALID;
  if (p->fresh_tokens < 0) return KVQ_ERR_INVALID;
  if (p->q_fp8 != 0 && p->q_fp8 != 1) return KVQ_ERR_INVALID;
  if (p->q_fp8 && !p->q_head_scale && !finite_pos(p->q_scale)) return KVQ_ERR_INVALID;
  return KVQ_OK;
}

kvq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

// ---------------------------------------------------------------------------
// Division by the prob scale (FP8 probabilities, vLLM PR 15734: softmax(QK^T)
// quantized to FP8 with prob_output_scale).  The kernels need E4M3(fl32(p /
// y)) for p in [0, 1] and the call's y = prob_scale.  With z = RN(1/y), the
// device's prob_quotient (q0 = RN(p z), r = RN(p - q0 y), q = RN(q0 + r z))
// is within one fp32 step of RN(p/y) for every p, and equals it unless p/y
// lies within about 2^-45 (relative) of the midpoint of two fp32 numbers.
// Two adjacent fp32 numbers can round to different E4M3 codes only if one of
// them is itself a rounding boundary of the E4M3 grid (a midpoint between two
// E4M3 values: every such midpoint is an fp32 number).  So the codes of the
// fast path equal those of the IEEE division for all p as soon as they do for
// every p whose quotient lies within 1.5 fp32 steps of a boundary; the check
// below runs the fast path on all p in a wider window (relative 2^-20) around
// each boundary's preimage and requires the correctly rounded quotient there.
// It is exact host arithmetic (this file is compiled with FP contraction off:
// the product and the two fused multiply-adds are the device's operations).
// ---------------------------------------------------------------------------

float fast_quotient(float p, float y, float z) {
  const float q0 = p * z;
  const float r = std::fma(-q0, y, p);
  return std::fma(r, z, q0);
}

// RN(p / y) in fp32: the double quotient is correctly rounded to 53 bits, and
// rounding it to 24 bits gives the correctly rounded fp32 quotient (53 >= 2 *
// 24 + 2).
float exact_quotient(float p, float y) { return (float)((double)p / (double)y); }

// Positive finite E4M3 values in increasing order (codes 0x00..0x7E).
double e4m3_positive(int code) {
  const int e = code >> 3, m = code & 7;
  return e == 0 ? std::ldexp((double)m, -9) : std::ldexp(1.0 + m / 8.0, e - 7);
}

bool prob_reciprocal_ok(float y, float* z_out) {
  if (!(y > 0.f) || !std::isfinite(y)) return false;
  const float z = (float)(1.0 / (double)y);
  if (!std::isfinite(z) || !(z > 0.f) || !std::isnormal(z)) return false;
  for (int c = 0; c < 0x7E; ++c) {
    const double mid = 0.5 * (e4m3_positive(c) + e4m3_positive(c + 1));   // a boundary
    const double lo = mid * (1.0 - std::ldexp(1.0, -20)) * y;
    const double hi = mid * (1.0 + std::ldexp(1.0, -20)) * y;
    if (lo > 1.0) break;   // no p in (0, 1] reaches this boundary
    float p = std::nextafter((float)lo, 0.f);
    const float end = std::nextafter((float)std::min(hi, 1.0), 2.f);
    for (; p <= end && p <= 1.f; p = std::nextafter(p, 2.f)) {
      if (!std::isnormal(p)) continue;
      if (fast_quotient(p, y, z) != exact_quotient(p, y)) return false;
    }
  }
  *z_out = z;
  return true;
}

}  // namespace

extern "C" {

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_WORKSPACE: return "workspace too small";
    case KVQ_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

kvq_status kvq_tensor_scale(int fmt, float amax, float* scale_out) {
  if (!scale_out) return KVQ_ERR_INVALID;
  if (!std::isfinite(amax) || amax < 0.f) return KVQ_ERR_INVALID;
  float top;
  if (fmt == KVQ_FP8_E4M3) top = 448.0f;
  else if (fmt == KVQ_NVFP4) top = 2688.0f;
  else return KVQ_ERR_INVALID;
  *scale_out = amax == 0.f ? 1.0f : amax / top;   // one IEEE fp32 division
  return KVQ_OK;
}

kvq_status kvq_amax_bf16(const void* x, size_t n, float* amax_out, void* stream) {
  if (!amax_out || (n > 0 && !x)) return KVQ_ERR_INVALID;
  return cuda_status(
      launch_amax_bf16(static_cast<const uint16_t*>(x), n, amax_out, as_stream(stream)));
}

kvq_status kvq_encode_e4m3(const float* x, uint8_t* out, size_t n, void* stream) {
  if (n > 0 && (!x || !out)) return KVQ_ERR_INVALID;
  return cuda_status(launch_encode(0, x, out, n, as_stream(stream)));
}

kvq_status kvq_encode_e2m1(const float* x, uint8_t* out, size_t n, void* stream) {
  if (n > 0 && (!x || !out)) return KVQ_ERR_INVALID;
  return cuda_status(launch_encode(1, x, out, n, as_stream(stream)));
}

kvq_status kvq_quantize_fp8(const void* x, size_t n, float scale, const float* head_scale,
                            int head_len, int num_heads, uint8_t* out, void* stream) {
  if (n == 0) return KVQ_OK;
  if (!x || !out || !aligned16(x) || n % 8 != 0) return KVQ_ERR_INVALID;
  if (head_scale) {
    if (head_len <= 0 || head_len % 8 != 0 || num_heads <= 0) return KVQ_ERR_INVALID;
  } else if (!finite_pos(scale)) {
    return KVQ_ERR_INVALID;
  }
  const float z = head_scale ? 0.f : (float)(1.0 / (double)scale);
  return cuda_status(launch_quantize_fp8(static_cast<const uint16_t*>(x), n, scale, z, head_scale,
                                         head_len, num_heads, out, as_stream(stream)));
}

kvq_status kvq_encode_prob_e4m3(const float* p, uint8_t* out, size_t n, float prob_scale,
                                int* used_reciprocal, void* stream) {
  if (!std::isfinite(prob_scale) || !(prob_scale > 0.f)) return KVQ_ERR_INVALID;
  if (n > 0 && (!p || !out)) return KVQ_ERR_INVALID;
  float z = 0.f;
  const int fast = prob_reciprocal_ok(prob_scale, &z) ? 1 : 0;
  if (used_reciprocal) *used_reciprocal = fast;
  return cuda_status(launch_encode_prob(p, out, n, prob_scale, z, fast, as_stream(stream)));
}

kvq_status kvq_quantize_append(const kvq_cache* c, const void* k_new, const void* v_new,
                               const void* kpe_new, const int32_t* start_pos, int batch,
                               int n_tokens, void* stream) {
  kvq_status s = check_cache(c);
  if (s != KVQ_OK) return s;
  if (batch < 0 || n_tokens < 0) return KVQ_ERR_INVALID;
  if (batch == 0 || n_tokens == 0) return KVQ_OK;
  if (!k_new || !aligned16(k_new) || !start_pos) return KVQ_ERR_INVALID;
  if (c->fmt == KVQ_FP8_E4M3 && c->head_dim % 8 != 0) return KVQ_ERR_INVALID;
  if (is_mla(c)) {
    if (v_new || !kpe_new || !aligned16(kpe_new)) return KVQ_ERR_INVALID;
  } else {
    if (!v_new || !aligned16(v_new) || kpe_new) return KVQ_ERR_INVALID;
  }
  if ((long long)batch * n_tokens * c->num_kv_heads * c->head_dim >= (1LL << 40))
    return KVQ_ERR_UNSUPPORTED;
  if (batch > 32767 || c->num_kv_heads > 65535 || n_tokens >= (1 << 30))
    return KVQ_ERR_UNSUPPORTED;
  AppendArgs a{};
  a.fmt = c->fmt;
  a.D = c->head_dim;
  a.Hkv = c->num_kv_heads;
  a.ps = c->page_size;
  a.max_pages = c->max_pages_per_seq;
  a.num_pages = c->num_pages;
  a.batch = batch;
  a.T = n_tokens;
  a.rope = is_mla(c) ? c->rope_dim : 0;
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.kpe_new = static_cast<const uint16_t*>(kpe_new);
  a.start_pos = start_pos;
  a.block_table = c->block_table;
  a.k_codes = static_cast<uint8_t*>(c->k_codes);
  a.v_codes = static_cast<uint8_t*>(c->v_codes);
  a.k_bscale = static_cast<uint8_t*>(c->k_bscale);
  a.v_bscale = static_cast<uint8_t*>(c->v_bscale);
  a.k_pe = static_cast<uint16_t*>(c->k_pe);
  a.k_scale = c->k_scale;
  a.v_scale = c->v_scale;
  // RN(1/scale): the double quotient rounded to fp32 is the correctly rounded
  // fp32 reciprocal (53 >= 2 * 24 + 2)
  a.k_recip = (float)(1.0 / (double)c->k_scale);
  a.v_recip = is_mla(c) ? a.k_recip : (float)(1.0 / (double)c->v_scale);
  a.k_hs = c->k_head_scale;
  a.v_hs = c->v_head_scale;
  a.has_v = is_mla(c) ? 0 : 1;
  return cuda_status(launch_append(a, as_stream(stream)));
}

kvq_status kvq_auto_splits(int num_sms, int batch, int num_kv_heads, int q_per_kv,
                           int max_kv_len, int fmt, int* out_s) {
  if (!out_s || num_sms < 1 || batch < 1 || num_kv_heads < 1 || max_kv_len < 0)
    return KVQ_ERR_INVALID;
  // When the (request, kv head) groups fit in one wave of the partial kernel
  // (two resident six-warp CTAs per SM, or three four-warp CTAs without wide
  // CTAs; two with more than eight query heads per kv head; one for the MLA
  // kernel: NVFP4, one kv head, 16 query heads), s fills that wave: a partly
  // filled second wave costs more than idle slots in the first (GQA FP8 batch
  // 16 x 8 kv heads at 8192 tokens: 52.3 us at s = 2, one wave, against 57.3
  // at s = 4 and 69.3 at s = 3; batch 8 at 32768: 91.6 us at s = 4 against
  // 106.6 at s = 16 and 128.7 at s = 5).  When they do not, the grid runs in
  // several waves anyway and chunks of at most kTargetChunk tokens cut long
  // or ragged requests into pieces that balance across them.
  // More than kManySplits splits of chunks shorter than kShortChunk tokens
  // lose to fewer, longer chunks (per-CTA fixed cost; the fused merge stages
  // about 30 splits in shared memory): measured on 8 kv-head groups at 8192
  // tokens, 28 splits 18.5 us against 21.0 us at 57.
  constexpr long long kMinChunk = 128, kMaxSplits = 64, kTargetChunk = 2048;
  constexpr long long kShortChunk = 256, kManySplits = 32;
  const bool mla_shape = fmt == KVQ_NVFP4 && num_kv_heads == 1 && q_per_kv == 16;
  const long long ctas_per_sm = mla_shape ? 1 : q_per_kv > 8 ? 2 : kWideCta ? 2 : 3;
  const long long base = (long long)batch * num_kv_heads;
  long long s = ctas_per_sm * num_sms / base;
  if (s < 1) s = ((long long)max_kv_len + kTargetChunk - 1) / kTargetChunk;
  if (s > kManySplits && (long long)max_kv_len < s * kShortChunk)
    s = std::max(kManySplits, ((long long)max_kv_len + kShortChunk - 1) / kShortChunk);
  const long long by_len = max_kv_len / kMinChunk;
  if (s > by_len) s = by_len;
  if (s < 1) s = 1;
  if (s > kMaxSplits) s = kMaxSplits;
  *out_s = (int)s;
  return KVQ_OK;
}

size_t kvq_partial_workspace_bytes(int batch, int num_q_heads, int num_splits, int v_dim) {
  if (batch < 0 || num_q_heads < 0 || num_splits < 0 || v_dim < 0) return 0;
  const size_t rows = (size_t)batch * num_q_heads * num_splits;
  return rows * (size_t)v_dim * sizeof(float) + rows * sizeof(float);
}

}  // extern "C"

namespace {

// Shared body of kvq_decode_partial and kvq_decode (fused when counters).
kvq_status decode_impl(const kvq_cache* c, const kvq_decode_params* p, const void* q,
                       float* part_o, float* part_lse, uint32_t* counters, void* out,
                       cudaStream_t stream) {
  kvq_status s = check_cache(c);
  if (s != KVQ_OK) return s;
  s = check_params(p);
  if (s != KVQ_OK) return s;
  if (p->batch == 0) return KVQ_OK;
  if (!q || !aligned16(q) || !part_o || !aligned16(part_o) || !part_lse) return KVQ_ERR_INVALID;
  if (counters && !out) return KVQ_ERR_INVALID;
  if (counters && p->num_splits > kMaxFusedSplits) return KVQ_ERR_UNSUPPORTED;
  if (p->num_q_heads % c->num_kv_heads != 0) return KVQ_ERR_INVALID;
  const int G = p->num_q_heads / c->num_kv_heads;
  if (G > kMaxGroup) return KVQ_ERR_UNSUPPORTED;
  if ((long long)p->max_kv_len > (long long)c->max_pages_per_seq * c->page_size)
    return KVQ_ERR_INVALID;
  if ((long long)p->batch * c->num_kv_heads >= (1LL << 31)) return KVQ_ERR_UNSUPPORTED;
  const bool probq = p->prob_scale > 0.f;
  long long score_floats = 0;
  if (probq) {
    long long chunk = ((long long)p->max_kv_len + p->num_splits - 1) / p->num_splits;
    chunk = (chunk + 15) / 16 * 16;
    score_floats = chunk * G;
    if (score_floats > kScoreCapacity) return KVQ_ERR_UNSUPPORTED;
  }
  const int D = c->head_dim;
  const uint64_t rows = (uint64_t)c->num_pages * c->num_kv_heads * c->page_size;

  PartialArgs a{};
  a.q = q;
  a.q_fp8 = p->q_fp8;
  a.q_scale = p->q_scale;
  a.q_hs = p->q_fp8 ? p->q_head_scale : nullptr;
  a.k_bscale = static_cast<const uint8_t*>(c->k_bscale);
  a.v_bscale = static_cast<const uint8_t*>(c->v_bscale);
  a.k_pe = static_cast<const uint16_t*>(c->k_pe);
  a.block_table = c->block_table;
  a.seq_lens = p->seq_lens;
  a.part_o = part_o;
  a.part_lse = part_lse;
  a.error_flag = p->error_flag;
  a.batch = p->batch;
  a.Hq = p->num_q_heads;
  a.Hkv = c->num_kv_heads;
  a.G = G;
  a.ps = c->page_size;
  a.max_pages = c->max_pages_per_seq;
  a.num_pages = c->num_pages;
  a.num_splits = p->num_splits;
  a.max_kv_len = p->max_kv_len;
  a.Dv = p->v_dim;
  a.score_floats = (int)score_floats;
  a.qk_scale_log2 = p->sm_scale * c->k_scale * 1.4426950408889634f;
  a.sm_scale = p->sm_scale;
  a.k_hs = c->k_head_scale;
  a.v_hs = c->v_head_scale;
  a.prob_scale = p->prob_scale;
  if (probq) a.prob_fast = prob_reciprocal_ok(p->prob_scale, &a.prob_recip) ? 1 : 0;
  a.fresh = p->fresh_tokens;
  a.counters = counters;
  a.out = out;
  a.out_dtype = p->out_dtype;
  a.out_scale = p->out_scale;

  if (is_mla(c)) {
    if (D != 512 || c->rope_dim != 64 || G != 16 || p->qk_dim != 576 || p->v_dim != 512)
      return KVQ_ERR_UNSUPPORTED;
    if (probq || p->q_fp8) return KVQ_ERR_UNSUPPORTED;
    a.out_mult = c->k_scale;   // the values are the latent itself
    a.pe_scale_log2 = p->sm_scale * 1.4426950408889634f;
    // latent codes as two 128-byte halves per row, rope keys as 128-byte rows,
    // both in 16-row boxes with the 128-byte swizzle
    // (and 64-row boxes for tiles inside one page)
    CUtensorMap tkv, tpe, tkv64, tpe64;
    if (!make_slice_map(&tkv, c->k_codes, 128, 2, rows, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_row_map(&tpe, c->k_pe, 128, rows) ||
        !make_slice_map(&tkv64, c->k_codes, 128, 2, rows, CU_TENSOR_MAP_SWIZZLE_128B,
                        rows >= 64 ? 64 : kBoxTokens) ||
        !make_row_map(&tpe64, c->k_pe, 128, rows, rows >= 64 ? 64 : kBoxTokens))
      return KVQ_ERR_CUDA;
    return cuda_status(launch_mla_partial(tkv, tpe, tkv64, tpe64, a, stream));
  }
  if (p->qk_dim != D || p->v_dim != D) return KVQ_ERR_INVALID;
  const bool ok_dims = (c->fmt == KVQ_FP8_E4M3 && (D == 64 || D == 128)) ||
                       (c->fmt == KVQ_NVFP4 && (D == 64 || D == 128 || D == 256));
  if (!ok_dims) return KVQ_ERR_UNSUPPORTED;
  a.out_mult = probq ? c->v_scale * p->prob_scale : c->v_scale;
  const uint64_t row_bytes = c->fmt == KVQ_FP8_E4M3 ? D : D / 2;
  TensorMaps maps;
  if (!make_row_map(&maps.k16, c->k_codes, row_bytes, rows) ||
      !make_row_map(&maps.v16, c->v_codes, row_bytes, rows))
    return KVQ_ERR_CUDA;
  return cuda_status(launch_partial(c->fmt, D, probq, maps, a, stream));
}

}  // namespace

extern "C" {

kvq_status kvq_decode_partial(const kvq_cache* c, const kvq_decode_params* p, const void* q,
                              float* part_o, float* part_lse, void* stream) {
  return decode_impl(c, p, q, part_o, part_lse, nullptr, nullptr, as_stream(stream));
}

kvq_status kvq_decode(const kvq_cache* c, const kvq_decode_params* p, const void* q,
                      float* part_o, float* part_lse, uint32_t* counters, void* out,
                      void* stream) {
  if (p && p->batch > 0 && (!counters || !out)) return KVQ_ERR_INVALID;
  return decode_impl(c, p, q, part_o, part_lse, counters, out,
                     as_stream(stream));
}

kvq_status kvq_decode_combine(const kvq_decode_params* p, const float* part_o,
                              const float* part_lse, void* out, void* stream) {
  kvq_status s = check_params(p);
  if (s != KVQ_OK) return s;
  if (p->batch == 0) return KVQ_OK;
  if (!part_o || !aligned16(part_o) || !part_lse || !out || p->v_dim % 4 != 0)
    return KVQ_ERR_INVALID;
  if ((long long)p->batch * p->num_q_heads >= (1LL << 31)) return KVQ_ERR_UNSUPPORTED;
  if (p->num_splits > kMaxFusedSplits) return KVQ_ERR_UNSUPPORTED;
  CombineArgs a{};
  a.part_o = part_o;
  a.part_lse = part_lse;
  a.out = out;
  a.rows = p->batch * p->num_q_heads;
  a.num_splits = p->num_splits;
  a.Dv = p->v_dim;
  a.out_dtype = p->out_dtype;
  a.out_scale = p->out_scale;
  return cuda_status(launch_combine(a, as_stream(stream)));
}

kvq_status kvq_prefill(const kvq_cache* c, const kvq_decode_params* p, int q_len, const void* q,
                       void* out, void* stream) {
  kvq_status s = check_cache(c);
  if (s != KVQ_OK) return s;
  s = check_params(p);
  if (s != KVQ_OK) return s;
  if (q_len < 1) return KVQ_ERR_INVALID;
  if (p->batch == 0) return KVQ_OK;
  if (!q || !aligned16(q) || !out) return KVQ_ERR_INVALID;
  if (p->num_q_heads % c->num_kv_heads != 0) return KVQ_ERR_INVALID;
  if (is_mla(c) || p->prob_scale > 0.f || p->q_fp8) return KVQ_ERR_UNSUPPORTED;
  const int D = c->head_dim;
  if (p->qk_dim != D || p->v_dim != D) return KVQ_ERR_INVALID;
  if (D != 64 && D != 128) return KVQ_ERR_UNSUPPORTED;
  if ((long long)p->max_kv_len > (long long)c->max_pages_per_seq * c->page_size)
    return KVQ_ERR_INVALID;
  const int G = p->num_q_heads / c->num_kv_heads;
  if ((long long)q_len * G >= (1LL << 30) || (long long)p->batch * c->num_kv_heads > 65535)
    return KVQ_ERR_UNSUPPORTED;
  PartialArgs a{};
  a.q = q;
  a.k_bscale = static_cast<const uint8_t*>(c->k_bscale);
  a.v_bscale = static_cast<const uint8_t*>(c->v_bscale);
  a.block_table = c->block_table;
  a.seq_lens = p->seq_lens;
  a.error_flag = p->error_flag;
  a.batch = p->batch;
  a.Hq = p->num_q_heads;
  a.Hkv = c->num_kv_heads;
  a.G = G;
  a.ps = c->page_size;
  a.max_pages = c->max_pages_per_seq;
  a.num_pages = c->num_pages;
  a.max_kv_len = p->max_kv_len;
  a.Dv = D;
  a.q_len = q_len;
  a.qk_scale_log2 = p->sm_scale * c->k_scale * 1.4426950408889634f;
  a.sm_scale = p->sm_scale;
  a.k_hs = c->k_head_scale;
  a.v_hs = c->v_head_scale;
  a.out_mult = c->v_scale;
  a.out = out;
  a.out_dtype = p->out_dtype;
  a.out_scale = p->out_scale;
  const uint64_t rows = (uint64_t)c->num_pages * c->num_kv_heads * c->page_size;
  const uint64_t row_bytes = c->fmt == KVQ_FP8_E4M3 ? D : D / 2;
  TensorMaps maps;
  if (!make_row_map(&maps.k16, c->k_codes, row_bytes, rows) ||
      !make_row_map(&maps.v16, c->v_codes, row_bytes, rows))
    return KVQ_ERR_CUDA;
  return cuda_status(launch_prefill(c->fmt, D, maps, a, as_stream(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free decode.
//
// Some callers cannot allocate device memory for the split partials: their
// device memory is owned by a host framework that hands out only the tensors
// it planned (a serving engine's fixed memory pool), or they run under a hard
// memory budget where an extra cudaMalloc is not allowed.  kvq_decode_noalloc
// serves them from one buffer the library itself carries: a file-scope device
// array of KVQ_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds
// until the process exits.  In host code the array's name is only a stand-in
// for the symbol, so the device's real address is looked up with
// cudaGetSymbolAddress (with that device current) on every call and passed
// to the kernel.
// ---------------------------------------------------------------------------

static __device__ __align__(256) unsigned char g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the scratch array on the current device.  Looked up on
// every call: after the first call on a device (which loads the module) it is
// a table lookup, and it stays right if the device's context is torn down
// and created again (the module, and so the array, may then move).
kvq_status noalloc_scratch(void** out) {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return KVQ_ERR_CUDA;
  *out = ptr;
  return KVQ_OK;
}

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" kvq_status kvq_decode_noalloc(const kvq_cache* c, const kvq_decode_params* p,
                                         const void* q, void* out, void* stream) {
  kvq_status st = check_cache(c);
  if (st != KVQ_OK) return st;
  st = check_params(p);
  if (st != KVQ_OK) return st;
  if (p->batch == 0) return KVQ_OK;
  if (!q || !out) return KVQ_ERR_INVALID;
  // scratch layout: [arrival counters][partial lse][partial o], 256-byte aligned
  const size_t rows = (size_t)p->batch * p->num_q_heads * p->num_splits;
  const size_t counter_bytes = up256((size_t)p->batch * c->num_kv_heads * sizeof(uint32_t));
  const size_t lse_bytes = up256(rows * sizeof(float));
  const size_t o_bytes = rows * (size_t)p->v_dim * sizeof(float);
  if (counter_bytes + lse_bytes + o_bytes > KVQ_NOALLOC_SCRATCH_BYTES) return KVQ_ERR_WORKSPACE;
  void* base = nullptr;
  st = noalloc_scratch(&base);
  if (st != KVQ_OK) return st;
  uint8_t* w = static_cast<uint8_t*>(base);
  uint32_t* counters = reinterpret_cast<uint32_t*>(w);
  float* part_lse = reinterpret_cast<float*>(w + counter_bytes);
  float* part_o = reinterpret_cast<float*>(w + counter_bytes + lse_bytes);
  // the arrival counters must start at zero (a previous call leaves them
  // zero; clearing them here keeps the contract independent of history)
  if (cudaMemsetAsync(counters, 0, counter_bytes, as_stream(stream)) != cudaSuccess)
    return KVQ_ERR_CUDA;
  return decode_impl(c, p, q, part_o, part_lse, counters, out, as_stream(stream));
}
