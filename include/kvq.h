/*
 * kvq.h -- C ABI of the GB300 (sm_103a) library for attention decode over a
 * quantized KV cache.
 *
 * What it computes (sources are the web pages the library follows):
 *  - Quantize-on-append of new K/V rows into the cache, as FP8 E4M3 with a
 *    static per-tensor scale (compressed-tensors PR 436, kv_cache_scheme:
 *    8-bit float, symmetric, strategy "tensor", dynamic false, minmax
 *    observer) or as NVFP4: E2M1 values in blocks of 16 along head_dim with a
 *    dynamic E4M3 block scale and an fp32 global scale (Model-Optimizer PR
 *    714, Testing: quantizers "(2, 1) bit ... block_sizes={-1: 16, 'type':
 *    'dynamic', 'scale_bits': (4, 3)}" with a calibrated amax).
 *  - Split-KV flash decode (Model-Optimizer PR 1832, notes under the latency
 *    tables): each (request, kv head) sequence is cut into s contiguous
 *    chunks; kvq_decode_partial runs one partial softmax (running max,
 *    denominator, weighted V) per chunk and kvq_decode_combine merges the s
 *    partials.  kvq_auto_splits picks s from the SM count and batch x heads.
 *  - Options: GQA/MHA head groups, paged blocks, FP8-quantized softmax
 *    probabilities with a prob scale and FP8 output with an out scale (vLLM
 *    PR 15734), and the MLA latent-cache variant (Model-Optimizer PR 714:
 *    kv_c_bmm_quantizer on the 512-wide latent cache, q_bmm_quantizer off).
 *
 * Conventions (all calls):
 *  - Every device buffer (cache, queries, outputs, workspace) is allocated
 *    and owned by the caller.  The library allocates no memory and keeps no
 *    per-call state; calls are re-entrant.  (It caches, per device, values
 *    that do not change: the number of MLA CTA clusters that fit at once.)
 *  - Pointers marked (device) must be device (or managed) memory of the
 *    current CUDA device; pointers marked (host) are read on the host.  The
 *    per-step inputs read with plain loads -- q, k_new, v_new, kpe_new --
 *    and the decode output may also be pinned host memory (page-locked and
 *    mapped, as cudaHostAlloc gives): the kernels then read and write it in
 *    place over the CPU-GPU link.  The cache, block table, seq_lens and the
 *    scratch must be device memory (the cache is read by TMA).
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream).  No call synchronizes.
 *  - Every call validates its arguments first and returns KVQ_ERR_INVALID or
 *    KVQ_ERR_UNSUPPORTED without launching anything.  After launching it
 *    returns KVQ_ERR_CUDA if the launch reported an error.
 *  - bf16 tensors are raw IEEE bfloat16 bit patterns (uint16).
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int kvq_status;
#define KVQ_OK 0
#define KVQ_ERR_INVALID 1      /* bad pointer, size, scale or layout */
#define KVQ_ERR_UNSUPPORTED 2  /* valid but not implemented (dims, format) */
#define KVQ_ERR_WORKSPACE 3    /* a workspace or scratch area is too small */
#define KVQ_ERR_CUDA 4         /* the CUDA runtime reported an error */

/* Cache formats */
#define KVQ_FP8_E4M3 1
#define KVQ_NVFP4 2

/* Output types of kvq_decode_combine */
#define KVQ_OUT_F32 0
#define KVQ_OUT_BF16 1
#define KVQ_OUT_E4M3 2

/* Bits that kernels OR into kvq_decode_params.error_flag */
#define KVQ_DEVERR_WAIT_TIMEOUT 1   /* a pipeline wait gave up (results invalid) */
#define KVQ_DEVERR_SEQ_CLAMPED 2    /* seq_lens[b] exceeded the cache; clamped */
#define KVQ_DEVERR_BAD_PAGE 4       /* a block-table entry was out of range; page 0 read */

/*
 * A paged quantized KV cache.  Caller-owned plain struct; the library only
 * reads it.
 *
 * Layout of one cache tensor (K or V), page-major then head-major, so one
 * (page, kv head) is a contiguous run of page_size rows:
 *   FP8:    codes  uint8 [num_pages][num_kv_heads][page_size][head_dim]
 *   NVFP4:  codes  uint8 [num_pages][num_kv_heads][page_size][head_dim/2]
 *                  (element 2i in the low nibble, 2i+1 in the high nibble)
 *           bscale uint8 [num_pages][num_kv_heads][page_size][head_dim/16]
 *                  (E4M3 block scales, one per 16 consecutive elements)
 * Token t of request b lives in page block_table[b*max_pages_per_seq + t /
 * page_size], row t % page_size.  A contiguous cache is the special case of
 * one page per request (page_size = capacity, block_table[b][0] = b).
 *
 * Dequantized values: FP8 x = dec(code) * scale; NVFP4 x = dec(e2m1) *
 * dec(bscale) * scale, where scale is k_scale or v_scale.
 *
 * MLA latent cache (rope_dim > 0): k_codes/k_bscale hold the NVFP4 latent
 * kv_c (num_kv_heads = 1, head_dim = 512), k_pe holds the bf16 rope keys
 * [num_pages][page_size][rope_dim], v_codes is NULL and v_is_k_latent = 1
 * (the values are the latent itself).
 */
typedef struct kvq_cache {
  int32_t fmt;               /* KVQ_FP8_E4M3 or KVQ_NVFP4 */
  int32_t num_pages;         /* >= 1 */
  int32_t page_size;         /* tokens per page, a multiple of 16 */
  int32_t num_kv_heads;      /* Hkv >= 1 */
  int32_t head_dim;          /* D: FP8 64 or 128; NVFP4 64, 128 or 256 (MLA 512) */
  void* k_codes;             /* (device) 16-byte aligned */
  void* v_codes;             /* (device) 16-byte aligned; NULL for MLA */
  void* k_bscale;            /* (device) NVFP4 only, 16-byte aligned */
  void* v_bscale;            /* (device) NVFP4 only, 16-byte aligned */
  float k_scale;             /* FP8 scale or NVFP4 global scale, finite > 0 */
  float v_scale;             /* as k_scale (ignored for MLA) */
                             /* (both ignored where per-head scales are given) */
  const int32_t* block_table;/* (device) [batch][max_pages_per_seq] */
  int32_t max_pages_per_seq; /* >= 1 */
  int32_t rope_dim;          /* MLA: 64; otherwise 0 */
  void* k_pe;                /* (device) MLA only: bf16 rope keys */
  int32_t v_is_k_latent;     /* MLA: 1; otherwise 0 */
  /*
   * Per-kv-head scales (compressed-tensors PR 436, "attn_head" strategy: one
   * static scale per attention head).  Optional, (device) float
   * [num_kv_heads] each: when non-NULL, kv head h of K (V) uses
   * k_head_scale[h] (v_head_scale[h]) wherever k_scale (v_scale) appears
   * above -- the FP8 scale or the NVFP4 global scale -- in the append and in
   * the decode, and k_scale (v_scale) is ignored.  Every entry must be
   * finite and > 0 (not checked: device memory).  They are read like the
   * block table, so nothing still running may write them (fresh_tokens).
   * Not for MLA (one latent kv head: use k_scale).
   */
  const float* k_head_scale;
  const float* v_head_scale;
} kvq_cache;

/* Parameters of one decode step (shared by partial and combine). */
typedef struct kvq_decode_params {
  int32_t batch;             /* B >= 0 (0 is a no-op) */
  int32_t num_q_heads;       /* Hq, a multiple of Hkv; Hq/Hkv <= 16 */
  int32_t qk_dim;            /* head_dim (MLA: 512 + 64 = 576) */
  int32_t v_dim;             /* head_dim (MLA: 512) */
  int32_t num_splits;        /* 1 <= s <= 64 (see kvq_auto_splits) */
  const int32_t* seq_lens;   /* (device) [batch] tokens per request */
  int32_t max_kv_len;        /* (host) upper bound of seq_lens[] */
  float sm_scale;            /* softmax scale (e.g. 1/sqrt(head_dim)) */
  float prob_scale;          /* > 0: FP8 softmax probabilities; 0: off */
  int32_t out_dtype;         /* KVQ_OUT_* (used by combine) */
  float out_scale;           /* KVQ_OUT_E4M3: output scale, finite > 0 */
  int32_t* error_flag;       /* (device, optional) KVQ_DEVERR_* bits OR-ed in */
  /*
   * Overlap with the append of this step (>= 0).  0: the decode waits for
   * the preceding kernel in the stream to finish before it reads any input
   * (always correct).  n > 0 declares that the work issued immediately
   * before on the same stream is one kvq_quantize_append call that wrote
   * only positions seq_lens[b] - n .. seq_lens[b] - 1 of each request, and
   * that q, seq_lens, the block table and every other cache position were
   * complete when that call was made (kvq_quantize_append starts after all
   * earlier work in the stream).  The decode then streams every other part
   * of the cache while the append runs and waits for it only before the
   * boxes that hold those positions.  q, seq_lens and the block table are
   * read before that wait, so the append (or anything else still running
   * when the decode starts) must not write them.  Not part of the pages'
   * method: a scheduling contract between two calls of this library.
   */
  int32_t fresh_tokens;
  /*
   * FP8 query (compressed-tensors PR 436: a query observer next to the K
   * and V ones, GSM8K rows "QKV-FP8-Tensor" / "QKV-FP8-Head"; vLLM PR 15734:
   * QK quantization in the attention loop).  q_fp8 = 0: q is bf16 (default).
   * q_fp8 = 1: q holds E4M3 codes [batch][Hq][qk_dim] (kvq_quantize_fp8
   * makes them) whose values are dec(code) * q_scale, or * q_head_scale[hq]
   * when that (device, [num_q_heads]) array is given.  With an FP8 cache the
   * scores run on E4M3 x E4M3 tensor-core MMAs straight from the cached
   * codes; with an NVFP4 cache the codes are widened exactly to f16.  Not
   * for MLA.
   */
  int32_t q_fp8;
  float q_scale;             /* q_fp8 without q_head_scale: finite > 0 */
  const float* q_head_scale; /* (device, optional) [num_q_heads] */
} kvq_decode_params;

/* Human-readable name of a status code (static string). */
const char* kvq_status_string(kvq_status s);

/*
 * Static per-tensor scale from a calibrated amax (the minmax observer of
 * compressed-tensors PR 436; the MaxCalibrator amax of Model-Optimizer PR
 * 714).  Host only.
 *   KVQ_FP8_E4M3: scale = fl32(amax / 448)   (448 = largest E4M3 value)
 *   KVQ_NVFP4:    scale = fl32(amax / 2688)  (2688 = 6 * 448: largest E2M1
 *                 value times largest E4M3 block scale)
 * amax == 0 gives 1.0.  Negative, NaN or infinite amax -> KVQ_ERR_INVALID.
 */
kvq_status kvq_tensor_scale(int fmt, float amax, float* scale_out /* host */);

/*
 * amax = max |x| over n bf16 values, written to *amax_out (device float).
 * The calibration step that feeds kvq_tensor_scale.  n may be 0 (gives 0).
 */
kvq_status kvq_amax_bf16(const void* x /* device bf16 [n] */, size_t n,
                         float* amax_out /* device */, void* stream);

/*
 * Quantize-on-append.  Writes n_tokens new rows per request into the cache:
 * row t of request b goes to position start_pos[b] + t.
 *   k_new   (device) bf16 [batch][n_tokens][num_kv_heads][head_dim]
 *   v_new   (device) bf16, same shape (NULL for MLA)
 *   kpe_new (device) bf16 [batch][n_tokens][rope_dim] (MLA only, else NULL)
 *   start_pos (device) int32 [batch]
 * FP8:   code = E4M3(fl32(x / scale)), round to nearest even, saturating at
 *        +-448 (the sign of zero is kept).
 * NVFP4, per 16-element block along head_dim:
 *        bamax = max |x|;  sc = E4M3(fl32(fl32(bamax / 6) / scale));
 *        es = fl32(dec(sc) * scale);  code = E2M1(fl32(x / es)) (all 0 when
 *        es == 0), round to nearest even, saturating at +-6.
 * The caller guarantees that the pages for positions start_pos[b] ..
 * start_pos[b] + n_tokens - 1 exist in the block table; positions past
 * max_pages_per_seq * page_size are skipped (not written).
 * Input pointers must be 16-byte aligned.  batch <= 32767, num_kv_heads <=
 * 65535 and n_tokens < 2^30 (else KVQ_ERR_UNSUPPORTED).
 */
kvq_status kvq_quantize_append(const kvq_cache* c, const void* k_new, const void* v_new,
                               const void* kpe_new, const int32_t* start_pos, int batch,
                               int n_tokens, void* stream);

/*
 * Split-count heuristic (host only, deterministic).  base = batch *
 * num_kv_heads (MLA: batch) CTAs per split; the partial kernel keeps
 * ctas_per_sm CTAs resident per SM (2: six-warp CTAs, or four-warp CTAs
 * with more than 8 query heads per kv head; 1 for the MLA shape:
 * KVQ_NVFP4, num_kv_heads 1, q_per_kv 16), so
 * s = floor(ctas_per_sm * num_sms / base) splits fill one wave; when that
 * is 0 (more groups than one wave holds), s = ceil(max_kv_len / 2048), so
 * that long or ragged requests are cut into chunks that balance across the
 * waves.  Above 32 splits with
 * chunks under 256 tokens (max_kv_len < 256 s), s becomes
 * max(32, ceil(max_kv_len / 256)).  s is then lowered so that every chunk
 * keeps at least 128 tokens and clamped to [1, 64].  num_sms is
 * the device's multiprocessor count (cudaDevAttrMultiProcessorCount).
 */
kvq_status kvq_auto_splits(int num_sms, int batch, int num_kv_heads, int q_per_kv,
                           int max_kv_len, int fmt, int* out_s /* host */);

/* Bytes of the split partials: part_o (fp32 [batch][Hq][s][v_dim]) plus
 * part_lse (fp32 [batch][Hq][s]). */
size_t kvq_partial_workspace_bytes(int batch, int num_q_heads, int num_splits, int v_dim);

/*
 * Split-KV partial.  For request b, query head hq (kv head hq / (Hq/Hkv))
 * and split j, over chunk j of the request's sequence (chunk length c =
 * ceil(L/s) rounded up to 16 tokens; chunk j = [j*c, min((j+1)*c, L))):
 *   S_i = sm_scale * q . k^_i;   m = max_i S_i;   l = sum_i exp(S_i - m)
 *   part_o[b][hq][j][:] = sum_i exp(S_i - m) v^_i / l
 *   part_lse[b][hq][j]  = m + ln l          (-inf and o = 0 for empty chunks)
 * With prob_scale > 0 (FP8 probabilities) the weight of v^_i is
 *   p_q = dec(E4M3(fl32(p~ / prob_scale))) * prob_scale, p~ = exp(S_i - m)
 * in fp32 with m the chunk max, while l sums the unquantized p~.
 *   q (device) bf16 [batch][Hq][qk_dim], 16-byte aligned.
 *   part_o, part_lse (device) as in kvq_partial_workspace_bytes; part_o
 *   16-byte aligned.
 * With prob_scale > 0 one chunk's scores must fit in on-chip memory:
 * ceil(max_kv_len / s) rounded up to 16, times Hq/Hkv, at most 16384;
 * larger chunks return KVQ_ERR_UNSUPPORTED (raise num_splits).
 */
kvq_status kvq_decode_partial(const kvq_cache* c, const kvq_decode_params* p, const void* q,
                              float* part_o, float* part_lse, void* stream);

/*
 * Combine of the s partials of kvq_decode_partial:
 *   M = max_j lse_j;  w_j = exp(lse_j - M);  O = sum_j w_j o_j / sum_j w_j
 * (partials with lse = -inf are skipped; O = 0 when all are empty), written
 * to out (device) [batch][Hq][v_dim] as fp32, bf16 (round to nearest even)
 * or E4M3 codes E4M3(fl32(O / out_scale)) per p->out_dtype.
 */
kvq_status kvq_decode_combine(const kvq_decode_params* p, const float* part_o,
                              const float* part_lse, void* out, void* stream);

/*
 * One decode step in a single launch: kvq_decode_partial followed by the
 * merge of kvq_decode_combine, which the last CTA to finish for each
 * (request, kv head) performs with the same arithmetic and output types.
 * MLA with 2..8 splits runs as thread-block clusters of a request's splits
 * when they fit the device in as many waves as single CTAs: the partials
 * then merge through distributed shared memory (part_o and part_lse are not
 * written, the counters not used), with the same results bit for bit.
 *   part_o, part_lse (device) split partials, as for kvq_decode_partial.
 *   counters (device) uint32 [batch * num_kv_heads] arrival counters.  They
 *   must be zero before the first call; every call leaves them at zero
 *   again, so one zero-filled array (sized for the largest batch *
 *   num_kv_heads) serves any number of later calls.  Calls that share
 *   counters or partials must not overlap on the GPU (stream-order them).
 *   out (device) [batch][Hq][v_dim] in p->out_dtype.
 */
kvq_status kvq_decode(const kvq_cache* c, const kvq_decode_params* p, const void* q,
                      float* part_o, float* part_lse, uint32_t* counters, void* out,
                      void* stream);

/*
 * Prefill attention over the cache (Model-Optimizer PR 1832: the prefill
 * kernel of its latency tables, timed against split-KV decode): causal, no
 * KV split.  Request b holds seq_lens[b] = L tokens, the last q_len of them
 * the new ones whose queries are given: query i (position L - q_len + i)
 * attends to keys 0 .. L - q_len + i,
 *   out[b][i][hq][:] = sum_j softmax_j(sm_scale q . k^_j) v^_j
 * in p->out_dtype (as kvq_decode_combine writes it).  With q_len = 1 this
 * is one program per (request, kv head) over the whole sequence.
 *   q   (device) bf16 [batch][q_len][Hq][head_dim], 16-byte aligned.
 *   out (device) [batch][q_len][Hq][head_dim].
 * Uses batch, num_q_heads, qk_dim = v_dim = head_dim, seq_lens, max_kv_len,
 * sm_scale, out_dtype, out_scale and error_flag of p (num_splits and
 * fresh_tokens are ignored; prob_scale must be 0 and q_fp8 0).  FP8 or
 * NVFP4 caches with head_dim 64 or 128, per-kv-head scales allowed; not MLA.
 * Requests with L < q_len: queries before position 0 attend to nothing and
 * give 0.  q_len >= 1.
 */
kvq_status kvq_prefill(const kvq_cache* c, const kvq_decode_params* p, int q_len, const void* q,
                       void* out, void* stream);

/*
 * Allocation-free decode step (the pages have no counterpart; this is a
 * convenience of this library).  For callers that cannot allocate device
 * memory -- their device memory is owned by a host framework's fixed pool,
 * or a hard memory budget forbids another cudaMalloc -- this does what
 * kvq_decode does, but keeps the split partials and arrival counters in a
 * static device buffer inside the library: KVQ_NOALLOC_SCRATCH_BYTES (4 MiB)
 * that every GPU loading the library holds until the process exits.  The
 * caller passes only inputs and the output.
 *   Needs 256-aligned (4 * batch * num_kv_heads) + 256-aligned
 *   (4 * batch * Hq * num_splits) + 4 * batch * Hq * num_splits * v_dim
 *   bytes <= KVQ_NOALLOC_SCRATCH_BYTES; larger requests return
 *   KVQ_ERR_WORKSPACE (use kvq_decode with caller-owned buffers).
 *   Every call looks up the buffer's device address on the current device
 *   (cudaGetSymbolAddress); the first call on a device also loads the
 *   library's device code there, so make it before any stream capture.
 *   Every call clears the counters (an asynchronous memset on `stream`)
 *   and then launches the decode; it allocates and frees nothing.  The
 *   memset sits between a preceding kvq_quantize_append and the decode, so
 *   p->fresh_tokens > 0 is accepted but gives no overlap here: the decode
 *   starts after the append has finished.
 *   All calls share the one buffer: calls that overlap on the GPU (other
 *   streams, other host threads) race and must be serialized by the caller.
 */
#define KVQ_NOALLOC_SCRATCH_BYTES (4u << 20)
kvq_status kvq_decode_noalloc(const kvq_cache* c, const kvq_decode_params* p, const void* q,
                              void* out, void* stream);

/*
 * FP8 quantization of bf16 values (e.g. the query of an FP8-query decode):
 *   out[i] = E4M3(fl32(x[i] / s)), s = head_scale[(i / head_len) % num_heads]
 * when head_scale (device, [num_heads]) is given, else scale (finite > 0);
 * round to nearest even, saturating at +-448, the sign of zero kept -- the
 * arithmetic of the FP8 append.  x (device, bf16, 16-byte aligned) and out
 * (device) hold n elements; n and head_len multiples of 8 (head_len > 0
 * when head_scale is given).
 */
kvq_status kvq_quantize_fp8(const void* x, size_t n, float scale, const float* head_scale,
                            int head_len, int num_heads, uint8_t* out, void* stream);

/*
 * Elementwise fp32 -> code conversions with the device encoders the append
 * path uses: out[i] = E4M3(x[i]) (round to nearest even, saturating at
 * +-448) or the E2M1 nibble of x[i] (saturating at +-6) in the low 4 bits.
 * x and out (device), n >= 0.  NaN inputs give unspecified codes.
 */
kvq_status kvq_encode_e4m3(const float* x, uint8_t* out, size_t n, void* stream);
kvq_status kvq_encode_e2m1(const float* x, uint8_t* out, size_t n, void* stream);

/*
 * The FP8-probability quantizer of the decode kernels (vLLM PR 15734:
 * softmax(QK^T) quantized to FP8 with prob_output_scale), elementwise:
 *   out[i] = E4M3(fl32(p[i] / prob_scale))   (round to nearest even, +-448)
 * computed exactly as kvq_decode_partial computes it for probabilities in
 * [0, 1].  The division by prob_scale takes a precomputed reciprocal and one
 * fused correction when a host check shows that, for this prob_scale, it
 * gives the codes of the IEEE division for every p in [0, 1] (it always does
 * near the E4M3 rounding boundaries, where it is checked, and it is within
 * one fp32 step of the IEEE quotient everywhere); otherwise it is the IEEE
 * division.  *used_reciprocal (host, optional) tells which.  prob_scale
 * finite > 0; p and out (device), n >= 0 (n = 0 runs only the host check).
 * Codes for p outside [0, 1] are unspecified.
 */
kvq_status kvq_encode_prob_e4m3(const float* p, uint8_t* out, size_t n, float prob_scale,
                                int* used_reciprocal /* host */, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
