// Plain CPU oracle for attention decode over a quantized KV cache.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
// reference that the CUDA library is checked against.  Only the tests, the
// smoke check and the benchmark's CPU-baseline leg may load it; the product
// path never does.  It shares no code, header, table or helper with the CUDA
// library under quantized_kv_cache_05_gb300/csrc.
//
// Sources (the web pages this build follows):
//   [MO-714]   NVIDIA Model-Optimizer PR 714, "KV cache quantization for vLLM
//              fakequant MLA attention" -- Testing section, module printout:
//              NVFP4 quantizers "(2, 1) bit fake block_sizes={-1: 16,
//              'type': 'dynamic', 'scale_bits': (4, 3)}" with a MaxCalibrator
//              amax, and kv_c_bmm_quantizer on the MLA latent cache.
//   [CT-436]   vllm-project/compressed-tensors PR 436, attention and KV-cache
//              quantization -- kv_cache_scheme JSON: 8-bit float, symmetric,
//              strategy "tensor", static (dynamic: false), minmax observer.
//   [VLLM-15734] vLLM PR 15734, "Add support for FP8 models with input_scale
//              for output projection and QK quantization" -- FP8 attention
//              output via _out_scale, FP8 softmax(QK^T) via prob_output_scale.
//   [MO-1832]  NVIDIA Model-Optimizer PR 1832, "Add quant+sparse attention for
//              vLLM serving" -- notes under the latency tables: s =
//              num_kv_splits contiguous chunks, per-chunk partial softmax
//              (running max, denominator, weighted V), combine of s partials.
//   [OCP-FP8]  OCP 8-bit floating point spec, E4M3 ("FN") encoding; the E2M1
//              element format of OCP MX / NVFP4.  The pages name these formats
//              by their bit splits ("(2, 1) bit", "scale_bits (4, 3)").
//
// Arithmetic conventions.
//  * Everything is computed in double.
//  * Where the quantizer contract calls for a single IEEE fp32 operation
//    (written fl32(a op b) below) the oracle computes it in double and rounds
//    the result to float.  For +, -, *, / of two floats this double rounding
//    is exact (double carries 53 >= 2*24+2 significand bits), so the result is
//    the correctly rounded fp32 value.
//  * Rounding onto the E4M3 / E2M1 grids is an explicit round-half-to-even on
//    the exact scaled value, written from the format definition.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <cstdio>
#include <cstdlib>
#include <vector>
#include <thread>
#include <algorithm>
#include <limits>

namespace {

// ---------------------------------------------------------------------------
// Small helpers
// ---------------------------------------------------------------------------

// Round a non-negative double to the nearest integer, ties to even.
double round_half_even(double v) {
  double fl = std::floor(v);
  double frac = v - fl;  // exact: v and fl share an exponent range
  if (frac > 0.5) return fl + 1.0;
  if (frac < 0.5) return fl;
  return (std::fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

// fl32(a / b): the correctly rounded IEEE single-precision quotient.
float fl32_div(float a, float b) { return (float)((double)a / (double)b); }
// fl32(a * b)
float fl32_mul(float a, float b) { return (float)((double)a * (double)b); }

// bf16 bit pattern -> exact value (bf16 is the top half of an fp32).
double bf16_value(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

void die(const char* what) {
  std::fprintf(stderr, "oracle: %s\n", what);
  std::abort();
}

// ---------------------------------------------------------------------------
// E4M3 ("FN" variant) codec -- [OCP-FP8]; named "(4, 3)" scale bits in
// [MO-714] and "num_bits: 8, type: float" in [CT-436].
// Layout: sign(1) exponent(4, bias 7) mantissa(3).  Exponent field 0 holds
// subnormals m * 2^-9.  There are no infinities; S.1111.111 is NaN, so the
// largest finite magnitude is 1.75 * 2^8 = 448.
// ---------------------------------------------------------------------------

double e4m3_decode(uint8_t code) {
  int s = code >> 7;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return std::numeric_limits<double>::quiet_NaN();
  if (e == 0)
    mag = std::ldexp((double)m, -9);               // m/8 * 2^(1-7)
  else
    mag = std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

// Round-to-nearest-even onto the E4M3 grid; |x| > 448 (and +-inf) saturate
// to +-448.  The sign of zero is kept.
uint8_t e4m3_encode(float xf) {
  if (std::isnan(xf)) die("e4m3_encode: NaN input");
  double x = xf;
  uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  double a = std::fabs(x);
  if (a > 448.0) return sign | 0x7E;
  const double min_normal = std::ldexp(1.0, -6);
  if (a < min_normal) {
    // Subnormal range: grid spacing 2^-9, integers 0..8 (8 == min normal).
    double n = round_half_even(std::ldexp(a, 9));
    if (n >= 8.0) return sign | 0x08;              // exponent field 1, m = 0
    return sign | (uint8_t)n;
  }
  int k;
  std::frexp(a, &k);                                // a = f * 2^k, f in [0.5,1)
  int e = k - 1;                                    // a in [2^e, 2^(e+1))
  double n = round_half_even(std::ldexp(a, 3 - e)); // a / 2^(e-3), in [8,16]
  if (n >= 16.0) { e += 1; n = 8.0; }
  int ef = e + 7;                                   // biased exponent
  int mf = (int)n - 8;
  // a <= 448 keeps the result at or below 0x7E; the check guards the logic.
  if (ef > 15 || (ef == 15 && mf > 6)) die("e4m3_encode: exponent overflow");
  return sign | (uint8_t)(ef << 3) | (uint8_t)mf;
}

// ---------------------------------------------------------------------------
// E2M1 codec -- the "(2, 1) bit" element type of [MO-714]; [OCP-FP8] MX
// element format.  Layout: sign(1) exponent(2, bias 1) mantissa(1).
// Values: 0, 0.5 (subnormal), 1, 1.5, 2, 3, 4, 6.  No NaN, no infinity.
// ---------------------------------------------------------------------------

double e2m1_decode(uint8_t nib) {
  int s = (nib >> 3) & 1;
  int e = (nib >> 1) & 3;
  int m = nib & 1;
  double mag = (e == 0) ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

// Round-to-nearest-even onto the E2M1 grid; |x| > 6 saturates to +-6.
uint8_t e2m1_encode(float xf) {
  if (std::isnan(xf)) die("e2m1_encode: NaN input");
  double x = xf;
  uint8_t sign = std::signbit(x) ? 0x8 : 0x0;
  double a = std::fabs(x);
  if (a > 6.0) return sign | 0x7;
  if (a < 1.0) {
    // Subnormal range: spacing 0.5, integers 0..2 (2 == 1.0, the min normal).
    double n = round_half_even(a * 2.0);
    if (n >= 2.0) return sign | 0x2;
    return sign | (uint8_t)n;
  }
  int k;
  std::frexp(a, &k);
  int e = k - 1;                                    // 0, 1 or 2
  double n = round_half_even(std::ldexp(a, 1 - e)); // a / 2^(e-1), in [2,4]
  if (n >= 4.0) { e += 1; n = 2.0; }
  int ef = e + 1;
  int mf = (int)n - 2;
  if (ef > 3) die("e2m1_encode: exponent overflow");
  return sign | (uint8_t)(ef << 1) | (uint8_t)mf;
}

// ---------------------------------------------------------------------------
// Attention pieces -- plain definitions.
// ---------------------------------------------------------------------------

double dot(const double* a, const double* b, int n) {
  double s = 0.0;
  for (int i = 0; i < n; ++i) s += a[i] * b[i];
  return s;
}

}  // namespace

extern "C" {

// ===========================================================================
// Codecs (exported for the oracle's own pins and for the codec sweeps)
// ===========================================================================

uint8_t orc_e4m3_encode(float x) { return e4m3_encode(x); }
double orc_e4m3_decode(uint8_t c) { return e4m3_decode(c); }
uint8_t orc_e2m1_encode(float x) { return e2m1_encode(x); }
double orc_e2m1_decode(uint8_t c) { return e2m1_decode(c); }

void orc_e4m3_encode_n(const float* x, size_t n, uint8_t* out) {
  for (size_t i = 0; i < n; ++i) out[i] = e4m3_encode(x[i]);
}
void orc_e2m1_encode_n(const float* x, size_t n, uint8_t* out) {
  for (size_t i = 0; i < n; ++i) out[i] = e2m1_encode(x[i]);
}

// Count, over the fp32 bit patterns [first, first + n), the non-NaN inputs
// whose code in `observed` (one byte per input) differs from the oracle's
// encoder.  kind 0 = E4M3, 1 = E2M1 (codes in the low nibble).  Threaded.
// Used to compare a device encoder with the oracle over all 2^32 patterns.
uint64_t orc_count_encode_mismatch(int kind, uint64_t first, uint64_t n,
                                   const uint8_t* observed, int nthreads,
                                   uint64_t* first_bad_pattern) {
  if (nthreads < 1) nthreads = 1;
  std::vector<uint64_t> bad(nthreads, 0), firstbad(nthreads, UINT64_MAX);
  std::vector<std::thread> th;
  for (int t = 0; t < nthreads; ++t) {
    th.emplace_back([&, t]() {
      uint64_t lo = n * t / nthreads, hi = n * (t + 1) / nthreads;
      for (uint64_t i = lo; i < hi; ++i) {
        uint32_t bits = (uint32_t)(first + i);
        float f;
        std::memcpy(&f, &bits, 4);
        if (std::isnan(f)) continue;
        uint8_t want = kind == 0 ? e4m3_encode(f) : e2m1_encode(f);
        if (observed[i] != want) {
          if (bad[t] == 0) firstbad[t] = first + i;
          ++bad[t];
        }
      }
    });
  }
  for (auto& x : th) x.join();
  uint64_t total = 0, fb = UINT64_MAX;
  for (int t = 0; t < nthreads; ++t) { total += bad[t]; fb = std::min(fb, firstbad[t]); }
  if (first_bad_pattern) *first_bad_pattern = fb;
  return total;
}

// Count, over the fp32 bit patterns [first, first + n) read as probabilities
// p, the inputs whose code in `observed` differs from E4M3(fl32(p /
// prob_scale)) -- the FP8-probability quantization step of
// orc_attention_partial_probq ([VLLM-15734]: softmax(QK^T) quantized to FP8
// with prob_output_scale).  Threaded.  Used to compare the device's division
// by the prob scale with the oracle over every p in (0, 1].
uint64_t orc_count_probq_mismatch(uint64_t first, uint64_t n, float prob_scale,
                                  const uint8_t* observed, int nthreads,
                                  uint64_t* first_bad_pattern) {
  if (nthreads < 1) nthreads = 1;
  std::vector<uint64_t> bad(nthreads, 0), firstbad(nthreads, UINT64_MAX);
  std::vector<std::thread> th;
  for (int t = 0; t < nthreads; ++t) {
    th.emplace_back([&, t]() {
      uint64_t lo = n * t / nthreads, hi = n * (t + 1) / nthreads;
      for (uint64_t i = lo; i < hi; ++i) {
        uint32_t bits = (uint32_t)(first + i);
        float p;
        std::memcpy(&p, &bits, 4);
        if (std::isnan(p)) continue;
        uint8_t want = e4m3_encode(fl32_div(p, prob_scale));
        if (observed[i] != want) {
          if (bad[t] == 0) firstbad[t] = first + i;
          ++bad[t];
        }
      }
    });
  }
  for (auto& x : th) x.join();
  uint64_t total = 0, fb = UINT64_MAX;
  for (int t = 0; t < nthreads; ++t) { total += bad[t]; fb = std::min(fb, firstbad[t]); }
  if (first_bad_pattern) *first_bad_pattern = fb;
  return total;
}

// Brute-force pin of the encoders: for every non-NaN fp32 pattern in
// [first, first+n), pick the nearest grid value by a search over the sorted
// table of decoded codes (ties to the code with an even mantissa, i.e. an
// even code index), saturating above the largest finite value, and count the
// disagreements with the encoder.  This path uses only the decoder and
// comparisons -- none of the encoder's scaling arithmetic.
uint64_t orc_bruteforce_encode_check(int kind, uint64_t first, uint64_t n,
                                     int nthreads, uint64_t* first_bad_pattern) {
  // Non-negative finite grid, sorted, with its codes.
  std::vector<double> val;
  std::vector<uint8_t> code;
  int ncodes = kind == 0 ? 0x7F : 0x8;              // positive half of the table
  for (int c = 0; c < ncodes; ++c) {
    double v = kind == 0 ? e4m3_decode((uint8_t)c) : e2m1_decode((uint8_t)c);
    if (std::isnan(v)) continue;
    val.push_back(v);
    code.push_back((uint8_t)c);
  }
  for (size_t i = 1; i < val.size(); ++i)
    if (!(val[i] > val[i - 1])) die("bruteforce: table not strictly increasing");
  const double top = val.back();
  const uint8_t sign_bit = kind == 0 ? 0x80 : 0x8;
  if (nthreads < 1) nthreads = 1;
  std::vector<uint64_t> bad(nthreads, 0), firstbad(nthreads, UINT64_MAX);
  std::vector<std::thread> th;
  for (int t = 0; t < nthreads; ++t) {
    th.emplace_back([&, t]() {
      uint64_t lo = n * t / nthreads, hi = n * (t + 1) / nthreads;
      for (uint64_t i = lo; i < hi; ++i) {
        uint32_t bits = (uint32_t)(first + i);
        float f;
        std::memcpy(&f, &bits, 4);
        if (std::isnan(f)) continue;
        double a = std::fabs((double)f);
        uint8_t c;
        if (a >= top) {
          c = code.back();
        } else {
          // first index with val > a
          size_t j = std::upper_bound(val.begin(), val.end(), a) - val.begin();
          double lo_v = val[j - 1], hi_v = val[j];
          double dlo = a - lo_v, dhi = hi_v - a;
          if (dlo < dhi) c = code[j - 1];
          else if (dhi < dlo) c = code[j];
          else c = (code[j - 1] % 2 == 0) ? code[j - 1] : code[j];
        }
        if (std::signbit(f)) c |= sign_bit;
        uint8_t enc = kind == 0 ? e4m3_encode(f) : e2m1_encode(f);
        if (enc != c) {
          if (bad[t] == 0) firstbad[t] = first + i;
          ++bad[t];
        }
      }
    });
  }
  for (auto& x : th) x.join();
  uint64_t total = 0, fb = UINT64_MAX;
  for (int t = 0; t < nthreads; ++t) { total += bad[t]; fb = std::min(fb, firstbad[t]); }
  if (first_bad_pattern) *first_bad_pattern = fb;
  return total;
}

// ===========================================================================
// Static scale setup -- [CT-436] kv_cache_scheme (static, minmax, per tensor);
// [MO-714] MaxCalibrator amax.
// ===========================================================================

// amax = max |x| over a bf16 tensor (exact: every bf16 is an fp32).
float orc_amax_bf16(const uint16_t* x, size_t n) {
  double m = 0.0;
  for (size_t i = 0; i < n; ++i) {
    double v = std::fabs(bf16_value(x[i]));
    if (std::isnan(v)) die("amax: NaN input");
    if (v > m) m = v;
  }
  return (float)m;
}

// FP8 per-tensor scale: fl32(amax / 448), the scale that maps the tensor's
// amax onto the largest finite E4M3 value.  amax == 0 gives 1.0 (every code is
// zero then, and the scale must stay a positive divisor).
float orc_fp8_tensor_scale(float amax) {
  if (!(amax > 0.0f)) return 1.0f;
  return fl32_div(amax, 448.0f);
}

// NVFP4 global scale: fl32(amax / 2688), 2688 = 6 * 448 = (largest E2M1) *
// (largest E4M3 block scale).  amax == 0 gives 1.0.
float orc_nvfp4_global_scale(float amax) {
  if (!(amax > 0.0f)) return 1.0f;
  return fl32_div(amax, 2688.0f);
}

// ===========================================================================
// Quantizers
// ===========================================================================

// FP8 E4M3 per-tensor: code = E4M3(fl32(x / scale)) for every element.
void orc_fp8_quantize(const uint16_t* x, size_t n, float scale, uint8_t* codes) {
  if (!(scale > 0.0f) || !std::isfinite(scale)) die("fp8_quantize: bad scale");
  for (size_t i = 0; i < n; ++i) {
    float xf = (float)bf16_value(x[i]);
    codes[i] = e4m3_encode(fl32_div(xf, scale));
  }
}

// NVFP4: blocks of 16 consecutive elements along the last dimension
// ([MO-714]: block_sizes={-1: 16}), a dynamic E4M3 block scale per block
// ([MO-714]: 'type': 'dynamic', 'scale_bits': (4, 3)) and the fp32 global
// scale g.  Per block, in this order:
//   bamax = max |x_i|
//   sc    = E4M3( fl32( fl32(bamax / 6) / g ) )
//   es    = fl32( dec(sc) * g )          (the quantized block scale, in fp32)
//   code_i = E2M1( fl32(x_i / es) )      (all codes 0 when es == 0)
// Codes are packed two per byte, element 2i in the low nibble.
// x is [rows][D] bf16; codes [rows][D/2]; bscales [rows][D/16].
void orc_nvfp4_quantize(const uint16_t* x, size_t rows, int D, float g,
                        uint8_t* codes, uint8_t* bscales) {
  if (D % 16 != 0) die("nvfp4_quantize: D % 16 != 0");
  if (!(g > 0.0f) || !std::isfinite(g)) die("nvfp4_quantize: bad global scale");
  for (size_t r = 0; r < rows; ++r) {
    const uint16_t* xr = x + r * (size_t)D;
    uint8_t* cr = codes + r * (size_t)(D / 2);
    uint8_t* sr = bscales + r * (size_t)(D / 16);
    for (int b = 0; b < D / 16; ++b) {
      float v[16];
      float bamax = 0.0f;
      for (int i = 0; i < 16; ++i) {
        v[i] = (float)bf16_value(xr[b * 16 + i]);
        bamax = std::max(bamax, std::fabs(v[i]));
      }
      uint8_t sc = e4m3_encode(fl32_div(fl32_div(bamax, 6.0f), g));
      float dsc = (float)e4m3_decode(sc);
      float es = fl32_mul(dsc, g);
      sr[b] = sc;
      uint8_t nib[16];
      for (int i = 0; i < 16; ++i)
        nib[i] = (es == 0.0f) ? 0 : e2m1_encode(fl32_div(v[i], es));
      for (int i = 0; i < 8; ++i)
        cr[b * 8 + i] = (uint8_t)(nib[2 * i] | (nib[2 * i + 1] << 4));
    }
  }
}

// ===========================================================================
// Per-kv-head static scales -- [CT-436] "Add support for 'attn_head' strategy"
// (kv-cache recipe: num_bits 8, type float, symmetric, static_minmax observer,
// strategy "attn_head"): one scale per attention head instead of one per
// tensor.  For the KV cache the head is the kv head.  Reading used here: the
// amax of kv head h runs over every token and dim of that head in the tensor
// (K and V separately); its scale is the per-tensor formula applied to that
// amax, and each element is quantized with its head's scale.
//   x [rows][H][D] bf16 (rows = the tensor's tokens).
// ===========================================================================

// amax[h] = max |x[r][h][d]| over r and d.
void orc_head_amax_bf16(const uint16_t* x, size_t rows, int H, int D, float* amax) {
  for (int h = 0; h < H; ++h) {
    double m = 0.0;
    for (size_t r = 0; r < rows; ++r)
      for (int d = 0; d < D; ++d) {
        double v = std::fabs(bf16_value(x[(r * H + h) * (size_t)D + d]));
        if (std::isnan(v)) die("head_amax: NaN input");
        if (v > m) m = v;
      }
    amax[h] = (float)m;
  }
}

// FP8: codes[r][h][d] = E4M3(fl32(x[r][h][d] / scales[h])).
void orc_fp8_quantize_heads(const uint16_t* x, size_t rows, int H, int D,
                            const float* scales, uint8_t* codes) {
  for (size_t r = 0; r < rows; ++r)
    for (int h = 0; h < H; ++h) {
      const float s = scales[h];
      if (!(s > 0.0f) || !std::isfinite(s)) die("fp8_quantize_heads: bad scale");
      for (int d = 0; d < D; ++d) {
        size_t i = (r * H + h) * (size_t)D + d;
        codes[i] = e4m3_encode(fl32_div((float)bf16_value(x[i]), s));
      }
    }
}

// NVFP4 with a global scale per kv head: the block quantizer of
// orc_nvfp4_quantize on each head's rows with g = gs[h].
// codes [rows][H][D/2], bscales [rows][H][D/16].
void orc_nvfp4_quantize(const uint16_t* x, size_t rows, int D, float g,
                        uint8_t* codes, uint8_t* bscales);
void orc_nvfp4_quantize_heads(const uint16_t* x, size_t rows, int H, int D,
                              const float* gs, uint8_t* codes, uint8_t* bscales) {
  for (size_t r = 0; r < rows; ++r)
    for (int h = 0; h < H; ++h) {
      size_t row = r * H + h;
      orc_nvfp4_quantize(x + row * (size_t)D, 1, D, gs[h], codes + row * (size_t)(D / 2),
                         bscales + row * (size_t)(D / 16));
    }
}

// Dequantization (the fake-quant meaning of a stored code, [MO-714] "fake"):
//   FP8:   x^ = dec(code) * scale
//   NVFP4: x^ = dec(e2m1) * dec(sc) * g
// Both products are exact in double.
void orc_fp8_dequant(const uint8_t* codes, size_t n, float scale, double* out) {
  for (size_t i = 0; i < n; ++i) out[i] = e4m3_decode(codes[i]) * (double)scale;
}

void orc_nvfp4_dequant(const uint8_t* codes, const uint8_t* bscales, size_t rows,
                       int D, float g, double* out) {
  for (size_t r = 0; r < rows; ++r) {
    for (int d = 0; d < D; ++d) {
      uint8_t byte = codes[r * (size_t)(D / 2) + d / 2];
      uint8_t nib = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      double sc = e4m3_decode(bscales[r * (size_t)(D / 16) + d / 16]);
      out[r * (size_t)D + d] = e2m1_decode(nib) * sc * (double)g;
    }
  }
}

// ===========================================================================
// Attention -- [MO-1832] split-KV decode notes.
// ===========================================================================

// Chunk j of s over a sequence of L tokens: the chunk length is ceil(L / s)
// rounded up to a multiple of 16 tokens; chunk j covers [j*c, min((j+1)*c, L))
// and is empty when j*c >= L.
void orc_chunk(int L, int s, int j, int* start, int* end) {
  if (s < 1 || L < 0) die("chunk: bad arguments");
  long c = ((long)L + s - 1) / s;
  c = (c + 15) / 16 * 16;
  long st = (long)j * c, en = std::min<long>((long)(j + 1) * c, L);
  if (st > L) st = L;
  if (en < st) en = st;
  *start = (int)st;
  *end = (int)en;
}

// Exact softmax attention for one query over L keys (plain definition):
//   S_i = sm_scale * q . k_i,  w_i = exp(S_i - max S) / sum_j exp(S_j - max S)
//   out = sum_i w_i v_i,  lse = log sum_i exp(S_i)   (natural log)
// L == 0 gives out = 0 and lse = -inf.
void orc_attention_exact(const double* q, const double* k, const double* v,
                         int L, int Dqk, int Dv, double sm_scale,
                         double* out, double* lse) {
  for (int d = 0; d < Dv; ++d) out[d] = 0.0;
  if (L == 0) { *lse = -INFINITY; return; }
  std::vector<double> S(L);
  double m = -INFINITY;
  for (int i = 0; i < L; ++i) {
    S[i] = sm_scale * dot(q, k + (size_t)i * Dqk, Dqk);
    m = std::max(m, S[i]);
  }
  double l = 0.0;
  for (int i = 0; i < L; ++i) l += std::exp(S[i] - m);
  for (int i = 0; i < L; ++i) {
    double w = std::exp(S[i] - m) / l;
    const double* vi = v + (size_t)i * Dv;
    for (int d = 0; d < Dv; ++d) out[d] += w * vi[d];
  }
  *lse = m + std::log(l);
}

// Partial over keys [start, end): o = normalized weighted V over the chunk,
// lse = log of the chunk's softmax denominator (natural log, including the
// chunk max).  An empty chunk gives o = 0, lse = -inf.
void orc_attention_partial(const double* q, const double* k, const double* v,
                           int start, int end, int Dqk, int Dv, double sm_scale,
                           double* o, double* lse) {
  orc_attention_exact(q, k + (size_t)start * Dqk, v + (size_t)start * Dv,
                      end - start, Dqk, Dv, sm_scale, o, lse);
}

// FP8-probability partial -- [VLLM-15734]: softmax(QK^T) quantized to FP8 in
// the attention loop with a prob scale.  Reading used here: within a chunk,
// p~_i = exp(S_i - m) with m the chunk max, computed and rounded to fp32;
// the weight that multiplies V is p_q = dec(E4M3(fl32(p~ / prob_scale))) *
// prob_scale; the denominator sums the unquantized p~.
//   o = sum p_q v / sum p~,  lse = m + log(sum p~)
void orc_attention_partial_probq(const double* q, const double* k, const double* v,
                                 int start, int end, int Dqk, int Dv,
                                 double sm_scale, float prob_scale,
                                 double* o, double* lse) {
  for (int d = 0; d < Dv; ++d) o[d] = 0.0;
  int L = end - start;
  if (L <= 0) { *lse = -INFINITY; return; }
  std::vector<double> S(L);
  double m = -INFINITY;
  for (int i = 0; i < L; ++i) {
    S[i] = sm_scale * dot(q, k + (size_t)(start + i) * Dqk, Dqk);
    m = std::max(m, S[i]);
  }
  double l = 0.0;
  for (int i = 0; i < L; ++i) {
    float pt = (float)std::exp(S[i] - m);
    l += (double)pt;
    double pq = e4m3_decode(e4m3_encode(fl32_div(pt, prob_scale))) * (double)prob_scale;
    const double* vi = v + (size_t)(start + i) * Dv;
    for (int d = 0; d < Dv; ++d) o[d] += pq * vi[d];
  }
  for (int d = 0; d < Dv; ++d) o[d] /= l;
  *lse = m + std::log(l);
}

// Combine of s partials ([MO-1832]: "a small combine kernel merges the s
// partials"): M = max_j lse_j, w_j = exp(lse_j - M),
// out = sum_j w_j o_j / sum_j w_j.  Partials with lse = -inf are skipped;
// if all are empty the output is 0.
void orc_combine(const double* o_parts, const double* lse, int s, int Dv, double* out) {
  for (int d = 0; d < Dv; ++d) out[d] = 0.0;
  double M = -INFINITY;
  for (int j = 0; j < s; ++j) M = std::max(M, lse[j]);
  if (M == -INFINITY) return;
  double wsum = 0.0;
  for (int j = 0; j < s; ++j) {
    if (lse[j] == -INFINITY) continue;
    double w = std::exp(lse[j] - M);
    wsum += w;
    for (int d = 0; d < Dv; ++d) out[d] += w * o_parts[(size_t)j * Dv + d];
  }
  for (int d = 0; d < Dv; ++d) out[d] /= wsum;
}

// Output quantization to E4M3 ([VLLM-15734] _out_scale):
// code = E4M3(fl32(fl32(o) / out_scale)).  The fp32 rounding of o is where
// the GPU's fp32 result enters; the oracle rounds its fp64 value once.
void orc_fp8_output(const double* o, size_t n, float out_scale, uint8_t* codes) {
  for (size_t i = 0; i < n; ++i) codes[i] = e4m3_encode(fl32_div((float)o[i], out_scale));
}

// ===========================================================================
// Batched decode over dequantized caches (threaded over (b, hq)).
//   q     [B][Hq][Dqk]          double
//   khat  [B][Hkv][Lcap][Dqk]   double (dequantized keys)
//   vhat  [B][Hkv][Lcap][Dv]    double (dequantized values)
//   seq_lens[B]
//   kv head of query head hq = hq / (Hq / Hkv)   (contiguous groups)
// mode 0: exact attention (split count does not matter);
// mode 1: FP8-probability reading above, with s splits and combine.
// out [B][Hq][Dv], lse [B][Hq]
// ===========================================================================
void orc_decode_batch(const double* q, const double* khat, const double* vhat,
                      int B, int Hq, int Hkv, int Lcap, const int* seq_lens,
                      int Dqk, int Dv, double sm_scale, int mode, int s,
                      float prob_scale, double* out, double* lse, int nthreads) {
  if (Hkv <= 0 || Hq % Hkv != 0) die("decode_batch: Hq % Hkv != 0");
  int G = Hq / Hkv;
  int units = B * Hq;
  if (nthreads < 1) nthreads = 1;
  std::vector<std::thread> th;
  for (int t = 0; t < nthreads; ++t) {
    th.emplace_back([&, t]() {
      std::vector<double> op((size_t)std::max(s, 1) * Dv), lp(std::max(s, 1));
      for (int u = t; u < units; u += nthreads) {
        int b = u / Hq, hq = u % Hq, hk = hq / G;
        int L = seq_lens[b];
        if (L < 0 || L > Lcap) die("decode_batch: bad seq_len");
        const double* qb = q + (size_t)u * Dqk;
        const double* kb = khat + ((size_t)b * Hkv + hk) * (size_t)Lcap * Dqk;
        const double* vb = vhat + ((size_t)b * Hkv + hk) * (size_t)Lcap * Dv;
        double* ob = out + (size_t)u * Dv;
        if (mode == 0) {
          orc_attention_exact(qb, kb, vb, L, Dqk, Dv, sm_scale, ob, lse + u);
        } else {
          for (int j = 0; j < s; ++j) {
            int st, en;
            orc_chunk(L, s, j, &st, &en);
            orc_attention_partial_probq(qb, kb, vb, st, en, Dqk, Dv, sm_scale,
                                        prob_scale, op.data() + (size_t)j * Dv, &lp[j]);
          }
          orc_combine(op.data(), lp.data(), s, Dv, ob);
          double M = -INFINITY, acc = 0.0;
          for (int j = 0; j < s; ++j) M = std::max(M, lp[j]);
          if (M == -INFINITY) lse[u] = -INFINITY;
          else {
            for (int j = 0; j < s; ++j) if (lp[j] != -INFINITY) acc += std::exp(lp[j] - M);
            lse[u] = M + std::log(acc);
          }
        }
      }
    });
  }
  for (auto& x : th) x.join();
}

}  // extern "C"
