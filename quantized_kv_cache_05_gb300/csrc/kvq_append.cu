// Quantize-on-append of K/V rows into the cache, the amax reduction that
// calibrates the static scales, and elementwise encoders (sm_103a).
//
// FP8 E4M3 per tensor (compressed-tensors PR 436, kv_cache_scheme: 8-bit
// float, symmetric, per tensor, static): code = E4M3(fl32(x / scale)).
// NVFP4 (Model-Optimizer PR 714, Testing: "(2, 1) bit ... block_sizes={-1:
// 16, 'type': 'dynamic', 'scale_bits': (4, 3)}"): per 16-element block along
// head_dim, sc = E4M3(fl32(fl32(bamax / 6) / g)), es = fl32(dec(sc) * g),
// code = E2M1(fl32(x / es)).
//
// Every fp32 step gives the IEEE result's code (the element divisions by a
// reciprocal with a guarded fallback to the IEEE division, see
// quotient_for_code; the block-scale steps are IEEE operations; this file is
// built without fast-math), and the grid rounding is the hardware cvt with
// round-to-nearest-even and saturation, so codes are bit-exact by contract.
// The work is HBM-bound (2 bytes in, 1 or 0.5625 bytes out per element):
// one thread per 8 (FP8) or 16 (NVFP4) elements with 16-byte loads, rows of
// a request spread over blocks without 64-bit index divisions.

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

__device__ __forceinline__ void bf16x8_to_f32(uint4 v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
    f[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
  }
}

// Cache row of (request b, position pos, kv head h), or -1 when the position
// is outside the request's block table.
__device__ __forceinline__ long cache_row(const AppendArgs& a, int b, int pos, int h) {
  if (pos < 0 || pos >= a.max_pages * a.ps) return -1;
  const int page = __ldg(a.block_table + (size_t)b * a.max_pages + (unsigned)pos / (unsigned)a.ps);
  if (page < 0 || page >= a.num_pages) return -1;
  return ((long)page * a.Hkv + h) * a.ps + (unsigned)pos % (unsigned)a.ps;
}

// fl32(x_i / s) for a grid encoder whose rounding boundaries have at most
// 24 - log2(lowmask + 1) significant bits (E4M3: 5, lowmask 2^19 - 1; E2M1: 3,
// lowmask 2^21 - 1), for N elements.  With z = RN(1/s), q0 = RN(x z), r =
// RN(x - q0 s) and q = RN(q0 + r z) is within one fp32 step of RN(x/s) (the
// correction step of P. Markstein, IBM J. Res. Dev. 34(1), 1990).  Two
// adjacent fp32 numbers round to different codes only if one of them is a
// boundary, whose low fraction bits are zero; so where some q has low bits 0,
// 1 or all ones, ((bits + 1) & lowmask) <= 2 -- which also holds for
// infinities and the canonical NaN -- the IEEE division gives all N.  Either
// way every code equals the code of the correctly rounded quotient.
template <int N>
struct Floats {
  float v[N];
};

// The IEEE quotients of a whole group: out of line, so that the rarely taken
// fallback stays off the common path (not merged into it as predicated code).
template <int N>
__device__ __noinline__ Floats<N> ieee_quotients(Floats<N> x, float s) {
#pragma unroll
  for (int i = 0; i < N; ++i) x.v[i] = __fdiv_rn(x.v[i], s);
  return x;
}

template <int N>
__device__ __forceinline__ void quotients_for_codes(float (&x)[N], float s, float z,
                                                    uint32_t lowmask) {
  float q[N];
  uint32_t m = 0xFFFFFFFFu;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float q0 = __fmul_rn(x[i], z);
    const float r = __fmaf_rn(-q0, s, x[i]);
    q[i] = __fmaf_rn(r, z, q0);
    m = min(m, (__float_as_uint(q[i]) + 1u) & lowmask);
  }
  if (m <= 2u) {
    Floats<N> in;
#pragma unroll
    for (int i = 0; i < N; ++i) in.v[i] = x[i];
    const Floats<N> out = ieee_quotients<N>(in, s);
#pragma unroll
    for (int i = 0; i < N; ++i) x[i] = out.v[i];
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) x[i] = q[i];
  }
}

constexpr uint32_t kE4m3Low = (1u << 19) - 1;   // E4M3 boundaries: <= 5 significant bits
constexpr uint32_t kE2m1Low = (1u << 21) - 1;   // E2M1 boundaries: <= 3 significant bits

// Thread layout of the append kernels: threadIdx.x = the thread's part of a
// row (8 FP8 or 16 NVFP4 elements); token tt = blockIdx.x * blockDim.y +
// threadIdx.y, kv head h = blockIdx.y, request b = blockIdx.z >> 1 (K, or V
// when blockIdx.z is odd; MLA: b = blockIdx.z, K only) -- no index division.
struct RowIdx {
  int b, tt, h, part;
  bool isv, ok;
};
__device__ __forceinline__ RowIdx row_index(const AppendArgs& a) {
  RowIdx r;
  r.part = threadIdx.x;
  r.tt = blockIdx.x * blockDim.y + threadIdx.y;
  r.h = blockIdx.y;
  r.b = a.has_v ? (int)(blockIdx.z >> 1) : (int)blockIdx.z;
  r.isv = a.has_v && (blockIdx.z & 1) != 0;
  r.ok = r.tt < a.T;
  return r;
}

__global__ void __launch_bounds__(256) append_fp8_kernel(const AppendArgs a) {
  griddep_launch_dependents();   // the decode kernel may launch now (it waits for us)
  const RowIdx ix = row_index(a);
  if (!ix.ok) return;
  const size_t row = ((size_t)ix.b * a.T + ix.tt) * a.Hkv + ix.h;
  const uint16_t* src = ix.isv ? a.v_new : a.k_new;
  // the row is read while the block-table lookup is in flight
  const uint4 x = *reinterpret_cast<const uint4*>(src + row * a.D + ix.part * 8);
  const long dst_row = cache_row(a, ix.b, __ldg(a.start_pos + ix.b) + ix.tt, ix.h);
  if (dst_row < 0) return;
  uint8_t* dst = ix.isv ? a.v_codes : a.k_codes;
  // the tensor's scale, or kv head h's (then its reciprocal here)
  const float* hs = ix.isv ? a.v_hs : a.k_hs;
  const float s = hs ? __ldg(hs + ix.h) : (ix.isv ? a.v_scale : a.k_scale);
  const float z = hs ? __frcp_rn(s) : (ix.isv ? a.v_recip : a.k_recip);
  float f[8];
  bf16x8_to_f32(x, f);
  quotients_for_codes<8>(f, s, z, kE4m3Low);
  const uint32_t lo = f32x2_to_e4m3x2(f[0], f[1]) | (f32x2_to_e4m3x2(f[2], f[3]) << 16);
  const uint32_t hi = f32x2_to_e4m3x2(f[4], f[5]) | (f32x2_to_e4m3x2(f[6], f[7]) << 16);
  *reinterpret_cast<uint2*>(dst + dst_row * a.D + ix.part * 8) = make_uint2(lo, hi);
}

__device__ __forceinline__ void nvfp4_block(float (&f)[16], float g, uint32_t& w0, uint32_t& w1,
                                            uint8_t& sc_out) {
  float bamax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) bamax = fmaxf(bamax, fabsf(f[i]));
  // the block scale's two divisions stay IEEE (their fp32 results feed on)
  const float scf = __fdiv_rn(__fdiv_rn(bamax, 6.0f), g);
  const uint32_t sc = f32x2_to_e4m3x2(scf, 0.f) & 0xFFu;
  const float dsc = unpack_f16x2(e4m3x2_to_f16x2(sc)).x;   // exact decode
  const float es = __fmul_rn(dsc, g);
  sc_out = (uint8_t)sc;
  if (es == 0.f) {
    w0 = w1 = 0u;
    return;
  }
  quotients_for_codes<16>(f, es, __frcp_rn(es), kE2m1Low);
  w0 = f32x8_to_e2m1x8(f);
  w1 = f32x8_to_e2m1x8(f + 8);
}

__global__ void __launch_bounds__(256) append_nvfp4_kernel(const AppendArgs a) {
  griddep_launch_dependents();   // the decode kernel may launch now (it waits for us)
  const RowIdx ix = row_index(a);
  if (!ix.ok) return;
  const size_t row = ((size_t)ix.b * a.T + ix.tt) * a.Hkv + ix.h;
  const uint16_t* src = (ix.isv ? a.v_new : a.k_new) + row * a.D + ix.part * 16;
  // the block is read while the block-table lookup is in flight
  const uint4 x0 = *reinterpret_cast<const uint4*>(src);
  const uint4 x1 = *reinterpret_cast<const uint4*>(src + 8);
  const long dst_row = cache_row(a, ix.b, __ldg(a.start_pos + ix.b) + ix.tt, ix.h);
  if (dst_row < 0) return;
  float f[16];
  bf16x8_to_f32(x0, f);
  bf16x8_to_f32(x1, f + 8);
  uint32_t w0, w1;
  uint8_t sc;
  const float* hs = ix.isv ? a.v_hs : a.k_hs;   // kv head h's global scale, if given
  nvfp4_block(f, hs ? __ldg(hs + ix.h) : (ix.isv ? a.v_scale : a.k_scale), w0, w1, sc);
  uint8_t* codes = ix.isv ? a.v_codes : a.k_codes;
  uint8_t* scales = ix.isv ? a.v_bscale : a.k_bscale;
  *reinterpret_cast<uint2*>(codes + dst_row * (a.D / 2) + ix.part * 8) = make_uint2(w0, w1);
  scales[dst_row * (a.D / 16) + ix.part] = sc;
}

// MLA rope keys: plain bf16 copy into k_pe [page][ps][rope] (Hkv = 1).
__global__ void __launch_bounds__(256) append_rope_kernel(const AppendArgs a) {
  griddep_launch_dependents();   // the decode kernel may launch now (it waits for us)
  const int per_row = a.rope / 8;
  const size_t rows = (size_t)a.batch * a.T;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows * per_row) return;
  const size_t row = i / per_row;
  const int part = (int)(i % per_row);
  const int tt = (int)(row % a.T), b = (int)(row / a.T);
  const long dst_row = cache_row(a, b, __ldg(a.start_pos + b) + tt, 0);
  if (dst_row < 0) return;
  *reinterpret_cast<uint4*>(a.k_pe + dst_row * a.rope + part * 8) =
      *reinterpret_cast<const uint4*>(a.kpe_new + row * a.rope + part * 8);
}

// amax = max |x| over bf16; non-negative floats order like their bit patterns.
__global__ void __launch_bounds__(256) amax_kernel(const uint16_t* x, size_t n, float* out) {
  uint32_t m = 0;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const bool vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
  size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  size_t nvec = vec ? n / 8 : 0;
  for (size_t i = i0; i < nvec; i += stride) {
    const uint4 v = reinterpret_cast<const uint4*>(x)[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      m = max(m, (w[k] & 0x7FFFu) << 16);
      m = max(m, (w[k] >> 16 & 0x7FFFu) << 16);
    }
  }
  for (size_t i = nvec * 8 + i0; i < n; i += stride) m = max(m, ((uint32_t)x[i] & 0x7FFFu) << 16);
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0 && m != 0) atomicMax(reinterpret_cast<unsigned int*>(out), m);
}

__global__ void __launch_bounds__(256) encode_kernel(int kind, const float* x, uint8_t* out,
                                                     size_t n) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float v = x[i];
    if (kind == 0) {
      out[i] = (uint8_t)(f32x2_to_e4m3x2(v, 0.f) & 0xFFu);
    } else {
      float q[8] = {v, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      out[i] = (uint8_t)(f32x8_to_e2m1x8(q) & 0xFu);
    }
  }
}

// FP8 quantizer of a bf16 array, 8 elements per thread (the append's
// arithmetic); s per tensor or per head of head_len elements.
__global__ void __launch_bounds__(256) quantize_fp8_kernel(const uint16_t* x, size_t n8,
                                                           float scale, float recip,
                                                           const float* head_scale, int head_len,
                                                           int num_heads, uint8_t* out) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const uint4 v = reinterpret_cast<const uint4*>(x)[i];
    float s = scale, z = recip;
    if (head_scale) {
      s = __ldg(head_scale + (int)((i * 8 / (size_t)head_len) % (size_t)num_heads));
      z = __frcp_rn(s);
    }
    float f[8];
    bf16x8_to_f32(v, f);
    quotients_for_codes<8>(f, s, z, kE4m3Low);
    const uint32_t lo = f32x2_to_e4m3x2(f[0], f[1]) | (f32x2_to_e4m3x2(f[2], f[3]) << 16);
    const uint32_t hi = f32x2_to_e4m3x2(f[4], f[5]) | (f32x2_to_e4m3x2(f[6], f[7]) << 16);
    reinterpret_cast<uint2*>(out)[i] = make_uint2(lo, hi);
  }
}

__global__ void __launch_bounds__(256) encode_prob_kernel(const float* p, uint8_t* out, size_t n,
                                                          float y, float z, int fast) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = (uint8_t)(f32x2_to_e4m3x2(prob_quotient(p[i], y, z, fast != 0), 0.f) & 0xFFu);
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t st) {
  const size_t rows = (size_t)a.batch * a.T * a.Hkv;
  if (rows == 0) return cudaSuccess;
  const int per = a.fmt == kFmtFp8 ? a.D / 8 : a.D / 16;   // threads per row
  const int rpb = per >= 256 ? 1 : 256 / per;               // tokens per block
  const size_t tblocks = ((size_t)a.T + rpb - 1) / rpb;
  if (tblocks > 0x7FFFFFFFu || a.Hkv > 65535 || a.batch > 32767) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)tblocks, (unsigned)a.Hkv, (unsigned)((a.has_v ? 2 : 1) * a.batch));
  const dim3 block((unsigned)per, (unsigned)rpb);
  if (a.fmt == kFmtFp8)
    append_fp8_kernel<<<grid, block, 0, st>>>(a);
  else
    append_nvfp4_kernel<<<grid, block, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.rope == 0) return e;
  const size_t rthreads = (size_t)a.batch * a.T * (a.rope / 8);
  append_rope_kernel<<<(unsigned)((rthreads + 255) / 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_amax_bf16(const uint16_t* x, size_t n, float* out, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float), st);
  if (e != cudaSuccess || n == 0) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  size_t want = (n / 8 + 255) / 256 + 1;
  unsigned blocks = (unsigned)(want < (size_t)sms * 8 ? want : (size_t)sms * 8);
  amax_kernel<<<blocks, 256, 0, st>>>(x, n, out);
  return cudaGetLastError();
}

cudaError_t launch_encode(int kind, const float* x, uint8_t* out, size_t n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  size_t want = (n + 255) / 256;
  unsigned blocks = (unsigned)(want < (size_t)sms * 16 ? want : (size_t)sms * 16);
  encode_kernel<<<blocks, 256, 0, st>>>(kind, x, out, n);
  return cudaGetLastError();
}

}  // namespace kvq

namespace kvq {

cudaError_t launch_encode_prob(const float* p, uint8_t* out, size_t n, float prob_scale,
                               float prob_recip, int prob_fast, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  size_t want = (n + 255) / 256;
  unsigned blocks = (unsigned)(want < (size_t)sms * 16 ? want : (size_t)sms * 16);
  encode_prob_kernel<<<blocks, 256, 0, st>>>(p, out, n, prob_scale, prob_recip, prob_fast);
  return cudaGetLastError();
}

}  // namespace kvq

namespace kvq {

cudaError_t launch_quantize_fp8(const uint16_t* x, size_t n, float scale, float recip,
                                const float* head_scale, int head_len, int num_heads,
                                uint8_t* out, cudaStream_t st) {
  const size_t n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  size_t want = (n8 + 255) / 256;
  unsigned blocks = (unsigned)(want < (size_t)sms * 16 ? want : (size_t)sms * 16);
  quantize_fp8_kernel<<<blocks, 256, 0, st>>>(x, n8, scale, recip, head_scale, head_len,
                                               num_heads, out);
  return cudaGetLastError();
}

}  // namespace kvq
