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
// Every fp32 step is one IEEE operation (__fdiv_rn / __fmul_rn; this file is
// built without fast-math), and the grid rounding is the hardware cvt with
// round-to-nearest-even and saturation, so codes are bit-exact by contract.
// The work is HBM-bound (2 bytes in, 1 or 0.5625 bytes out per element):
// one thread per 8 (FP8) or 16 (NVFP4) elements with 16-byte loads.

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
  const int page = __ldg(a.block_table + (size_t)b * a.max_pages + pos / a.ps);
  if (page < 0 || page >= a.num_pages) return -1;
  return ((long)page * a.Hkv + h) * a.ps + pos % a.ps;
}

// grid.y = 0: K, 1: V (or the MLA rope keys)
__global__ void __launch_bounds__(256) append_fp8_kernel(const AppendArgs a) {
  griddep_launch_dependents();   // the decode kernel may launch now (it waits for us)
  const int per_row = a.D / 8;
  const size_t rows = (size_t)a.batch * a.T * a.Hkv;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows * per_row) return;
  const size_t row = i / per_row;
  const int part = (int)(i % per_row);
  const int h = (int)(row % a.Hkv);
  const size_t bt = row / a.Hkv;
  const int tt = (int)(bt % a.T), b = (int)(bt / a.T);
  const bool isv = blockIdx.y == 1;
  const uint16_t* src = isv ? a.v_new : a.k_new;
  // the row is read while the block-table lookup is in flight
  const uint4 x = *reinterpret_cast<const uint4*>(src + row * a.D + part * 8);
  const long dst_row = cache_row(a, b, __ldg(a.start_pos + b) + tt, h);
  if (dst_row < 0) return;
  uint8_t* dst = isv ? a.v_codes : a.k_codes;
  const float s = isv ? a.v_scale : a.k_scale;
  float f[8];
  bf16x8_to_f32(x, f);
  uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(f[0], s), __fdiv_rn(f[1], s)) |
                (f32x2_to_e4m3x2(__fdiv_rn(f[2], s), __fdiv_rn(f[3], s)) << 16);
  uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(f[4], s), __fdiv_rn(f[5], s)) |
                (f32x2_to_e4m3x2(__fdiv_rn(f[6], s), __fdiv_rn(f[7], s)) << 16);
  *reinterpret_cast<uint2*>(dst + dst_row * a.D + part * 8) = make_uint2(lo, hi);
}

__device__ __forceinline__ void nvfp4_block(const float* f, float g, uint32_t& w0, uint32_t& w1,
                                            uint8_t& sc_out) {
  float bamax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) bamax = fmaxf(bamax, fabsf(f[i]));
  const float scf = __fdiv_rn(__fdiv_rn(bamax, 6.0f), g);
  const uint32_t sc = f32x2_to_e4m3x2(scf, 0.f) & 0xFFu;
  const float dsc = unpack_f16x2(e4m3x2_to_f16x2(sc)).x;   // exact decode
  const float es = __fmul_rn(dsc, g);
  sc_out = (uint8_t)sc;
  if (es == 0.f) {
    w0 = w1 = 0u;
    return;
  }
  float q[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) q[i] = __fdiv_rn(f[i], es);
  w0 = f32x8_to_e2m1x8(q);
  w1 = f32x8_to_e2m1x8(q + 8);
}

__global__ void __launch_bounds__(256) append_nvfp4_kernel(const AppendArgs a) {
  griddep_launch_dependents();   // the decode kernel may launch now (it waits for us)
  const int per_row = a.D / 16;
  const size_t rows = (size_t)a.batch * a.T * a.Hkv;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows * per_row) return;
  const size_t row = i / per_row;
  const int blk = (int)(i % per_row);
  const int h = (int)(row % a.Hkv);
  const size_t bt = row / a.Hkv;
  const int tt = (int)(bt % a.T), b = (int)(bt / a.T);
  const bool isv = blockIdx.y == 1;
  const uint16_t* src = (isv ? a.v_new : a.k_new) + row * a.D + blk * 16;
  // the block is read while the block-table lookup is in flight
  const uint4 x0 = *reinterpret_cast<const uint4*>(src);
  const uint4 x1 = *reinterpret_cast<const uint4*>(src + 8);
  const long dst_row = cache_row(a, b, __ldg(a.start_pos + b) + tt, h);
  if (dst_row < 0) return;
  float f[16];
  bf16x8_to_f32(x0, f);
  bf16x8_to_f32(x1, f + 8);
  uint32_t w0, w1;
  uint8_t sc;
  nvfp4_block(f, isv ? a.v_scale : a.k_scale, w0, w1, sc);
  uint8_t* codes = isv ? a.v_codes : a.k_codes;
  uint8_t* scales = isv ? a.v_bscale : a.k_bscale;
  *reinterpret_cast<uint2*>(codes + dst_row * (a.D / 2) + blk * 8) = make_uint2(w0, w1);
  scales[dst_row * (a.D / 16) + blk] = sc;
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

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t st) {
  const size_t rows = (size_t)a.batch * a.T * a.Hkv;
  if (rows == 0) return cudaSuccess;
  const int per = a.fmt == kFmtFp8 ? a.D / 8 : a.D / 16;
  const size_t threads = rows * per;
  dim3 grid((unsigned)((threads + 255) / 256), a.has_v ? 2 : 1);
  if (a.fmt == kFmtFp8)
    append_fp8_kernel<<<grid, 256, 0, st>>>(a);
  else
    append_nvfp4_kernel<<<grid, 256, 0, st>>>(a);
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
