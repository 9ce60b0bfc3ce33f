// Device-side building blocks for the sm_103a kernels: format conversions,
// warp-level MMA, mbarriers and TMA (bulk async copies).  Inline PTX only.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace kvq {

// ---------------------------------------------------------------------------
// Format conversions (hardware cvt instructions of sm_100+ family targets)
// ---------------------------------------------------------------------------

// Two fp32 -> packed E4M3 pair, round to nearest even, saturating to +-448
// (NaN stays NaN).  `lo` lands in bits 0..7, `hi` in bits 8..15.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Packed E4M3 pair (bits 0..15) -> f16x2 (exact: every E4M3 value is an f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  uint32_t r;
  uint16_t h = (uint16_t)(v & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
  return r;
}

// Four E4M3 codes (bytes 0..3 of w) -> two f16x2: lo = (b0, b1), hi = (b2, b3).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Eight fp32 -> eight E2M1 nibbles packed in a u32 (element i in nibble i),
// round to nearest even, saturating to +-6.
__device__ __forceinline__ uint32_t f32x8_to_e2m1x8(const float* x) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]),
        "f"(x[7]));
  return r;
}

// Four bytes, each an E2M1 pair (low nibble -> low half), to four f16x2.
// Exact: every E2M1 value is an f16.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t v, uint32_t& o0, uint32_t& o1,
                                                  uint32_t& o2, uint32_t& o3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(v));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// fp32 pair -> f16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t v) {
  __half2 h = *reinterpret_cast<__half2*>(&v);
  return __half22float2(h);
}

// bf16 bits -> fp32 (exact)
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// 2^n as an fp32, for -126 <= n <= 127 (a normal number: exact).
__device__ __forceinline__ float exp2i(int n) { return __uint_as_float((uint32_t)(n + 127) << 23); }

// Power-of-two prescale of a bf16 query head for the f16 tensor-core
// operand.  `bits` is the head's largest |q| as bf16 magnitude bits.  The
// result e puts that element into [2^14, 2^15) (0 for an all-zero head; at
// most 127, reached only when the largest |q| is below 2^-113): every element
// of the head within 2^-31 of its largest then converts to f16 exactly (bf16
// keeps 8 significant bits, f16 11 down to 2^-14 and 8 down to 2^-17), and
// smaller ones are rounded at the f16 subnormal step, at most 2^-40 of the
// head's largest |q| -- whatever q's magnitude.  x * 2^e is one exact fp32
// product (e in [-113, 127]); the score scale takes 2^-e.
__device__ __forceinline__ int q_prescale_exp(uint32_t bits) {
  if (bits == 0) return 0;
  const int E = (int)(bits >> 7);
  const int lg = E > 0 ? E - 127 : (31 - __clz((int)bits)) - 133;   // floor(log2 |q|max)
  return min(14 - lg, 127);
}

// x * 2^e for e in [-252, 254], as two exact power-of-two products (only a
// result below the fp32 normal range is rounded).
__device__ __forceinline__ float scale_pow2(float x, int e) {
  const int e1 = e >> 1;
  return (x * exp2i(e1)) * exp2i(e - e1);
}

// ---------------------------------------------------------------------------
// Warp-level tensor-core MMA: D(16x8,f32) += A(16x16) * B(16x8)
// Fragment layout (g = lane >> 2, t = lane & 3):
//   A: a0 = (row g,   col 2t..2t+1)  a1 = (row g+8, col 2t..2t+1)
//      a2 = (row g,   col 2t+8..9)   a3 = (row g+8, col 2t+8..9)
//   B: b0 = (row 2t..2t+1, col g)    b1 = (row 2t+8..9, col g)
//   C: c0,c1 = (row g, col 2t..2t+1) c2,c3 = (row g+8, col 2t..2t+1)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_f16(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 b16 matrix across the warp: lane (g, t) holds row g,
// columns 2t, 2t+1 before and after.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// 2^x (hardware approximation, flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// D(16x8,f32) += A(16x32) * B(32x8) on E4M3 codes (products exact, fp32
// accumulation).  Fragments of 8-bit elements, 4 per register:
//   A: a0 = (row g, cols 4t..4t+3)   a1 = (row g+8, cols 4t..4t+3)
//      a2 = (row g, cols 4t+16..19)  a3 = (row g+8, cols 4t+16..19)
//   B: b0 = (rows 4t..4t+3, col g)   b1 = (rows 4t+16..19, col g)
//   C: as for m16n8k16.
__device__ __forceinline__ void mma_e4m3(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// Shared memory, mbarriers, TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy accesses to shared memory before
// its later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for the phase with the given parity to complete.  Gives up
// after ~0.25 s (or 2^28 polls) and returns false; callers record the error
// and leave their loops.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0; i < (1u << 28); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0 && globaltimer_ns() - t0 > 250000000ull) return false;
  }
  return false;
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------------------------
// Thread-block clusters: barrier and distributed shared memory
// ---------------------------------------------------------------------------
// Every thread of every CTA of the cluster: this thread's earlier writes
// (shared memory included) become visible to the cluster's later reads.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The address in CTA `rank`'s shared memory of this CTA's shared address.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds8(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel in the stream runs; it
// must wait here before reading anything that kernel produces.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next (programmatically serialized) kernel in the stream launch.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// fl32(p / y) for the FP8 probabilities, with y = prob_scale known per call.
// fast: z = RN(1/y) precomputed; q0 = RN(p z) has a relative error of at most
// about 2^-23, the remainder r = RN(p - q0 y) is then accurate to 2^-24, and
// RN(q0 + r z) = RN(p/y + h) with |h| below 2^-45 (p/y).  The result is the
// correctly rounded quotient except where p/y lies that close to the midpoint
// of two fp32 numbers, and is always within one fp32 step of it (the
// correction step of P. Markstein, "Computation of elementary functions on the
// IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990; division by
// a divisor known in advance: N. Brisebarre, J.-M. Muller, S. K. Raina, IEEE
// Trans. Computers 53(8), 2004).  The host enables it for a prob_scale only
// after checking that it returns the correctly rounded quotient for every p
// whose quotient lies near an E4M3 rounding boundary, so that the E4M3 codes
// equal those of the IEEE division for all p; otherwise the IEEE division.
__device__ __forceinline__ float prob_quotient(float p, float y, float z, bool fast) {
  if (!fast) return __fdiv_rn(p, y);
  const float q0 = __fmul_rn(p, z);
  const float r = __fmaf_rn(-q0, y, p);
  return __fmaf_rn(r, z, q0);
}

__device__ __forceinline__ void record_error(int32_t* flag, int bits) {
  if (flag) atomicOr(flag, bits);
}

}  // namespace kvq
