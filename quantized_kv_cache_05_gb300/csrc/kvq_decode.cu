// Split-KV flash-decode over a quantized KV cache (sm_103a).
//
// Method (Model-Optimizer PR 1832, notes under the latency tables): each
// (request, kv head) sequence is cut into s contiguous chunks; one CTA runs
// the partial softmax (running max, denominator, weighted V) of one chunk for
// all Hq/Hkv query heads of the kv head, and a small combine kernel merges the
// s partials.  FP8 probabilities and FP8 output follow vLLM PR 15734.
//
// GB300 design of the partial kernel
//  * One producer warp streams the chunk's K/V code tiles HBM -> shared
//    memory with TMA (cp.async.bulk.tensor, 16-row boxes = one 16-token page,
//    hardware swizzle) into a 4-stage ring guarded by mbarriers; NVFP4 block
//    scales come by 1-D bulk copies.
//  * Four consumer warps each take one 16-token box per stage.  Codes are
//    decoded in registers straight into tensor-core fragments (E4M3 -> f16 and
//    E2M1 -> f16 with cvt, block scales by f16x2 multiply: all exact), and
//    the scores Q.K^T and the update P.V run on mma.sync m16n8k16 with fp32
//    accumulation.  The query heads of a group are the MMA's 16 rows.
//  * Head-dim order inside a K row is permuted per lane so that each lane's
//    codes come from one 16-byte shared-memory load; Q is loaded with the same
//    permutation.  The token-pair layout the P.V fragment needs is built with
//    byte permutes (FP8) or nibble masks (E2M1).
//  * P is split into an f16 high part and an f16 residual (two MMAs), so the
//    probabilities keep ~22 bits; with FP8 probabilities the E4M3 code itself
//    is the (exact) f16 operand.
//  * Warps merge their (max, sum, O) states through shared memory at the end.
// Every mbarrier wait is bounded; a timeout sets an error bit and the CTA
// writes NaN for its partial instead of hanging.

#include <cfloat>
#include <cmath>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr float kLn2 = 0.6931471805599453f;

template <int FMT, int D>
struct Geom {
  static constexpr int kRow = FMT == kFmtFp8 ? D : D / 2;   // code bytes per token row
  static constexpr int kSRow = FMT == kFmtFp8 ? 0 : D / 16; // scale bytes per token row
  static constexpr int kTileK = kTileTokens * kRow;
  static constexpr int kTileS = kTileTokens * kSRow;
  static constexpr int kStage = 2 * (kTileK + kTileS);
  static constexpr int kBoxK = kBoxTokens * kRow;
  static constexpr int kBoxS = kBoxTokens * kSRow;
  static constexpr int kKSteps = D / 16;                     // MMA k-steps over head_dim
  static constexpr int kNT = D / 8;                          // n-tiles over v_dim
  // physical 16-byte chunk of logical chunk `ch` in row `row` of a box
  __device__ static __forceinline__ int swz(int row, int ch) {
    if constexpr (kRow == 128) return ch ^ (row & 7);
    else return ch ^ ((row >> 1) & 3);                        // 64-byte rows
  }
};

struct Smem {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int abort_flag;
  float m[kConsumerWarps][kMaxGroup];
  float l[kConsumerWarps][kMaxGroup];
  float fac[kConsumerWarps][kMaxGroup];
  float lse[kMaxGroup];
};

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > 250000000ull || i > (1u << 28)) return false;
    }
  }
}

// ---------------------------------------------------------------------------
// K fragments for one n-tile (8 tokens): b[j][0..1] for k-step j.
// Lane (g, t) holds token row `row` (= 8u + g) and head-dim indices
//   d = (D/4) * t + 4 j + {0, 1} (b[j][0]) and + {2, 3} (b[j][1]).
// ---------------------------------------------------------------------------
template <int FMT, int D>
__device__ __forceinline__ void k_frag(uint32_t boxK, uint32_t boxKs, int row, int t,
                                       uint32_t (&b)[D / 16][2]) {
  using Gm = Geom<FMT, D>;
  if constexpr (FMT == kFmtFp8) {
    constexpr int NCH = D / 64;  // 16-byte chunks per lane per row
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      uint4 v = lds128(boxK + row * Gm::kRow + (Gm::swz(row, t * NCH + i) << 4));
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        b[i * 4 + k][0] = e4m3x2_to_f16x2(w[k] & 0xFFFFu);
        b[i * 4 + k][1] = e4m3x2_to_f16x2(w[k] >> 16);
      }
    }
  } else {
    static_assert(D == 128, "NVFP4 decode supports head_dim 128");
    uint4 v = lds128(boxK + row * Gm::kRow + (Gm::swz(row, t) << 4));
    uint32_t sc = lds16(boxKs + row * Gm::kSRow + 2 * t);   // blocks 2t, 2t+1
    uint32_t s2 = e4m3x2_to_f16x2(sc);
    uint32_t s_lo = __byte_perm(s2, 0, 0x1010), s_hi = __byte_perm(s2, 0, 0x3232);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t o0, o1, o2, o3;
      e2m1x8_to_f16x2x4(w[k], o0, o1, o2, o3);
      uint32_t s = k < 2 ? s_lo : s_hi;
      b[2 * k][0] = hmul2(o0, s);
      b[2 * k][1] = hmul2(o1, s);
      b[2 * k + 1][0] = hmul2(o2, s);
      b[2 * k + 1][1] = hmul2(o3, s);
    }
  }
}

// ---------------------------------------------------------------------------
// V fragments of a token pair (ta, tb) for all n-tiles: bv[j] = f16x2
// (V[ta][d_j], V[tb][d_j]) with d_j = (D/8) * g + j for lane group g.
// Invalid tokens read as zero codes.
// ---------------------------------------------------------------------------
template <int FMT, int D>
__device__ __forceinline__ void v_pair(uint32_t boxV, uint32_t boxVs, int ta, int tb,
                                       bool va, bool vb, int g, uint32_t (&bv)[D / 8]) {
  using Gm = Geom<FMT, D>;
  if constexpr (FMT == kFmtFp8 && D == 128) {
    uint4 A = lds128(boxV + ta * 128 + (Gm::swz(ta, g) << 4));
    uint4 B = lds128(boxV + tb * 128 + (Gm::swz(tb, g) << 4));
    if (!va) A = make_uint4(0, 0, 0, 0);
    if (!vb) B = make_uint4(0, 0, 0, 0);
    uint32_t a[4] = {A.x, A.y, A.z, A.w}, bb[4] = {B.x, B.y, B.z, B.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t p0 = __byte_perm(a[w], bb[w], 0x5140);
      uint32_t p1 = __byte_perm(a[w], bb[w], 0x7362);
      bv[4 * w + 0] = e4m3x2_to_f16x2(p0 & 0xFFFFu);
      bv[4 * w + 1] = e4m3x2_to_f16x2(p0 >> 16);
      bv[4 * w + 2] = e4m3x2_to_f16x2(p1 & 0xFFFFu);
      bv[4 * w + 3] = e4m3x2_to_f16x2(p1 >> 16);
    }
  } else if constexpr (FMT == kFmtFp8 && D == 64) {
    // 8 bytes per token: bytes [8g, 8g+8) = half (g & 1) of logical chunk g >> 1
    uint2 A = lds64(boxV + ta * 64 + (Gm::swz(ta, g >> 1) << 4) + ((g & 1) << 3));
    uint2 B = lds64(boxV + tb * 64 + (Gm::swz(tb, g >> 1) << 4) + ((g & 1) << 3));
    if (!va) A = make_uint2(0, 0);
    if (!vb) B = make_uint2(0, 0);
    uint32_t a[2] = {A.x, A.y}, bb[2] = {B.x, B.y};
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      uint32_t p0 = __byte_perm(a[w], bb[w], 0x5140);
      uint32_t p1 = __byte_perm(a[w], bb[w], 0x7362);
      bv[4 * w + 0] = e4m3x2_to_f16x2(p0 & 0xFFFFu);
      bv[4 * w + 1] = e4m3x2_to_f16x2(p0 >> 16);
      bv[4 * w + 2] = e4m3x2_to_f16x2(p1 & 0xFFFFu);
      bv[4 * w + 3] = e4m3x2_to_f16x2(p1 >> 16);
    }
  } else {
    static_assert(FMT == kFmtNvfp4 && D == 128, "unsupported V layout");
    // 16 elements per token: bytes [8g, 8g+8) of the 64-byte row, block g
    uint2 A = lds64(boxV + ta * 64 + (Gm::swz(ta, g >> 1) << 4) + ((g & 1) << 3));
    uint2 B = lds64(boxV + tb * 64 + (Gm::swz(tb, g >> 1) << 4) + ((g & 1) << 3));
    uint32_t sa = lds8(boxVs + ta * 8 + g), sb = lds8(boxVs + tb * 8 + g);
    if (!va) { A = make_uint2(0, 0); sa = 0; }
    if (!vb) { B = make_uint2(0, 0); sb = 0; }
    uint32_t s2 = e4m3x2_to_f16x2(sa | (sb << 8));   // (scale_a, scale_b)
    uint32_t a[2] = {A.x, A.y}, bb[2] = {B.x, B.y};
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      uint32_t ev = (a[w] & 0x0F0F0F0Fu) | ((bb[w] & 0x0F0F0F0Fu) << 4);
      uint32_t od = ((a[w] >> 4) & 0x0F0F0F0Fu) | (bb[w] & 0xF0F0F0F0u);
      uint32_t e0, e1, e2, e3, o0, o1, o2, o3;
      e2m1x8_to_f16x2x4(ev, e0, e1, e2, e3);
      e2m1x8_to_f16x2x4(od, o0, o1, o2, o3);
      bv[8 * w + 0] = hmul2(e0, s2);
      bv[8 * w + 1] = hmul2(o0, s2);
      bv[8 * w + 2] = hmul2(e1, s2);
      bv[8 * w + 3] = hmul2(o1, s2);
      bv[8 * w + 4] = hmul2(e2, s2);
      bv[8 * w + 5] = hmul2(o2, s2);
      bv[8 * w + 6] = hmul2(e3, s2);
      bv[8 * w + 7] = hmul2(o3, s2);
    }
  }
}

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
  return v;
}
__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v;
}

template <int FMT, int D, bool PROBQ>
__global__ void __launch_bounds__(kDecodeThreads, 1)
    partial_kernel(const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const PartialArgs a) {
  using Gm = Geom<FMT, D>;
  constexpr int KS = Gm::kKSteps;
  constexpr int NT = Gm::kNT;

  extern __shared__ uint8_t dyn_smem[];
  __shared__ Smem sm;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int bh = blockIdx.x;                 // b * Hkv + kv head
  const int b = bh / a.Hkv, h = bh % a.Hkv;
  const int split = blockIdx.y;

  // ring base, aligned for the 128-byte swizzle pattern
  const uint32_t ring = (smem_u32(dyn_smem) + 1023u) & ~1023u;
  const uint32_t scores = ring + kStages * Gm::kStage;   // FP8-prob mode only

  // chunk of this split
  int L = a.seq_lens[b];
  const int cap = min(a.max_pages * a.ps, a.max_kv_len);
  if (L > cap || L < 0) {
    if (threadIdx.x == 0) record_error(a.error_flag, 2);
    L = L < 0 ? 0 : cap;
  }
  long c = ((long)L + a.num_splits - 1) / a.num_splits;
  c = (c + 15) / 16 * 16;
  const int cstart = (int)min((long)split * c, (long)L);
  const int cend = (int)min((long)cstart + c, (long)L);
  const int ntiles = (cend - cstart + kTileTokens - 1) / kTileTokens;
  constexpr int kSweeps = PROBQ ? 2 : 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&sm.full[i]), 1);
      mbar_init(smem_u32(&sm.empty[i]), kConsumerWarps);
    }
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the loop (uniform control flow); lane 0 issues.
    if (ntiles > 0) {
      if (lane == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
      }
      const int32_t* bt = a.block_table + (size_t)b * a.max_pages;
      int last_pidx = -1, last_page = 0;
      int it = 0;
      bool ok = true;
      for (int sweep = 0; sweep < kSweeps && ok; ++sweep) {
        const bool loadK = !PROBQ || sweep == 0;
        const bool loadV = !PROBQ || sweep == 1;
        for (int tile = 0; tile < ntiles; ++tile, ++it) {
          const int st = it % kStages;
          if (it >= kStages) {
            const bool got =
                wait_or_abort(smem_u32(&sm.empty[st]), ((it / kStages) - 1) & 1, abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
              ok = false;
              break;
            }
          }
          if (lane == 0) {
            const int t0 = cstart + tile * kTileTokens;
            const int nbox =
                min(kTileTokens / kBoxTokens, (cend - t0 + kBoxTokens - 1) / kBoxTokens);
            uint32_t bytes = 0;
            if (loadK) bytes += nbox * (Gm::kBoxK + Gm::kBoxS);
            if (loadV) bytes += nbox * (Gm::kBoxK + Gm::kBoxS);
            const uint32_t full = smem_u32(&sm.full[st]);
            mbar_arrive_expect_tx(full, bytes);
            const uint32_t sbase = ring + st * Gm::kStage;
            for (int bx = 0; bx < nbox; ++bx) {
              const int tok = t0 + bx * kBoxTokens;
              const int pidx = tok / a.ps;
              if (pidx != last_pidx) {
                last_pidx = pidx;
                last_page = __ldg(bt + pidx);
                if (last_page < 0 || last_page >= a.num_pages) {
                  record_error(a.error_flag, 4);
                  last_page = 0;
                }
              }
              const long row = ((long)last_page * a.Hkv + h) * a.ps + (tok % a.ps);
              if (loadK) tma_load_2d(sbase + bx * Gm::kBoxK, &tmK, 0, (int)row, full);
              if (loadV)
                tma_load_2d(sbase + Gm::kTileK + bx * Gm::kBoxK, &tmV, 0, (int)row, full);
              if constexpr (FMT == kFmtNvfp4) {
                if (loadK)
                  bulk_load(sbase + 2 * Gm::kTileK + bx * Gm::kBoxS,
                            a.k_bscale + row * Gm::kSRow, Gm::kBoxS, full);
                if (loadV)
                  bulk_load(sbase + 2 * Gm::kTileK + Gm::kTileS + bx * Gm::kBoxS,
                            a.v_bscale + row * Gm::kSRow, Gm::kBoxS, full);
              }
            }
          }
          __syncwarp();
        }
      }
      if (!ok && lane == 0) {
        *abort_flag = 1;
        record_error(a.error_flag, 1);
      }
      // Drain: no copy may still be writing shared memory when the CTA exits.
      for (int k = max(0, it - kStages); k < it; ++k)
        mbar_wait(smem_u32(&sm.full[k % kStages]), (k / kStages) & 1);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int cw = warp - 1;
    const int hq0 = h * a.G;
    // Q fragments, head-dim permuted like the K fragments
    uint32_t qa[KS][4];
    {
      const int rows[2] = {g, g + 8};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int row = rows[half];
        const bool valid = row < a.G;
        const uint16_t* qp = a.q + ((size_t)b * a.Hq + hq0 + (valid ? row : 0)) * D + (D / 4) * t;
#pragma unroll
        for (int j = 0; j < KS; ++j) {
          uint2 v = valid ? *reinterpret_cast<const uint2*>(qp + 4 * j) : make_uint2(0, 0);
          float f0 = bf16_bits_to_f32(v.x & 0xFFFFu), f1 = bf16_bits_to_f32(v.x >> 16);
          float f2 = bf16_bits_to_f32(v.y & 0xFFFFu), f3 = bf16_bits_to_f32(v.y >> 16);
          qa[j][half] = pack_f16x2(f0, f1);       // a0 / a1
          qa[j][half + 2] = pack_f16x2(f2, f3);   // a2 / a3
        }
      }
    }

    float o[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    bool aborted = false;
    int it = 0;

    for (int sweep = 0; sweep < kSweeps; ++sweep) {
      for (int tile = 0; tile < ntiles && !aborted; ++tile, ++it) {
        const int st = it % kStages;
        const bool got = wait_or_abort(smem_u32(&sm.full[st]), (it / kStages) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          aborted = true;
          break;
        }
        const int tbase = cstart + tile * kTileTokens + cw * kBoxTokens;
        const int nvalid = max(0, min(kBoxTokens, cend - tbase));
        const uint32_t sbase = ring + st * Gm::kStage;
        const uint32_t boxK = sbase + cw * Gm::kBoxK;
        const uint32_t boxV = sbase + Gm::kTileK + cw * Gm::kBoxK;
        const uint32_t boxKs = sbase + 2 * Gm::kTileK + cw * Gm::kBoxS;
        const uint32_t boxVs = sbase + 2 * Gm::kTileK + Gm::kTileS + cw * Gm::kBoxS;
        const int tok_in_chunk = tbase - cstart;

        if (nvalid > 0) {
          float x[2][4];
          if (!PROBQ || sweep == 0) {
            // ---- scores S = Q K^T for the box's 16 tokens (two n-tiles)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              uint32_t kb[KS][2];
              k_frag<FMT, D>(boxK, boxKs, 8 * u + g, t, kb);
              float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int j = 0; j < KS; ++j)
                mma_f16(s, qa[j][0], qa[j][1], qa[j][2], qa[j][3], kb[j][0], kb[j][1]);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int tk = 8 * u + 2 * t + (e & 1);
                x[u][e] = tk < nvalid ? s[e] * a.qk_scale_log2 : -INFINITY;
              }
            }
          }
          if constexpr (PROBQ) {
            if (sweep == 0) {
              // keep the scores of the valid head rows; track the chunk max
#pragma unroll
              for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int row = g + 8 * (e >> 1);
                  const int tk = 8 * u + 2 * t + (e & 1);
                  if (row < a.G && tk < nvalid) {
                    asm volatile("st.shared.f32 [%0], %1;" ::"r"(
                                     scores + 4u * ((tok_in_chunk + tk) * a.G + row)),
                                 "f"(x[u][e]));
                  }
                }
              m0 = fmaxf(m0, quad_max(fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]))));
              m1 = fmaxf(m1, quad_max(fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]))));
            } else {
              // ---- FP8 probabilities against the chunk max (m0/m1 hold it)
              const float b0 = m0 == -INFINITY ? 0.f : m0;
              const float b1 = m1 == -INFINITY ? 0.f : m1;
              uint32_t pa[4];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                float p[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int row = g + 8 * (e >> 1);
                  const int tk = 8 * u + 2 * t + (e & 1);
                  float xs = -INFINITY;
                  if (row < a.G && tk < nvalid) {
                    asm volatile("ld.shared.f32 %0, [%1];"
                                 : "=f"(xs)
                                 : "r"(scores + 4u * ((tok_in_chunk + tk) * a.G + row)));
                  }
                  p[e] = exp2f(xs - ((e >> 1) ? b1 : b0));
                }
                l0 += p[0] + p[1];
                l1 += p[2] + p[3];
                const float ps = a.prob_scale;
                uint32_t c01 = f32x2_to_e4m3x2(__fdiv_rn(p[0], ps), __fdiv_rn(p[1], ps));
                uint32_t c23 = f32x2_to_e4m3x2(__fdiv_rn(p[2], ps), __fdiv_rn(p[3], ps));
                pa[2 * u + 0] = e4m3x2_to_f16x2(c01);   // row g   (a0 / a2)
                pa[2 * u + 1] = e4m3x2_to_f16x2(c23);   // row g+8 (a1 / a3)
              }
              uint32_t bv0[NT], bv1[NT];
              v_pair<FMT, D>(boxV, boxVs, 2 * t, 2 * t + 1, 2 * t < nvalid, 2 * t + 1 < nvalid, g,
                             bv0);
              v_pair<FMT, D>(boxV, boxVs, 2 * t + 8, 2 * t + 9, 2 * t + 8 < nvalid,
                             2 * t + 9 < nvalid, g, bv1);
#pragma unroll
              for (int j = 0; j < NT; ++j) mma_f16(o[j], pa[0], pa[1], pa[2], pa[3], bv0[j], bv1[j]);
            }
          } else {
            // ---- online softmax update (log2 domain)
            const float mx0 = quad_max(fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1])));
            const float mx1 = quad_max(fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3])));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float b0 = mn0 == -INFINITY ? 0.f : mn0;
            const float b1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = exp2f(m0 - b0), al1 = exp2f(m1 - b1);
            m0 = mn0;
            m1 = mn1;
            float p[2][4];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              p[u][0] = exp2f(x[u][0] - b0);
              p[u][1] = exp2f(x[u][1] - b0);
              p[u][2] = exp2f(x[u][2] - b1);
              p[u][3] = exp2f(x[u][3] - b1);
            }
            l0 = l0 * al0 + (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
            l1 = l1 * al1 + (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
            if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
              for (int j = 0; j < NT; ++j) {
                o[j][0] *= al0;
                o[j][1] *= al0;
                o[j][2] *= al1;
                o[j][3] *= al1;
              }
            }
            // P as f16 high part + f16 residual
            uint32_t ph[4], pl[4];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              ph[2 * u + 0] = pack_f16x2(p[u][0], p[u][1]);
              ph[2 * u + 1] = pack_f16x2(p[u][2], p[u][3]);
              const float2 r0 = unpack_f16x2(ph[2 * u + 0]);
              const float2 r1 = unpack_f16x2(ph[2 * u + 1]);
              pl[2 * u + 0] = pack_f16x2(p[u][0] - r0.x, p[u][1] - r0.y);
              pl[2 * u + 1] = pack_f16x2(p[u][2] - r1.x, p[u][3] - r1.y);
            }
            uint32_t bv0[NT], bv1[NT];
            v_pair<FMT, D>(boxV, boxVs, 2 * t, 2 * t + 1, 2 * t < nvalid, 2 * t + 1 < nvalid, g,
                           bv0);
            v_pair<FMT, D>(boxV, boxVs, 2 * t + 8, 2 * t + 9, 2 * t + 8 < nvalid,
                           2 * t + 9 < nvalid, g, bv1);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              mma_f16(o[j], ph[0], ph[1], ph[2], ph[3], bv0[j], bv1[j]);
              mma_f16(o[j], pl[0], pl[1], pl[2], pl[3], bv0[j], bv1[j]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.empty[st]));
      }
      if constexpr (PROBQ) {
        if (sweep == 0) {
          // chunk max across the consumer warps (every consumer warp takes
          // part in both barriers, aborted or not)
          __syncwarp();
          if (t == 0) {
            sm.m[cw][g] = m0;
            sm.m[cw][g + 8] = m1;
          }
          asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps) : "memory");
          float a0 = -INFINITY, a1 = -INFINITY;
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            a0 = fmaxf(a0, sm.m[w][g]);
            a1 = fmaxf(a1, sm.m[w][g + 8]);
          }
          m0 = a0;
          m1 = a1;
          asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps) : "memory");
        }
      }
    }
    if (aborted) {
      *abort_flag = 1;
      record_error(a.error_flag, 1);
    }
    // per-warp state -> shared memory
    l0 = quad_sum(l0);
    l1 = quad_sum(l1);
    if (t == 0) {
      sm.m[cw][g] = m0;
      sm.m[cw][g + 8] = m1;
      sm.l[cw][g] = l0;
      sm.l[cw][g + 8] = l1;
    }
    // O tiles go to the (drained) ring: obuf[cw][row][d], rows < G
    __syncwarp();
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps) : "memory");
    float* obuf = reinterpret_cast<float*>(dyn_smem + (ring - smem_u32(dyn_smem)));
    if (!*abort_flag) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = g + 8 * (e >> 1);
          const int col = 2 * t + (e & 1);
          const int d = (D / 8) * col + j;
          if (row < a.G) obuf[(cw * a.G + row) * D + d] = o[j][e];
        }
      }
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- merge
  const size_t part_row = ((size_t)b * a.Hq + (size_t)h * a.G);   // first query head
  const bool bad = *abort_flag != 0;
  if (threadIdx.x < a.G) {
    const int row = threadIdx.x;
    float M = -INFINITY;
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm.m[w][row]);
    float Ltot = 0.f;
    for (int w = 0; w < kConsumerWarps; ++w)
      if (sm.m[w][row] != -INFINITY) Ltot += exp2f(sm.m[w][row] - M) * sm.l[w][row];
    for (int w = 0; w < kConsumerWarps; ++w)
      sm.fac[w][row] = (M == -INFINITY || sm.m[w][row] == -INFINITY)
                           ? 0.f
                           : exp2f(sm.m[w][row] - M) / Ltot * a.out_mult;
    float lse = (M == -INFINITY) ? -INFINITY : (M + log2f(Ltot)) * kLn2;
    if (bad) lse = NAN;
    a.part_lse[(part_row + row) * a.num_splits + split] = lse;
  }
  __syncthreads();
  const float* obuf = reinterpret_cast<const float*>(dyn_smem + (ring - smem_u32(dyn_smem)));
  for (int i = threadIdx.x; i < a.G * D; i += blockDim.x) {
    const int row = i / D, d = i % D;
    float acc = 0.f;
    if (!bad) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) acc += sm.fac[w][row] * obuf[(w * a.G + row) * D + d];
    } else {
      acc = NAN;
    }
    a.part_o[((part_row + row) * a.num_splits + split) * D + d] = acc;
  }
}

// ---------------------------------------------------------------------------
// Combine: one CTA per (request, query head).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) combine_kernel(const CombineArgs a) {
  extern __shared__ float w[];   // num_splits weights
  __shared__ float wsum_s;
  const int row = blockIdx.x;
  const float* lse = a.part_lse + (size_t)row * a.num_splits;
  if (threadIdx.x < 32) {
    float M = -INFINITY;
    for (int j = threadIdx.x; j < a.num_splits; j += 32) M = fmaxf(M, lse[j]);
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float s = 0.f;
    for (int j = threadIdx.x; j < a.num_splits; j += 32) {
      const float v = (M == -INFINITY || lse[j] == -INFINITY) ? 0.f : expf(lse[j] - M);
      w[j] = v;
      s += v;
    }
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (threadIdx.x == 0) wsum_s = s;
  }
  __syncthreads();
  const float inv = wsum_s > 0.f ? 1.f / wsum_s : 0.f;
  const float* po = a.part_o + (size_t)row * a.num_splits * a.Dv;
  for (int d = threadIdx.x; d < a.Dv; d += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < a.num_splits; ++j)
      if (w[j] != 0.f) acc += w[j] * po[(size_t)j * a.Dv + d];
    const float v = wsum_s > 0.f ? acc * inv : 0.f;
    const size_t oi = (size_t)row * a.Dv + d;
    if (a.out_dtype == 0) {
      static_cast<float*>(a.out)[oi] = v;
    } else if (a.out_dtype == 1) {
      static_cast<__nv_bfloat16*>(a.out)[oi] = __float2bfloat16_rn(v);
    } else {
      static_cast<uint8_t*>(a.out)[oi] =
          (uint8_t)(f32x2_to_e4m3x2(__fdiv_rn(v, a.out_scale), 0.f) & 0xFFu);
    }
  }
}

template <int FMT, int D, bool PROBQ>
cudaError_t launch_partial_t(const CUtensorMap& tk, const CUtensorMap& tv, const PartialArgs& a,
                             cudaStream_t st) {
  using Gm = Geom<FMT, D>;
  size_t smem = 1024 + (size_t)kStages * Gm::kStage;
  if (PROBQ) smem += (size_t)kScoreCapacity * 4;
  // the merge buffer reuses the ring
  const size_t merge = (size_t)kConsumerWarps * kMaxGroup * D * 4;
  if (1024 + (size_t)kStages * Gm::kStage < 1024 + merge) smem = 1024 + merge + (PROBQ ? (size_t)kScoreCapacity * 4 : 0);
  auto kern = partial_kernel<FMT, D, PROBQ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.batch * a.Hkv, a.num_splits);
  kern<<<grid, kDecodeThreads, smem, st>>>(tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_partial(int fmt, int D, bool probq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const PartialArgs& a, cudaStream_t st) {
  if (fmt == kFmtFp8 && D == 128)
    return probq ? launch_partial_t<kFmtFp8, 128, true>(tk, tv, a, st)
                 : launch_partial_t<kFmtFp8, 128, false>(tk, tv, a, st);
  if (fmt == kFmtFp8 && D == 64)
    return probq ? launch_partial_t<kFmtFp8, 64, true>(tk, tv, a, st)
                 : launch_partial_t<kFmtFp8, 64, false>(tk, tv, a, st);
  if (fmt == kFmtNvfp4 && D == 128)
    return probq ? launch_partial_t<kFmtNvfp4, 128, true>(tk, tv, a, st)
                 : launch_partial_t<kFmtNvfp4, 128, false>(tk, tv, a, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st) {
  combine_kernel<<<a.rows, 128, (size_t)a.num_splits * sizeof(float), st>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
