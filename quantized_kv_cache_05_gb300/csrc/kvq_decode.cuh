// Split-KV flash-decode over a quantized KV cache (sm_103a): the partial
// kernel template and its launcher, instantiated per cache format in
// kvq_decode.cu (FP8) and kvq_decode_nvfp4.cu (NVFP4).
//
// Method (Model-Optimizer PR 1832, notes under the latency tables): each
// (request, kv head) sequence is cut into s contiguous chunks; one CTA runs
// the partial softmax (running max, denominator, weighted V) of one chunk for
// all Hq/Hkv query heads of the kv head, and a small combine kernel merges the
// s partials.  FP8 probabilities and FP8 output follow vLLM PR 15734.
//
// GB300 design of the partial kernel
//  * NW warps per CTA: six, two CTAs per SM, for the common decode (up to 8
//    query heads per kv head, head_dim <= 128, no FP8 probabilities); four
//    otherwise (three CTAs per SM, four in the FP8-probability mode, whose
//    ring holds one tensor per stage).  Twelve warps per SM either way; the
//    six-warp CTAs leave a third fewer split partials for the merge.  Each
//    warp streams its own 16-token boxes (box w, w+NW, w+2NW, ... of the
//    chunk) HBM -> shared memory with TMA (cp.async.bulk.tensor, 16-row box
//    = one 16-token page, hardware swizzle; NVFP4 block scales by 1-D bulk
//    copies) into a private 2-deep (six warps) or 3-deep ring with its own
//    mbarriers, and consumes them itself: no producer warp, no cross-warp
//    hand-off per box, and twelve warps per SM issuing copies (one issuing
//    thread per CTA cannot keep HBM busy).  The
//    chunk's block-table entries are cached in shared memory.
//  * Codes are decoded in registers straight into tensor-core fragments
//    (E4M3 -> f16 and E2M1 -> f16 with cvt, block scales by an f16x2
//    multiply: all exact), and the contractions run on mma.sync m16n8k16 with
//    fp32 accumulation:
//      S^T = K Q^T     M = 16 tokens, N = 8 query heads, K = 16 head dims
//      O^T = V^T P^T   M = 16 value dims, N = 8 query heads, K = 16 tokens
//    P^T comes from the S^T accumulator by one movmatrix transpose per 8x8
//    block, so every lane keeps the softmax state of the two heads its own
//    accumulator columns hold (no shuffles on the common path).
//  * Head-dim order inside a K row is permuted per lane so that each lane's
//    codes come from 16-byte shared-memory loads; Q is loaded with the same
//    permutation.  The token-pair layout of the V^T operand is built with
//    byte permutes (FP8) or nibble masks (E2M1).
//  * P is split into an f16 high part and an f16 residual (two MMAs), so the
//    probabilities keep ~22 bits; with FP8 probabilities the E4M3 code itself
//    is the (exact) f16 operand.
//  * The running max moves only when a box's max exceeds it by more than
//    2^8 (log2 domain), so O is rarely rescaled; the final normalization by
//    the denominator is exact whatever the reference max.
//  * Warps merge their (max, sum, O) states through shared memory at the end
//    (O in MMA-fragment order); the last CTA of a (request, kv head) merges
//    the split partials in the same launch when the arrival counters are given.
// Every mbarrier wait is bounded; a timeout sets an error bit and the CTA
// writes NaN for its partial instead of hanging.

#include <cfloat>
#include <cmath>

#pragma once

#include <algorithm>

#include "kvq_attn.cuh"

namespace kvq {
namespace decode_impl {

// Boxes in flight per warp: two for six-warp CTAs, three for four-warp ones
// (measured: with six-warp CTAs two stages gave the shorter GQA steps, 34.9
// against 35.3 us at 32k and 20.3 against 20.8 at 8k; four were slower in
// every mode).
template <int NW>
constexpr int ring_stages() { return NW == kWideWarps ? 2 : kStages; }

template <int NW>
struct Smem {
  uint64_t full[NW][ring_stages<NW>()];
  uint64_t comb_full;   // fused combine: partials landed
  int abort_flag;
  int pages[kPageCache];
  float m[NW][kMaxGroup];
  float l[NW][kMaxGroup];
  float fac[NW][kMaxGroup];
};

// Shared-memory ring of the partial kernel: the TMA stages, reused after the
// loop for the warps' O fragments and the fused combine's weights.
template <int FMT, int D, bool PROBQ, int NH, int NW>
struct Ring {
  using Gm = Geom<FMT, D>;
  static constexpr int kStageBytes = PROBQ ? Gm::kStage1 : Gm::kStage;
  static constexpr int kEpilogue = NW * Gm::kMT * NH * 32 * 16 +
                                   (kMaxGroup * kMaxFusedSplits + kMaxGroup) * 4;
  static constexpr int kStream = NW * ring_stages<NW>() * kStageBytes;
  static constexpr int kBytes =
      kStream > kEpilogue ? kStream : (kEpilogue + 1023) / 1024 * 1024;
};

// Resident CTAs per SM the kernel is compiled for: four for the half-size
// ring of the FP8-probability mode with up to eight query heads per kv head,
// three otherwise, two with sixteen heads (twice the accumulators); head_dim
// 256 has twice the fragments and ring of 128: two, one with sixteen heads.
// Six-warp CTAs (NW = 6): two per SM.
template <int FMT, int D, bool PROBQ, int NH, int NW>
constexpr int ctas_per_sm() {
  if (NW == 6) return 2;
  if (D >= 256) return NH == 2 ? 1 : 2;
  return NH == 2 ? 2 : PROBQ ? 4 : 3;
}

// NH = number of 8-head groups (1: up to 8 query heads per kv head, 2: up to
// 16); QF8: the query is E4M3 codes (FP8 query), and with an FP8 cache the
// scores run on the E4M3 x E4M3 MMA straight from the cached code bytes.
template <int FMT, int D, bool PROBQ, int NH, bool QF8, int NW>
__global__ void __launch_bounds__(32 * NW, ctas_per_sm<FMT, D, PROBQ, NH, NW>())
    partial_kernel(const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const PartialArgs a) {
  using Gm = Geom<FMT, D>;
  constexpr int kRingStages = ring_stages<NW>();
  constexpr int KS = Gm::kKSteps;
  constexpr bool kRawK = QF8 && FMT == kFmtFp8;   // scores on e4m3 x e4m3 (k32)
  constexpr int KS8 = D / 32;                      // its k-steps
  constexpr int MT = Gm::kMT;
  constexpr int kSweeps = PROBQ ? 2 : 1;

  extern __shared__ uint8_t dyn_smem[];
  __shared__ Smem<NW> sm;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int bh = blockIdx.x;                 // b * Hkv + kv head
  const int b = bh / a.Hkv, h = bh % a.Hkv;
  const int split = blockIdx.y;

  // ring base, aligned for the 128-byte swizzle pattern
  const uint32_t ring = (smem_u32(dyn_smem) + 1023u) & ~1023u;
  using Rg = Ring<FMT, D, PROBQ, NH, NW>;
  const uint32_t scores = ring + Rg::kBytes;   // FP8-prob mode only

  const int cap = min(a.max_pages * a.ps, a.max_kv_len);
  // Launched with programmatic serialization, this kernel can start before
  // the previous kernel in the stream ends, and its inputs may come from that
  // kernel.  Before the wait it only sets up its barriers -- unless the
  // caller declared that kernel to be the append of the last a.fresh
  // positions: then only the loads of boxes holding those positions wait.
  if (threadIdx.x == 0) sm.abort_flag = 0;
  if (lane == 0) {
    for (int i = 0; i < kRingStages; ++i) mbar_init(smem_u32(&sm.full[warp][i]), 1);
    if (warp == 0) mbar_init(smem_u32(&sm.comb_full), 1);
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  if (a.fresh == 0) griddep_wait();

  // one-page requests: the page index does not depend on the length, so its
  // load overlaps the length's
  const int32_t* bt = a.block_table + (size_t)b * a.max_pages;
  int pg_single = 0;
  if (a.max_pages == 1 && threadIdx.x == 0) pg_single = __ldg(bt);

  // chunk of this split
  int L = a.seq_lens[b];
  if (L > cap || L < 0) {
    if (threadIdx.x == 0) record_error(a.error_flag, 2);
    L = L < 0 ? 0 : cap;
  }
  long c = ((long)L + a.num_splits - 1) / a.num_splits;
  c = (c + 15) / 16 * 16;
  const int cstart = (int)min((long)split * c, (long)L);
  const int cend = (int)min((long)cstart + c, (long)L);
  const int nboxes = (cend - cstart + kBoxTokens - 1) / kBoxTokens;
  // first box of the chunk that holds an appended position (overlap mode)
  const int fresh_box = a.fresh == 0 ? 0 : (max(L - a.fresh, cstart) - cstart) / kBoxTokens;
  bool dep_done = a.fresh == 0;   // this thread has waited for the preceding kernel
  // this warp's boxes: warp, warp + NW, ...
  const int nw = nboxes > warp ? (nboxes - warp + NW - 1) / NW : 0;
  const int total = kSweeps * nw;

  // block-table entries of the chunk -> shared memory
  const int p0 = cstart / a.ps;
  const int npages = cend > cstart ? (cend - 1) / a.ps - p0 + 1 : 0;
  for (int i = threadIdx.x; i < min(npages, kPageCache); i += (32 * NW)) {
    int pg = a.max_pages == 1 ? pg_single : __ldg(bt + p0 + i);
    if (pg < 0 || pg >= a.num_pages) {
      record_error(a.error_flag, 4);
      pg = 0;
    }
    sm.pages[i] = pg;
  }
  __syncthreads();
  volatile int* abort_flag = &sm.abort_flag;

  // Issue the copies of this warp's j-th load (lane 0 only) into stage st:
  // load j covers box w + NW (j % nw); in FP8-prob mode loads [0, nw) bring
  // K, [nw, 2nw) V.  Loads are issued in order; the page and in-page offset
  // of the next one advance by 16 NW tokens per load (no division per box).
  const int tok_first = cstart + warp * kBoxTokens;
  int nx_pidx = tok_first / a.ps;
  int nx_off = tok_first - nx_pidx * a.ps;
  auto issue = [&](int j, int st) {
    const int sweep = PROBQ ? (j >= nw ? 1 : 0) : 0;
    const int box = warp + NW * (j - sweep * nw);
    const bool loadK = !PROBQ || sweep == 0;
    const bool loadV = !PROBQ || sweep == 1;
    if (PROBQ && j == nw) {   // the V sweep starts over at the warp's first box
      nx_pidx = tok_first / a.ps;
      nx_off = tok_first - nx_pidx * a.ps;
    }
    const int pidx = nx_pidx, off = nx_off;
    nx_off += NW * kBoxTokens;
    while (nx_off >= a.ps) {
      nx_off -= a.ps;
      ++nx_pidx;
    }
    int page;
    if (pidx - p0 < kPageCache) {
      page = sm.pages[pidx - p0];
    } else {
      page = __ldg(bt + pidx);
      if (page < 0 || page >= a.num_pages) {
        record_error(a.error_flag, 4);
        page = 0;
      }
    }
    const long row = ((long)page * a.Hkv + h) * a.ps + off;
    if (!dep_done && box >= fresh_box) {
      griddep_wait();
      dep_done = true;
    }
    const uint32_t full = smem_u32(&sm.full[warp][st]);
    const uint32_t sbase = ring + (warp * kRingStages + st) * Rg::kStageBytes;
    const uint32_t bytes = (loadK ? Gm::kBoxK + Gm::kBoxS : 0) + (loadV ? Gm::kBoxK + Gm::kBoxS : 0);
    mbar_arrive_expect_tx(full, bytes);
    if constexpr (PROBQ) {   // one tensor per stage: [codes][scales]
      tma_load_2d(sbase, loadK ? &tmK : &tmV, 0, (int)row, full);
      if constexpr (FMT == kFmtNvfp4)
        bulk_load(sbase + Gm::kBoxK, (loadK ? a.k_bscale : a.v_bscale) + row * Gm::kSRow,
                  Gm::kBoxS, full);
    } else {                 // [K codes][V codes][K scales][V scales]
      tma_load_2d(sbase, &tmK, 0, (int)row, full);
      tma_load_2d(sbase + Gm::kBoxK, &tmV, 0, (int)row, full);
      if constexpr (FMT == kFmtNvfp4) {
        bulk_load(sbase + 2 * Gm::kBoxK, a.k_bscale + row * Gm::kSRow, Gm::kBoxS, full);
        bulk_load(sbase + 2 * Gm::kBoxK + Gm::kBoxS, a.v_bscale + row * Gm::kSRow, Gm::kBoxS,
                  full);
      }
    }
  };

  // FP8 caches, short chunks (fewer than 8 loads per warp): only the first
  // load of every warp goes out now, the rest of the ring once the query is
  // loaded, so the grid's first burst of copies is smaller and every warp's
  // first box lands sooner (GQA FP8 8k: step 19.7 -> 18.9 us).  Long chunks,
  // and NVFP4 (whose decode work per box is the bottleneck: 8k 0.5 us
  // slower deferred), fill the ring at once.
  const int early = (FMT == kFmtFp8 && total < 8) ? 1 : kRingStages;
  int issued = 0;
  if (lane == 0) {
#pragma unroll 1   // one copy of the issue code (it runs cold, once per CTA)
    for (; issued < min(total, early); ++issued) issue(issued, issued);
  }

  const int hq0 = h * a.G;
  // score and output factors of this kv head: the tensor's scales, or the
  // head's own (per-kv-head scales)
  const float qk_scale_log2 =
      a.k_hs ? (a.sm_scale * __ldg(a.k_hs + h)) * 1.4426950408889634f : a.qk_scale_log2;
  const float out_mult =
      a.v_hs ? (a.prob_scale > 0.f ? __ldg(a.v_hs + h) * a.prob_scale : __ldg(a.v_hs + h))
             : a.out_mult;
  // Q^T fragments (B operand of S^T = K Q^T: k = head dims, n = query heads
  // g + 8 hh), head dims permuted like the K fragments; qsc[hh][e] is the
  // score scale of head 2t + e + 8hh, the head of this lane's accumulator
  // columns.
  //  bf16 q: each head is scaled by its power of two 2^e (q_prescale_exp)
  //    before the f16 conversion, so the query keeps the full bf16 range;
  //    qsc = sm_scale * k_scale * log2 e * 2^-e.
  //  FP8 q (QF8): the codes themselves (exact in f16; raw bytes for the
  //    e4m3 x e4m3 MMA); qsc = sm_scale * k_scale * log2 e * q_scale.
  uint32_t qb[kRawK ? 1 : KS][NH][2];
  uint32_t qb8[kRawK ? KS8 : 1][NH][2];
  float qsc[NH][2];
#pragma unroll
  for (int hh = 0; hh < NH; ++hh) {
    const int head = g + 8 * hh;
    const bool valid = head < a.G;
    const size_t qrow = (size_t)b * a.Hq + hq0 + (valid ? head : 0);
    if constexpr (QF8) {
      const uint8_t* qp = static_cast<const uint8_t*>(a.q) + qrow * D + (D / 4) * t;
      if constexpr (kRawK) {
#pragma unroll
        for (int j = 0; j < KS8; ++j) {
          const uint2 v = valid ? *reinterpret_cast<const uint2*>(qp + 8 * j) : make_uint2(0, 0);
          qb8[j][hh][0] = v.x;
          qb8[j][hh][1] = v.y;
        }
      } else {
#pragma unroll
        for (int j = 0; j < KS; ++j) {
          const uint32_t v = valid ? *reinterpret_cast<const uint32_t*>(qp + 4 * j) : 0u;
          e4m3x4_to_f16x2x2(v, qb[j][hh][0], qb[j][hh][1]);
        }
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int hc = 2 * t + e + 8 * hh;   // this lane's accumulator column
        const float qs = a.q_hs ? __ldg(a.q_hs + hq0 + min(hc, a.G - 1)) : a.q_scale;
        qsc[hh][e] = qk_scale_log2 * qs;
      }
    } else {
      const uint16_t* qp = static_cast<const uint16_t*>(a.q) + qrow * D + (D / 4) * t;
      uint2 raw[KS];
      uint32_t mx2 = 0;   // two packed 16-bit maxima of |q|
#pragma unroll
      for (int j = 0; j < KS; ++j) {
        raw[j] = valid ? *reinterpret_cast<const uint2*>(qp + 4 * j) : make_uint2(0, 0);
        mx2 = __vmaxu2(mx2, __vmaxu2(raw[j].x & 0x7FFF7FFFu, raw[j].y & 0x7FFF7FFFu));
      }
      // the head's D elements sit in the four lanes t = 0..3 of row g
      uint32_t mx = max(mx2 & 0xFFFFu, mx2 >> 16);
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const int e = q_prescale_exp(mx);
      const float f = exp2i(e);
#pragma unroll
      for (int j = 0; j < KS; ++j) {
        const uint2 v = raw[j];
        qb[j][hh][0] = pack_f16x2(__uint_as_float(v.x << 16) * f, __uint_as_float(v.x & 0xFFFF0000u) * f);
        qb[j][hh][1] = pack_f16x2(__uint_as_float(v.y << 16) * f, __uint_as_float(v.y & 0xFFFF0000u) * f);
      }
      const float my = scale_pow2(qk_scale_log2, -e);   // head g + 8hh
      qsc[hh][0] = __shfl_sync(0xffffffffu, my, 4 * (2 * t));
      qsc[hh][1] = __shfl_sync(0xffffffffu, my, 4 * (2 * t + 1));
    }
  }

  if (lane == 0) {
#pragma unroll 1
    for (; issued < min(total, kRingStages); ++issued) issue(issued, issued);
  }

  // O^T accumulators: m-tile i (value dims), head group hh; C layout
  // c0,c1 = (dim row g, heads 2t, 2t+1), c2,c3 = (dim row g+8, same heads)
  float o[MT][NH][4];
#pragma unroll
  for (int i = 0; i < MT; ++i)
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) o[i][hh][0] = o[i][hh][1] = o[i][hh][2] = o[i][hh][3] = 0.f;
  // reference max (log2 domain) and partial denominator of heads
  // 2t + e + 8 hh -- the same heads as this lane's S^T and O^T columns
  float m[NH][2], l[NH][2];
#pragma unroll
  for (int hh = 0; hh < NH; ++hh) m[hh][0] = m[hh][1] = -INFINITY, l[hh][0] = l[hh][1] = 0.f;
  bool aborted = false;

  int st = 0;          // stage of the current load
  uint32_t phase = 0;  // its mbarrier phase parity
  for (int sweep = 0; sweep < kSweeps; ++sweep) {
    for (int jj = 0; jj < nw && !aborted; ++jj) {
      // one lane polls the barrier; the vote tells the warp the outcome
      bool got = true;
      if (lane == 0) got = wait_or_abort(smem_u32(&sm.full[warp][st]), phase, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        aborted = true;
        break;
      }
      __syncwarp();   // the other lanes read the box after lane 0's acquire
      const int tbase = cstart + (warp + NW * jj) * kBoxTokens;
      const int nvalid = min(kBoxTokens, cend - tbase);
      const uint32_t sbase = ring + (warp * kRingStages + st) * Rg::kStageBytes;
      const uint32_t boxK = sbase;
      const uint32_t boxV = PROBQ ? sbase : sbase + Gm::kBoxK;
      const uint32_t boxKs = PROBQ ? sbase + Gm::kBoxK : sbase + 2 * Gm::kBoxK;
      const uint32_t boxVs = PROBQ ? boxKs : boxKs + Gm::kBoxS;
      const int tok_in_chunk = tbase - cstart;

      // x[hh][e]: scaled score of token g + 8 (e >> 1), head 2t + (e & 1) + 8 hh
      float x[NH][4];
      if (!PROBQ || sweep == 0) {
        // two accumulators halve the dependent MMA chain
        float s0[NH][4], s1[NH][4];
#pragma unroll
        for (int hh = 0; hh < NH; ++hh)
#pragma unroll
          for (int e = 0; e < 4; ++e) s0[hh][e] = s1[hh][e] = 0.f;
        if constexpr (kRawK) {
          uint32_t kw[D / 16], kw8[D / 16];
          k_raw_fp8<D>(boxK, g, t, kw);
          k_raw_fp8<D>(boxK, g + 8, t, kw8);
#pragma unroll
          for (int hh = 0; hh < NH; ++hh)
#pragma unroll
            for (int j = 0; j < KS8; ++j)
              mma_e4m3((j & 1) ? s1[hh] : s0[hh], kw[2 * j], kw8[2 * j], kw[2 * j + 1],
                       kw8[2 * j + 1], qb8[j][hh][0], qb8[j][hh][1]);
        } else {
          uint32_t kg[KS][2], kg8[KS][2];
          k_frag<FMT, D>(boxK, boxKs, g, t, kg);
          k_frag<FMT, D>(boxK, boxKs, g + 8, t, kg8);
#pragma unroll
          for (int hh = 0; hh < NH; ++hh)
#pragma unroll
            for (int kk = 0; kk < KS; kk += 2) {
              mma_f16(s0[hh], kg[kk][0], kg8[kk][0], kg[kk][1], kg8[kk][1], qb[kk][hh][0],
                      qb[kk][hh][1]);
              mma_f16(s1[hh], kg[kk + 1][0], kg8[kk + 1][0], kg[kk + 1][1], kg8[kk + 1][1],
                      qb[kk + 1][hh][0], qb[kk + 1][hh][1]);
            }
        }
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
#pragma unroll
          for (int e = 0; e < 4; ++e) x[hh][e] = (s0[hh][e] + s1[hh][e]) * qsc[hh][e & 1];
          if (nvalid < kBoxTokens) {   // ragged tail of the chunk
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (g + 8 * (e >> 1) >= nvalid) x[hh][e] = -INFINITY;
          }
        }
      }
      if constexpr (PROBQ) {
        if (sweep == 0) {
          // keep the scores of the valid heads; track the chunk max
#pragma unroll
          for (int hh = 0; hh < NH; ++hh) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int head = 2 * t + (e & 1) + 8 * hh;
              const int tk = g + 8 * (e >> 1);
              if (head < a.G && tk < nvalid)
                asm volatile("st.shared.f32 [%0], %1;" ::"r"(
                                 scores + 4u * ((tok_in_chunk + tk) * a.G + head)),
                             "f"(x[hh][e]));
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float mx = fmaxf(x[hh][e], x[hh][e + 2]);
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
              m[hh][e] = fmaxf(m[hh][e], mx);
            }
          }
        } else {
          // FP8 probabilities against the chunk max (m holds it)
          uint32_t pb[NH][2];
#pragma unroll
          for (int hh = 0; hh < NH; ++hh) {
            float p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int head = 2 * t + (e & 1) + 8 * hh;
              const int tk = g + 8 * (e >> 1);
              float xs = -INFINITY;
              if (head < a.G && tk < nvalid)
                asm volatile("ld.shared.f32 %0, [%1];"
                             : "=f"(xs)
                             : "r"(scores + 4u * ((tok_in_chunk + tk) * a.G + head)));
              const float mm = m[hh][e & 1];
              p[e] = ex2(xs - (mm == -INFINITY ? 0.f : mm));
            }
            l[hh][0] += p[0] + p[2];
            l[hh][1] += p[1] + p[3];
            const float ps = a.prob_scale, pz = a.prob_recip;
            const bool fast = a.prob_fast != 0;
            const uint32_t c01 = e4m3x2_to_f16x2(f32x2_to_e4m3x2(
                prob_quotient(p[0], ps, pz, fast), prob_quotient(p[1], ps, pz, fast)));
            const uint32_t c23 = e4m3x2_to_f16x2(f32x2_to_e4m3x2(
                prob_quotient(p[2], ps, pz, fast), prob_quotient(p[3], ps, pz, fast)));
            pb[hh][0] = movmatrix_trans(c01);   // (tokens 2t, 2t+1; head g)
            pb[hh][1] = movmatrix_trans(c23);   // (tokens 2t+8, 2t+9; head g)
          }
          uint32_t va[MT][4];
          v_frag<FMT, D>(boxV, boxVs, t, g, nvalid, va);
#pragma unroll
          for (int i = 0; i < MT; ++i)
#pragma unroll
            for (int hh = 0; hh < NH; ++hh)
              mma_f16(o[i][hh], va[i][0], va[i][1], va[i][2], va[i][3], pb[hh][0], pb[hh][1]);
        }
      } else {
        // ---- softmax update with a lazily moving reference max
        bool need = false;
#pragma unroll
        for (int hh = 0; hh < NH; ++hh)
#pragma unroll
          for (int e = 0; e < 4; ++e) need |= x[hh][e] > m[hh][e & 1] + kLazyMax;
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int hh = 0; hh < NH; ++hh)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float mx = fmaxf(x[hh][e], x[hh][e + 2]);
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
              const bool mv = mx > m[hh][e] + kLazyMax;   // also the first finite box
              const float alpha = mv ? ex2(m[hh][e] - mx) : 1.f;
              m[hh][e] = mv ? mx : m[hh][e];
              l[hh][e] *= alpha;
#pragma unroll
              for (int i = 0; i < MT; ++i) {
                o[i][hh][e] *= alpha;
                o[i][hh][e + 2] *= alpha;
              }
            }
        }
        uint32_t ph[NH][2], pl[NH][2];
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
          const float b0 = m[hh][0] == -INFINITY ? 0.f : m[hh][0];
          const float b1 = m[hh][1] == -INFINITY ? 0.f : m[hh][1];
          const float p0 = ex2(x[hh][0] - b0), p1 = ex2(x[hh][1] - b1);
          const float p2 = ex2(x[hh][2] - b0), p3 = ex2(x[hh][3] - b1);
          l[hh][0] += p0 + p2;
          l[hh][1] += p1 + p3;
          // P as f16 high part + f16 residual, moved into the P^T layout
          const uint32_t h01 = pack_f16x2(p0, p1), h23 = pack_f16x2(p2, p3);
          const float2 r01 = unpack_f16x2(h01), r23 = unpack_f16x2(h23);
          ph[hh][0] = movmatrix_trans(h01);
          ph[hh][1] = movmatrix_trans(h23);
          pl[hh][0] = movmatrix_trans(pack_f16x2(p0 - r01.x, p1 - r01.y));
          pl[hh][1] = movmatrix_trans(pack_f16x2(p2 - r23.x, p3 - r23.y));
        }
        uint32_t va[MT][4];
        v_frag<FMT, D>(boxV, boxVs, t, g, nvalid, va);
#pragma unroll
        for (int i = 0; i < MT; ++i)
#pragma unroll
          for (int hh = 0; hh < NH; ++hh) {
            mma_f16(o[i][hh], va[i][0], va[i][1], va[i][2], va[i][3], ph[hh][0], ph[hh][1]);
            mma_f16(o[i][hh], va[i][0], va[i][1], va[i][2], va[i][3], pl[hh][0], pl[hh][1]);
          }
      }
      // the box is consumed: refill its stage with this warp's load j + kRingStages
      __syncwarp();
      if (lane == 0 && issued < total) {
        fence_proxy_async_shared();   // generic reads of the stage before the async overwrite
        issue(issued++, st);
      }
      if (++st == kRingStages) {
        st = 0;
        phase ^= 1u;
      }
    }
    if constexpr (PROBQ) {
      if (sweep == 0) {
        // chunk max across the warps (every warp takes part, aborted or not)
        __syncwarp();
        if (g == 0) {
#pragma unroll
          for (int hh = 0; hh < NH; ++hh) {
            sm.m[warp][2 * t + 8 * hh] = m[hh][0];
            sm.m[warp][2 * t + 1 + 8 * hh] = m[hh][1];
          }
        }
        __syncthreads();
#pragma unroll
        for (int hh = 0; hh < NH; ++hh)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float mm = -INFINITY;
#pragma unroll
            for (int w = 0; w < NW; ++w) mm = fmaxf(mm, sm.m[w][2 * t + e + 8 * hh]);
            m[hh][e] = mm;
          }
        __syncthreads();
      }
    }
  }
  if (aborted) {
    *abort_flag = 1;
    record_error(a.error_flag, 1);
  }
  // Drain: no copy of this warp may still be writing shared memory later.
  if (lane == 0) {
    const int done = aborted ? 0 : total;
    for (int k = max(done, issued - kRingStages); k < issued; ++k)
      mbar_wait(smem_u32(&sm.full[warp][k % kRingStages]), (k / kRingStages) & 1);
  }
  __syncwarp();
  // per-warp state -> shared memory (m is uniform over the 8 lanes of a
  // head; l is summed over them)
#pragma unroll
  for (int hh = 0; hh < NH; ++hh)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = l[hh][e];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      l[hh][e] = v;
    }
  if (g == 0) {
#pragma unroll
    for (int hh = 0; hh < NH; ++hh)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        sm.m[warp][2 * t + e + 8 * hh] = m[hh][e];
        sm.l[warp][2 * t + e + 8 * hh] = l[hh][e];
      }
  }
  __syncthreads();   // every warp's ring is drained; m and l are in shared memory

  // O fragments -> the ring in fragment order, one 16-byte store per m-tile:
  // ofrag[warp][i][hh][lane] = (d0, 2t) (d0, 2t+1) (d0+1, 2t) (d0+1, 2t+1)
  // with d0 = (D/8) g + 2i, heads 2t + 8hh.  Meanwhile the first G threads
  // compute the warps' merge factors and the chunk's lse.
  float4* ofrag = reinterpret_cast<float4*>(dyn_smem + (ring - smem_u32(dyn_smem)));
  const bool bad = *abort_flag != 0;
#pragma unroll
  for (int i = 0; i < MT; ++i)
#pragma unroll
    for (int hh = 0; hh < NH; ++hh)
      ofrag[((warp * MT + i) * NH + hh) * 32 + lane] =
          make_float4(o[i][hh][0], o[i][hh][1], o[i][hh][2], o[i][hh][3]);
  const size_t part_row = ((size_t)b * a.Hq + (size_t)h * a.G);   // first query head
  // the grid ends after the preceding kernel in every mode
  if (!dep_done && threadIdx.x == 0) griddep_wait();
  if (threadIdx.x < a.G) {
    const int row = threadIdx.x;
    float M = -INFINITY;
    for (int w = 0; w < NW; ++w) M = fmaxf(M, sm.m[w][row]);
    float Ltot = 0.f;
    for (int w = 0; w < NW; ++w)
      if (sm.m[w][row] != -INFINITY) Ltot += ex2(sm.m[w][row] - M) * sm.l[w][row];
    for (int w = 0; w < NW; ++w)
      sm.fac[w][row] = (M == -INFINITY || sm.m[w][row] == -INFINITY || Ltot == 0.f)
                           ? 0.f
                           : ex2(sm.m[w][row] - M) / Ltot * out_mult;
    float lse = (M == -INFINITY || Ltot == 0.f) ? -INFINITY : (M + log2f(Ltot)) * kLn2;
    if (bad) lse = NAN;
    a.part_lse[(part_row + row) * a.num_splits + split] = lse;
  }
  __syncthreads();

  // ---------------------------------------------------------------- merge
  // item (i, hh, lane'): heads h0 = 2t' + 8hh and h0 + 1, dims d0 and d0 + 1
  for (int it = threadIdx.x; it < MT * NH * 32; it += (32 * NW)) {
    const int ln = it & 31, hh = (it >> 5) % NH, i = (it >> 5) / NH;
    const int h0 = 2 * (ln & 3) + 8 * hh;
    if (h0 >= a.G) continue;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float4 v = ofrag[((w * MT + i) * NH + hh) * 32 + ln];
      const float f0 = sm.fac[w][h0], f1 = sm.fac[w][h0 + 1];
      acc.x += f0 * v.x;
      acc.y += f1 * v.y;
      acc.z += f0 * v.z;
      acc.w += f1 * v.w;
    }
    if (bad) acc = make_float4(NAN, NAN, NAN, NAN);
    const int d0 = (D / 8) * (ln >> 2) + 2 * i;
    float* r0 = a.part_o + ((part_row + h0) * a.num_splits + split) * D + d0;
    *reinterpret_cast<float2*>(r0) = make_float2(acc.x, acc.z);
    if (h0 + 1 < a.G) *reinterpret_cast<float2*>(r0 + (size_t)a.num_splits * D) =
        make_float2(acc.y, acc.w);
  }
  // fused combine: the G rows' partials staged at the ring base (the O
  // fragments are written out), the weights at the ring end
  if (a.counters) {
    // staging area: everything from the ring base to the end of the dynamic
    // shared memory (the launcher sizes it for the call's partials when the
    // SM's residency allows), the weights at its end
    constexpr uint32_t kWbuf = (kMaxGroup * kMaxFusedSplits + kMaxGroup) * 4;
    uint32_t dyn_bytes;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_bytes));
    const uint32_t usable = dyn_bytes - (ring - smem_u32(dyn_smem));
    fused_combine_staged<ctas_per_sm<FMT, D, PROBQ, NH, NW>() == 4 ? 16 : 32>(
        a, bh, part_row, a.G, ring, reinterpret_cast<const float*>(ofrag), usable - kWbuf,
        reinterpret_cast<float*>(dyn_smem + (ring - smem_u32(dyn_smem)) + usable - kWbuf),
        smem_u32(&sm.comb_full));
  }
}

template <int FMT, int D, bool PROBQ, int NH, bool QF8, int NW>
cudaError_t launch_partial_t(const TensorMaps& m, const PartialArgs& a, cudaStream_t st) {
  using Rg = Ring<FMT, D, PROBQ, NH, NW>;
  static_assert(Rg::kBytes >= Rg::kEpilogue && Rg::kBytes >= Rg::kStream, "ring too small");
  size_t smem = 1024 + (size_t)Rg::kBytes + (PROBQ ? (size_t)a.score_floats * 4 : 0);
  if (a.counters) {
    // room for the fused merge to stage its partials (G rows x s splits x Dv
    // floats, and the weights) in one bulk copy, within the shared memory
    // that keeps ctas_per_sm CTAs resident (228 KB per SM, 1 KB reserved per
    // CTA, the static part under 4 KB, the alignment slack)
    constexpr size_t kPerCta = 233472 / ctas_per_sm<FMT, D, PROBQ, NH, NW>() - 1024 - 4096 - 1024;
    const size_t need = 1024 + (size_t)a.G * a.num_splits * a.Dv * 4 +
                        (kMaxGroup * kMaxFusedSplits + kMaxGroup) * 4;
    smem = std::max(smem, std::min(need, kPerCta));
  }
  smem = (smem + 15) / 16 * 16;
  auto kern = partial_kernel<FMT, D, PROBQ, NH, QF8, NW>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(a.batch * a.Hkv, a.num_splits), dim3(32 * NW), smem, st,
                    m.k16, m.v16, a);
}

template <int FMT, int D, bool QF8>
cudaError_t dispatch_nh(bool probq, const TensorMaps& m, const PartialArgs& a, cudaStream_t st) {
  if (a.G <= 8) {
    if (probq) return launch_partial_t<FMT, D, true, 1, QF8, kDecodeWarps>(m, a, st);
    if constexpr (D <= 128)
      if (wide_cta(D, false, a.G)) return launch_partial_t<FMT, D, false, 1, QF8, kWideWarps>(m, a, st);
    return launch_partial_t<FMT, D, false, 1, QF8, kDecodeWarps>(m, a, st);
  }
  return probq ? launch_partial_t<FMT, D, true, 2, QF8, kDecodeWarps>(m, a, st)
               : launch_partial_t<FMT, D, false, 2, QF8, kDecodeWarps>(m, a, st);
}

template <int FMT, int D>
cudaError_t dispatch_q(bool probq, const TensorMaps& m, const PartialArgs& a, cudaStream_t st) {
  return a.q_fp8 ? dispatch_nh<FMT, D, true>(probq, m, a, st)
                 : dispatch_nh<FMT, D, false>(probq, m, a, st);
}

}  // namespace decode_impl
}  // namespace kvq
