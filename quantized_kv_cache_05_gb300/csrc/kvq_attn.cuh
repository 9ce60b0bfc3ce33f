// Device-side pieces shared by the split-KV decode kernels (GQA/MHA and
// MLA): ring geometry, register-level fragment decoders for the tensor-core
// operands, bounded barrier waits, and the merge of split partials.
#pragma once

#include <cmath>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazyMax = 8.0f;   // log2 headroom before the running max moves

template <int FMT, int D>
struct Geom {
  static constexpr int kRow = FMT == kFmtFp8 ? D : D / 2;   // code bytes per token row
  static constexpr int kSRow = FMT == kFmtFp8 ? 0 : D / 16; // scale bytes per token row
  static constexpr int kBoxK = kBoxTokens * kRow;            // code bytes of one box
  static constexpr int kBoxS = kBoxTokens * kSRow;           // scale bytes of one box
  // one ring stage: [K codes][V codes][K scales][V scales], padded so that
  // every stage starts on the swizzle period (1024 bytes; 128 bytes for
  // unswizzled 32-byte rows)
  static constexpr int kAlign = kRow >= 64 ? 1024 : 128;
  static constexpr int kStage = (2 * (kBoxK + kBoxS) + kAlign - 1) / kAlign * kAlign;
  // FP8-probability mode streams K and V in separate sweeps: a stage holds
  // one box of one tensor, [codes][scales]
  static constexpr int kStage1 = (kBoxK + kBoxS + kAlign - 1) / kAlign * kAlign;
  static constexpr int kKSteps = D / 16;   // QK k-steps over head_dim
  static constexpr int kMT = D / 16;       // PV m-tiles over v_dim
  static_assert(kRow == 32 || kRow == 64 || kRow == 128, "code rows of 32, 64 or 128 bytes");
  // physical 16-byte chunk of logical chunk `ch` in row `row` of a box (the
  // TMA swizzle of the row width: 128-byte, 64-byte, none for 32 bytes)
  __device__ static __forceinline__ int swz(int row, int ch) {
    if constexpr (kRow == 128) return ch ^ (row & 7);
    else if constexpr (kRow == 64) return ch ^ ((row >> 1) & 3);
    else return ch;
  }
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
// K fragments (B operand of S = Q K^T) for one 8-token n-tile: b[j][0..1] for
// k-step j.  Lane (g, t) holds token row `row` (= 8u + g) and head dims
//   d = (D/4) t + 4 j + {0, 1} (b[j][0]) and + {2, 3} (b[j][1]).
// ---------------------------------------------------------------------------
template <int FMT, int D, int SSTRIDE = Geom<FMT, D>::kSRow>
__device__ __forceinline__ void k_frag(uint32_t boxK, uint32_t boxKs, int row, int t,
                                       uint32_t (&b)[D / 16][2]) {
  using Gm = Geom<FMT, D>;
  if constexpr (FMT == kFmtFp8) {
    constexpr int NCH = D / 64;  // 16-byte chunks per lane per row
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      uint4 v = lds128(boxK + row * Gm::kRow + (Gm::swz(row, t * NCH + i) << 4));
      e4m3x4_to_f16x2x2(v.x, b[i * 4 + 0][0], b[i * 4 + 0][1]);
      e4m3x4_to_f16x2x2(v.y, b[i * 4 + 1][0], b[i * 4 + 1][1]);
      e4m3x4_to_f16x2x2(v.z, b[i * 4 + 2][0], b[i * 4 + 2][1]);
      e4m3x4_to_f16x2x2(v.w, b[i * 4 + 3][0], b[i * 4 + 3][1]);
    }
  } else {
    // NVFP4: the lane's D/4 dims are D/8 code bytes (D/32 words) and D/64
    // blocks; word k is scaled by block k/2 of the lane's range
    constexpr int NWK = D / 32;
    uint32_t w[NWK];
    if constexpr (D == 64) {
      const uint2 v = lds64(boxK + row * Gm::kRow + 8 * t);
      w[0] = v.x; w[1] = v.y;
    } else if constexpr (D == 128) {
      const uint4 v = lds128(boxK + row * Gm::kRow + (Gm::swz(row, t) << 4));
      w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else {
      static_assert(D == 256, "NVFP4 decode supports head_dim 64, 128 and 256");
      const uint4 v0 = lds128(boxK + row * Gm::kRow + (Gm::swz(row, 2 * t) << 4));
      const uint4 v1 = lds128(boxK + row * Gm::kRow + (Gm::swz(row, 2 * t + 1) << 4));
      w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
      w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
    }
    // f16 block scales, each duplicated into both halves
    constexpr int NB = (NWK + 1) / 2;
    uint32_t sc[NB];
    if constexpr (D == 64) {
      const uint32_t s2 = e4m3x2_to_f16x2(lds8(boxKs + row * SSTRIDE + t));
      sc[0] = __byte_perm(s2, 0, 0x1010);
    } else if constexpr (D == 128) {
      const uint32_t s2 = e4m3x2_to_f16x2(lds16(boxKs + row * SSTRIDE + 2 * t));
      sc[0] = __byte_perm(s2, 0, 0x1010);
      sc[1] = __byte_perm(s2, 0, 0x3232);
    } else {
      const uint32_t s4 = lds32(boxKs + row * SSTRIDE + 4 * t);
      const uint32_t sa = e4m3x2_to_f16x2(s4 & 0xFFFFu), sb = e4m3x2_to_f16x2(s4 >> 16);
      sc[0] = __byte_perm(sa, 0, 0x1010);
      sc[1] = __byte_perm(sa, 0, 0x3232);
      sc[2] = __byte_perm(sb, 0, 0x1010);
      sc[3] = __byte_perm(sb, 0, 0x3232);
    }
#pragma unroll
    for (int k = 0; k < NWK; ++k) {
      uint32_t o0, o1, o2, o3;
      e2m1x8_to_f16x2x4(w[k], o0, o1, o2, o3);
      const uint32_t s = sc[k >> 1];
      b[2 * k][0] = hmul2(o0, s);
      b[2 * k][1] = hmul2(o1, s);
      b[2 * k + 1][0] = hmul2(o2, s);
      b[2 * k + 1][1] = hmul2(o3, s);
    }
  }
}

// ---------------------------------------------------------------------------
// Raw FP8 K codes for the E4M3 x E4M3 score MMA (m16n8k32; FP8 query): lane
// (g, t) takes the D/4 code bytes (D/4) t .. of token row `row` as D/16
// words, unconverted.  Word 2j feeds the k-columns 4t..4t+3 of k-step j
// (head dims (D/4) t + 8j .. +3), word 2j + 1 the columns 4t+16..19 (dims
// (D/4) t + 8j + 4 .. +7); the FP8 query is loaded with the same mapping.
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void k_raw_fp8(uint32_t boxK, int row, int t, uint32_t (&w)[D / 16]) {
  using Gm = Geom<kFmtFp8, D>;
  constexpr int NCH = D / 64;   // 16-byte chunks per lane per row
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const uint4 v = lds128(boxK + row * Gm::kRow + (Gm::swz(row, t * NCH + i) << 4));
    w[4 * i + 0] = v.x;
    w[4 * i + 1] = v.y;
    w[4 * i + 2] = v.z;
    w[4 * i + 3] = v.w;
  }
}

// ---------------------------------------------------------------------------
// V^T fragments (A operand of O^T = V^T P^T) for the box's 16 tokens:
// a[i][0..3] for m-tile i.  Lane (g, t) covers tokens 2t, 2t+1 (a0, a1) and
// 2t+8, 2t+9 (a2, a3); m-tile i, row g is value dim (D/8) g + 2 i and row
// g + 8 is (D/8) g + 2 i + 1.  Invalid tokens (rows past the chunk) give
// zero: FP8 codes are zeroed, NVFP4 block scales are zeroed (every E2M1 code
// is finite, so the products are zero).
// ---------------------------------------------------------------------------
template <int FMT, int D, int SSTRIDE = Geom<FMT, D>::kSRow>
__device__ __forceinline__ void v_frag(uint32_t boxV, uint32_t boxVs, int t, int g, int nvalid,
                                       uint32_t (&a)[D / 16][4]) {
  using Gm = Geom<FMT, D>;
  const int tk[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
  if constexpr (FMT == kFmtFp8) {
    constexpr int NW = D / 32;   // words per lane per token (4 for D=128, 2 for D=64)
    uint32_t w[4][NW];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if constexpr (D == 128) {
        uint4 v = lds128(boxV + tk[r] * 128 + (Gm::swz(tk[r], g) << 4));
        w[r][0] = v.x; w[r][1] = v.y; w[r][2] = v.z; w[r][3] = v.w;
      } else {
        uint2 v = lds64(boxV + tk[r] * 64 + (Gm::swz(tk[r], g >> 1) << 4) + ((g & 1) << 3));
        w[r][0] = v.x; w[r][1] = v.y;
      }
    }
    if (nvalid < kBoxTokens) {   // ragged box: rows past the chunk read as zero codes
#pragma unroll
      for (int r = 0; r < 4; ++r)
        if (tk[r] >= nvalid) {
#pragma unroll
          for (int k = 0; k < NW; ++k) w[r][k] = 0u;
        }
    }
#pragma unroll
    for (int k = 0; k < NW; ++k) {
      // token pairs (2t, 2t+1) and (2t+8, 2t+9), one byte of each per value dim
      const uint32_t p0 = __byte_perm(w[0][k], w[1][k], 0x5140);
      const uint32_t p1 = __byte_perm(w[0][k], w[1][k], 0x7362);
      const uint32_t q0 = __byte_perm(w[2][k], w[3][k], 0x5140);
      const uint32_t q1 = __byte_perm(w[2][k], w[3][k], 0x7362);
      e4m3x4_to_f16x2x2(p0, a[2 * k][0], a[2 * k][1]);
      e4m3x4_to_f16x2x2(q0, a[2 * k][2], a[2 * k][3]);
      e4m3x4_to_f16x2x2(p1, a[2 * k + 1][0], a[2 * k + 1][1]);
      e4m3x4_to_f16x2x2(q1, a[2 * k + 1][2], a[2 * k + 1][3]);
    }
  } else {
    // NVFP4: lane g's value dims (D/8) g .. are D/16 code bytes per token
    // (NW words) in D/128 blocks (one for D <= 128); word k is scaled by
    // block k/2 of the lane's range
    constexpr int NW = D / 64;
    constexpr int NB = (NW + 1) / 2;
    uint32_t v[4][NW];
    uint32_t sc[4][NB];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if constexpr (D == 64) {
        v[r][0] = lds32(boxV + tk[r] * Gm::kRow + 4 * g);
        sc[r][0] = lds8(boxVs + tk[r] * SSTRIDE + (g >> 1));
      } else if constexpr (D == 128) {
        const uint2 x = lds64(boxV + tk[r] * Gm::kRow + (Gm::swz(tk[r], g >> 1) << 4) +
                              ((g & 1) << 3));
        v[r][0] = x.x; v[r][1] = x.y;
        sc[r][0] = lds8(boxVs + tk[r] * SSTRIDE + g);
      } else {
        static_assert(FMT == kFmtNvfp4 && D == 256, "unsupported V layout");
        const uint4 x = lds128(boxV + tk[r] * Gm::kRow + (Gm::swz(tk[r], g) << 4));
        v[r][0] = x.x; v[r][1] = x.y; v[r][2] = x.z; v[r][3] = x.w;
        const uint32_t s2 = lds16(boxVs + tk[r] * SSTRIDE + 2 * g);
        sc[r][0] = s2 & 0xFFu;
        sc[r][1] = s2 >> 8;
      }
    }
    if (nvalid < kBoxTokens) {   // ragged box: rows past the chunk scale to zero
#pragma unroll
      for (int r = 0; r < 4; ++r)
        if (tk[r] >= nvalid) {
#pragma unroll
          for (int k = 0; k < NB; ++k) sc[r][k] = 0u;
        }
    }
    uint32_t s01[NB], s89[NB];   // (scale of token 2t, 2t+1) and (2t+8, 2t+9)
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      s01[k] = e4m3x2_to_f16x2(sc[0][k] | (sc[1][k] << 8));
      s89[k] = e4m3x2_to_f16x2(sc[2][k] | (sc[3][k] << 8));
    }
#pragma unroll
    for (int k = 0; k < NW; ++k) {
      const uint32_t A = v[0][k], B = v[1][k], C = v[2][k], E = v[3][k];
      const uint32_t evAB = (A & 0x0F0F0F0Fu) | ((B & 0x0F0F0F0Fu) << 4);
      const uint32_t odAB = ((A >> 4) & 0x0F0F0F0Fu) | (B & 0xF0F0F0F0u);
      const uint32_t evCE = (C & 0x0F0F0F0Fu) | ((E & 0x0F0F0F0Fu) << 4);
      const uint32_t odCE = ((C >> 4) & 0x0F0F0F0Fu) | (E & 0xF0F0F0F0u);
      uint32_t e[4], o[4], f[4], h[4];
      e2m1x8_to_f16x2x4(evAB, e[0], e[1], e[2], e[3]);
      e2m1x8_to_f16x2x4(odAB, o[0], o[1], o[2], o[3]);
      e2m1x8_to_f16x2x4(evCE, f[0], f[1], f[2], f[3]);
      e2m1x8_to_f16x2x4(odCE, h[0], h[1], h[2], h[3]);
      const uint32_t sa = s01[k >> 1], sb = s89[k >> 1];
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        const int i = 4 * k + bb;   // value dims (D/8) g + 8k + 2bb (+1)
        a[i][0] = hmul2(e[bb], sa);
        a[i][1] = hmul2(o[bb], sa);
        a[i][2] = hmul2(f[bb], sb);
        a[i][3] = hmul2(h[bb], sb);
      }
    }
  }
}

// Column swizzle of the end-of-chunk O buffer [warp][head][d]: XOR-ing the
// low bits of d with (head pair, high bits of the lane group) makes both the
// fragment stores and the row-wise merge reads conflict-free.
template <int D>
__device__ __forceinline__ int obuf_swz(int head, int d) {
  constexpr int kLog = D == 128 ? 4 : 3;   // log2(D / 8): dims per lane group
  const int grp = d >> kLog;
  return d ^ ((((head >> 1) & 3) | ((grp >> (5 - kLog)) << 2)) & ((D / 8) - 1));
}

// Output of one element in the requested type: fp32, bf16 (round to nearest
// even) or the E4M3 code of fl32(o / out_scale).
template <int DT>
__device__ __forceinline__ void store_out_t(void* out, float out_scale, size_t i, float v) {
  if constexpr (DT == 0) {
    static_cast<float*>(out)[i] = v;
  } else if constexpr (DT == 1) {
    static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
  } else {
    static_cast<uint8_t*>(out)[i] = (uint8_t)(f32x2_to_e4m3x2(__fdiv_rn(v, out_scale), 0.f) & 0xFFu);
  }
}


// Merge of the s split partials of `rows` consecutive query heads starting at
// partial row `row0` (M = max lse, w_j = e^(lse_j - M), O = sum w_j o_j /
// sum w_j; O = 0 when every split is empty), written to `out` in the
// requested type.  Threads own float4 columns (four consecutive value dims
// of one row); one round of loads covers NI columns x NS splits (NI * NS =
// DEPTH): one column at a time for many splits, several for few splits, so
// that a thread's columns need few memory round trips.  The first round is
// issued before the weights are known.  One warp per head row computes the
// weights (warp reductions).  w: rows * kMaxFusedSplits floats of shared
// memory (s <= kMaxFusedSplits), winv: rows floats.  The caller
// synchronizes before.
template <int NI, int NS>
struct MergeRound {
  float4 v[NI][NS];
  __device__ __forceinline__ void load(const float* __restrict__ part_o, size_t row0, int s,
                                       int nq, int items, int i, int j0) {
#pragma unroll
    for (int u = 0; u < NI; ++u) {
      const int it = i + u * (int)blockDim.x;
      const float4* po =
          reinterpret_cast<const float4*>(part_o + (row0 + it / nq) * (size_t)s * nq * 4) + it % nq;
#pragma unroll
      for (int k = 0; k < NS; ++k)
        v[u][k] = (it < items && j0 + k < s) ? __ldcg(po + (size_t)(j0 + k) * nq)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
};

template <int NI, int NS, int DT>
__device__ __forceinline__ void merge_columns(const float* __restrict__ part_o, size_t row0,
                                              int rows, int s, int Dv, const float* w,
                                              const float* winv, void* out, float out_scale,
                                              MergeRound<NI, NS>& rd, bool first_loaded) {
  const int nq = Dv / 4, items = rows * nq, nt = blockDim.x;
  for (int i = threadIdx.x; i < items; i += NI * nt) {
    float4 acc[NI];
#pragma unroll
    for (int u = 0; u < NI; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < s; j0 += NS) {
      if (!(first_loaded && i == (int)threadIdx.x && j0 == 0))
        rd.load(part_o, row0, s, nq, items, i, j0);
#pragma unroll
      for (int u = 0; u < NI; ++u) {
        const int it = min(i + u * nt, items - 1);
        const float* wr = w + (it / nq) * kMaxFusedSplits;
#pragma unroll
        for (int k = 0; k < NS; ++k) {
          const float wk = j0 + k < s ? wr[j0 + k] : 0.f;
          acc[u].x += wk * rd.v[u][k].x;
          acc[u].y += wk * rd.v[u][k].y;
          acc[u].z += wk * rd.v[u][k].z;
          acc[u].w += wk * rd.v[u][k].w;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < NI; ++u) {
      const int it = i + u * nt;
      if (it >= items) break;
      const int r = it / nq;
      const float iv = winv[r];
      const size_t o = (row0 + r) * Dv + 4 * (it % nq);
      store_out_t<DT>(out, out_scale, o + 0, acc[u].x * iv);
      store_out_t<DT>(out, out_scale, o + 1, acc[u].y * iv);
      store_out_t<DT>(out, out_scale, o + 2, acc[u].z * iv);
      store_out_t<DT>(out, out_scale, o + 3, acc[u].w * iv);
    }
  }
}

__device__ __forceinline__ void merge_weights(const float* __restrict__ part_lse, size_t row0,
                                              int rows, int s, float* w, float* winv) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = warp; r < rows; r += blockDim.x >> 5) {
    const float* lse = part_lse + (row0 + r) * s;
    float lv[kMaxFusedSplits / 32];
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kMaxFusedSplits / 32; ++k) {
      const int j = lane + 32 * k;
      lv[k] = j < s ? __ldcg(lse + j) : -INFINITY;
      M = fmaxf(M, lv[k]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxFusedSplits / 32; ++k) {
      const int j = lane + 32 * k;
      const float e = (M == -INFINITY || lv[k] == -INFINITY) ? 0.f : expf(lv[k] - M);
      if (j < s) w[r * kMaxFusedSplits + j] = e;
      sum += e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) winv[r] = sum > 0.f ? 1.f / sum : (sum == 0.f ? 0.f : NAN);
  }
}

template <int NI, int NS>
__device__ __forceinline__ void merge_rows_t(const float* __restrict__ part_o,
                                             const float* __restrict__ part_lse, size_t row0,
                                             int rows, int s, int Dv, float* w, float* winv,
                                             void* out, int out_dtype, float out_scale) {
  MergeRound<NI, NS> rd;
  const int items = rows * (Dv / 4);
  if ((int)threadIdx.x < items) rd.load(part_o, row0, s, Dv / 4, items, threadIdx.x, 0);
  merge_weights(part_lse, row0, rows, s, w, winv);
  __syncthreads();
  const bool first = (int)threadIdx.x < items;
  if (out_dtype == 0)
    merge_columns<NI, NS, 0>(part_o, row0, rows, s, Dv, w, winv, out, out_scale, rd, first);
  else if (out_dtype == 1)
    merge_columns<NI, NS, 1>(part_o, row0, rows, s, Dv, w, winv, out, out_scale, rd, first);
  else
    merge_columns<NI, NS, 2>(part_o, row0, rows, s, Dv, w, winv, out, out_scale, rd, first);
}

template <int DEPTH = 32>
__device__ __forceinline__ void merge_rows(const float* __restrict__ part_o,
                                           const float* __restrict__ part_lse, size_t row0,
                                           int rows, int s, int Dv, float* w, float* winv,
                                           void* out, int out_dtype, float out_scale) {
  const int cols_per_thread = (rows * (Dv / 4) + (int)blockDim.x - 1) / (int)blockDim.x;
  if (cols_per_thread >= 4 && 4 * s <= DEPTH)
    merge_rows_t<4, DEPTH / 4>(part_o, part_lse, row0, rows, s, Dv, w, winv, out, out_dtype,
                               out_scale);
  else
    merge_rows_t<1, DEPTH>(part_o, part_lse, row0, rows, s, Dv, w, winv, out, out_dtype,
                           out_scale);
}

// Weighted sum of cnt staged splits of one (row, 4 value dims) item: p points
// at the item's first split, consecutive splits nq float4 apart; wr holds the
// splits' weights.  The loads run four splits ahead, the adds stay in split
// order (the same sums, bit for bit, as the global-memory merge).
__device__ __forceinline__ float4 accum_splits(const float4* p, int nq, const float* wr, int cnt,
                                               float4 acc) {
  int j = 0;
#pragma unroll 1
  for (; j + 4 <= cnt; j += 4) {
    float4 v[4];
    float wj[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[k] = p[(size_t)(j + k) * nq];
      wj[k] = wr[j + k];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc.x += wj[k] * v[k].x;
      acc.y += wj[k] * v[k].y;
      acc.z += wj[k] * v[k].z;
      acc.w += wj[k] * v[k].w;
    }
  }
#pragma unroll 1
  for (; j < cnt; ++j) {
    const float4 v = p[(size_t)j * nq];
    const float wj = wr[j];
    acc.x += wj * v.x;
    acc.y += wj * v.y;
    acc.z += wj * v.z;
    acc.w += wj * v.w;
  }
  return acc;
}

template <int DT>
__device__ __forceinline__ void store_item(const PartialArgs& a, size_t row0, int r, int d4,
                                           float4 acc, float iv) {
  const size_t o = (row0 + r) * a.Dv + 4 * d4;
  store_out_t<DT>(a.out, a.out_scale, o + 0, acc.x * iv);
  store_out_t<DT>(a.out, a.out_scale, o + 1, acc.y * iv);
  store_out_t<DT>(a.out, a.out_scale, o + 2, acc.z * iv);
  store_out_t<DT>(a.out, a.out_scale, o + 3, acc.w * iv);
}

// Staged merge: the s partials of rows [row0, row0 + rows) are contiguous in
// global memory ([row][split][Dv] floats); with them in shared memory (one
// bulk copy) the weighted sum is a short loop, four value dims per thread and
// step.
template <int DT>
__device__ __forceinline__ void merge_staged(const PartialArgs& a, size_t row0, int rows,
                                             const float* staged, const float* w,
                                             const float* winv, bool ok) {
  const int s = a.num_splits, nq = a.Dv / 4;
  const float4* po = reinterpret_cast<const float4*>(staged);
#pragma unroll 1
  for (int i = threadIdx.x; i < rows * nq; i += blockDim.x) {
    const int r = i / nq, d4 = i % nq;
    const float4 acc = accum_splits(po + (size_t)r * s * nq + d4, nq, w + r * kMaxFusedSplits, s,
                                    make_float4(0.f, 0.f, 0.f, 0.f));
    store_item<DT>(a, row0, r, d4, acc, ok ? winv[r] : NAN);
  }
}

// Fused combine with staging: the arrival protocol of fused_combine; the
// last CTA brings its rows' partials into shared memory with one bulk copy
// when they fit in `cap` bytes at `stage` (16-byte aligned, free), else it
// runs the general merge from global memory.  (Splitting the copy into
// rounds of a few splits per row was measured slower than the global merge:
// the row pieces are separate bulk copies, each a full round trip.)  The
// async-proxy read follows the acquire, behind a proxy fence.  bar: an
// mbarrier initialized with one arrival and unused so far; wbuf: kMaxGroup *
// (kMaxFusedSplits + 1) floats outside the stage.
template <int DEPTH = 32, int NI = 1>
__device__ __forceinline__ void fused_combine_staged(const PartialArgs& a, int bh, size_t part_row,
                                                     int rows, uint32_t stage, const float* stage_p,
                                                     uint32_t cap, float* wbuf, uint32_t bar) {
  __shared__ int is_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(prev)
                 : "l"(a.counters + bh)
                 : "memory");
    is_last = prev == (unsigned)(a.num_splits - 1);
    if (is_last) a.counters[bh] = 0u;
  }
  __syncthreads();
  if (!is_last) return;
  const int s = a.num_splits;
  float* winv = wbuf + kMaxGroup * kMaxFusedSplits;
  const uint64_t bytes = (uint64_t)rows * s * a.Dv * 4;
  if (bytes > cap) {
    merge_rows_t<NI, DEPTH / NI>(a.part_o, a.part_lse, part_row, rows, s, a.Dv, wbuf, winv,
                                 a.out, a.out_dtype, a.out_scale);
    return;
  }
  if (threadIdx.x == 0) {
    asm volatile("fence.proxy.async.global;" ::: "memory");   // acquired data -> bulk copy
    mbar_arrive_expect_tx(bar, (uint32_t)bytes);
    bulk_load(stage, a.part_o + part_row * s * a.Dv, (uint32_t)bytes, bar);
  }
  merge_weights(a.part_lse, part_row, rows, s, wbuf, winv);
  const bool ok = __syncthreads_and(mbar_wait(bar, 0) ? 1 : 0) != 0;
  if (a.out_dtype == 0)
    merge_staged<0>(a, part_row, rows, stage_p, wbuf, winv, ok);
  else if (a.out_dtype == 1)
    merge_staged<1>(a, part_row, rows, stage_p, wbuf, winv, ok);
  else
    merge_staged<2>(a, part_row, rows, stage_p, wbuf, winv, ok);
  if (!ok && threadIdx.x == 0) record_error(a.error_flag, 1);
}

// Merge through distributed shared memory, for a launch in clusters of the
// s <= 8 splits of a request (cluster rank = split): every CTA holds its
// normalized partial [rows][Dv] fp32 at shared address `own` and its lse
// [rows] at `own_lse`.  After a cluster barrier eight lanes per row form the
// row's weights from the peers' lse, and CTA rank r computes items
// [r n / s, (r + 1) n / s) of the n = rows Dv / 4 (row, 4 value dims) items,
// loading each item's s partials from the peers' shared memory in one round;
// a second barrier keeps every CTA's shared memory until its peers are done.
// No partial goes to global memory and no arrival counter is used.
//
// The result is bit for bit that of the global-memory merge: the weights are
// merge_weights' (the max is order-free; its butterfly sum over 32 lanes, of
// which lanes >= s hold exact zeros, is for s <= 8 the pairwise sum
// ((e0 + e4) + (e2 + e6)) + ((e1 + e5) + (e3 + e7)) with e_j = 0 for j >= s),
// and the weighted sum runs in split order like accum_splits.
// wbuf: kMaxGroup * (kMaxFusedSplits + 1) floats of this CTA's shared memory.
// (Measured on MLA: loading two items per thread before the weights, or
// forming the weights in every thread, made the merge slower.)
constexpr int kMaxClusterSplits = 8;   // portable cluster size

template <int DT>
__device__ __forceinline__ void merge_cluster_items(const PartialArgs& a, size_t row0, int rows,
                                                    uint32_t own, const float* w,
                                                    const float* winv) {
  const int s = a.num_splits, nq = a.Dv / 4, n = rows * nq;
  const int rank = (int)cluster_ctarank();
  const int i0 = (int)(((long)n * rank) / s), i1 = (int)(((long)n * (rank + 1)) / s);
  uint32_t peer[kMaxClusterSplits];
#pragma unroll
  for (int j = 0; j < kMaxClusterSplits; ++j) peer[j] = cluster_map(own, j < s ? j : 0);
#pragma unroll 1
  for (int i = i0 + (int)threadIdx.x; i < i1; i += blockDim.x) {
    const int r = i / nq, d4 = i % nq;
    const uint32_t off = (uint32_t)(r * a.Dv + 4 * d4) * 4u;
    float4 v[kMaxClusterSplits];
#pragma unroll
    for (int j = 0; j < kMaxClusterSplits; ++j)
      if (j < s) v[j] = ld_cluster_v4(peer[j] + off);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kMaxClusterSplits; ++j)
      if (j < s) {
        const float wj = w[r * kMaxFusedSplits + j];
        acc.x += wj * v[j].x;
        acc.y += wj * v[j].y;
        acc.z += wj * v[j].z;
        acc.w += wj * v[j].w;
      }
    store_item<DT>(a, row0, r, d4, acc, winv[r]);
  }
}

__device__ __forceinline__ void fused_combine_cluster(const PartialArgs& a, size_t row0, int rows,
                                                      uint32_t own, uint32_t own_lse,
                                                      float* wbuf) {
  cluster_sync_all();   // every split's partial and lse are written
  const int s = a.num_splits;
  float* winv = wbuf + kMaxGroup * kMaxFusedSplits;
  // weights: eight lanes per row, lane j for split j (lse -inf for j >= s);
  // the xor-4/2/1 butterfly of (own + other) leaves lane 0 of the group with
  // ((e0 + e4) + (e2 + e6)) + ((e1 + e5) + (e3 + e7))
  if ((int)threadIdx.x < ((rows * kMaxClusterSplits + 31) & ~31)) {
    const int r = (int)threadIdx.x / kMaxClusterSplits, j = (int)threadIdx.x % kMaxClusterSplits;
    const bool in = r < rows && j < s;
    const float lv = in ? ld_cluster_f32(cluster_map(own_lse + 4u * r, j)) : -INFINITY;
    float M = lv;
#pragma unroll
    for (int o = kMaxClusterSplits / 2; o > 0; o >>= 1)
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float e = (M == -INFINITY || lv == -INFINITY) ? 0.f : expf(lv - M);
    if (in) wbuf[r * kMaxFusedSplits + j] = e;
    float sum = e;
#pragma unroll
    for (int o = kMaxClusterSplits / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (r < rows && j == 0) winv[r] = sum > 0.f ? 1.f / sum : (sum == 0.f ? 0.f : NAN);
  }
  __syncthreads();
  if (a.out_dtype == 0)
    merge_cluster_items<0>(a, row0, rows, own, wbuf, winv);
  else if (a.out_dtype == 1)
    merge_cluster_items<1>(a, row0, rows, own, wbuf, winv);
  else
    merge_cluster_items<2>(a, row0, rows, own, wbuf, winv);
  cluster_sync_all();   // the peers have read this CTA's partial
}

}  // namespace kvq
