// Prefill attention over a quantized KV cache (sm_103a): causal, no KV split.
//
// Model-Optimizer PR 1832 times a prefill attention kernel next to its
// split-KV decode (the latency tables' prefill column, with "batch=1 x 32
// heads = 32 base programs").  This kernel computes, for Tq new tokens per
// request that the cache already holds (query i at position L - Tq + i),
// causal attention over the cache: query i attends to keys 0 .. L - Tq + i.
// With Tq = 1 it is one program per (request, kv head) over the whole
// sequence -- the pages' comparison setting.
//
// GB300 design.  A CTA takes 64 query rows (row = query token * G + head of
// one kv head) -- 16 per consumer warp -- of one (request, kv head); a fifth
// warp streams the 16-token K/V boxes with TMA into a 4-stage ring that the
// consumer warps read (full/empty mbarriers).  A tile with fewer than four
// 16-row groups (few new tokens, e.g. one: the decode shape) lends its idle
// warps to the keys: with nrg row groups, nkg = 4 / nrg warps share each
// group's rows and take every nkg-th box, and their softmax states are merged
// through shared memory at the end.  Per box and warp, on mma.sync
// m16n8k16 (f16 operands, fp32 accumulation):
//   S = Q K^T   A = Q (16 rows, head dims permuted per lane like the K
//               fragments), B = K^T from the decoded K box (k_frag), two
//               8-key n-tiles
//   O += P V    A = P straight from the S accumulators (f16 high part plus
//               f16 residual), B = V from the decoded V box (v_frag), D/8
//               n-tiles of value dims
// with the online softmax per row (lazy reference max) and the causal mask.
// The query rows are prescaled per row by a power of two (the full bf16
// range, as in the decode).  Every wait is bounded; a timeout sets an error
// bit and the rows become NaN.

#include "kvq_attn.cuh"

namespace kvq {
namespace {

constexpr int kPfConsumers = 4;                      // 16 query rows each
constexpr int kPfRows = 16 * kPfConsumers;           // query rows per CTA
constexpr int kPfThreads = 32 * (kPfConsumers + 1);  // + the producer warp
constexpr int kPfStages = 4;

struct PfSmem {
  uint64_t full[kPfStages];
  uint64_t empty[kPfStages];
  int pages[kPageCache];
  int abort_flag;
};

template <int FMT, int D>
__global__ void __launch_bounds__(kPfThreads)
    prefill_kernel(const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const PartialArgs a) {
  using Gm = Geom<FMT, D>;
  constexpr int KS = Gm::kKSteps;
  constexpr int MT = Gm::kMT;
  constexpr int NT = D / 8;   // value-dim n-tiles of O

  extern __shared__ uint8_t dyn_smem[];
  __shared__ PfSmem sm;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int bh = blockIdx.y, b = bh / a.Hkv, h = bh % a.Hkv;
  const int R = a.q_len * a.G;                  // query rows of the request
  const int r0 = blockIdx.x * kPfRows;          // first row of this tile
  const int nrg = min(kPfConsumers, (R - r0 + 15) / 16);   // 16-row groups with rows
  const int nkg = kPfConsumers / nrg;           // warps sharing a row group's keys
  const int nact = nrg * nkg;                   // consumer warps at work
  const uint32_t ring = (smem_u32(dyn_smem) + 1023u) & ~1023u;

  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    for (int i = 0; i < kPfStages; ++i) {
      mbar_init(smem_u32(&sm.full[i]), 1);
      mbar_init(smem_u32(&sm.empty[i]), nrg);   // each box has nrg consumers
    }
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  griddep_wait();

  const int cap = min(a.max_pages * a.ps, a.max_kv_len);
  int L = a.seq_lens[b];
  if (L > cap || L < 0) {
    if (threadIdx.x == 0) record_error(a.error_flag, 2);
    L = L < 0 ? 0 : cap;
  }
  // keys this tile needs: up to the position of its last query token
  const int i_last = min(a.q_len - 1, (r0 + kPfRows - 1) / a.G);
  const int kend = max(0, L - a.q_len + i_last + 1);
  const int nboxes = (kend + kBoxTokens - 1) / kBoxTokens;
  const int32_t* bt = a.block_table + (size_t)b * a.max_pages;
  const int npages = kend > 0 ? (kend - 1) / a.ps + 1 : 0;
  for (int i = threadIdx.x; i < min(npages, kPageCache); i += kPfThreads) {
    int pg = __ldg(bt + i);
    if (pg < 0 || pg >= a.num_pages) {
      record_error(a.error_flag, 4);
      pg = 0;
    }
    sm.pages[i] = pg;
  }
  __syncthreads();
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == kPfConsumers) {
    // ================================================= producer (one lane)
    if (lane == 0) {
      int issued = 0;
      for (int j = 0; j < nboxes; ++j) {
        const int st = j % kPfStages;
        if (j >= kPfStages &&
            !wait_or_abort(smem_u32(&sm.empty[st]), ((j / kPfStages) - 1) & 1, abort_flag)) {
          *abort_flag = 1;
          break;
        }
        const int tok = j * kBoxTokens, pidx = tok / a.ps;
        int page;
        if (pidx < kPageCache) {
          page = sm.pages[pidx];
        } else {
          page = __ldg(bt + pidx);
          if (page < 0 || page >= a.num_pages) {
            record_error(a.error_flag, 4);
            page = 0;
          }
        }
        const long row = ((long)page * a.Hkv + h) * a.ps + (tok % a.ps);
        const uint32_t full = smem_u32(&sm.full[st]);
        const uint32_t sbase = ring + st * Gm::kStage;
        mbar_arrive_expect_tx(full, 2 * (Gm::kBoxK + Gm::kBoxS));
        tma_load_2d(sbase, &tmK, 0, (int)row, full);
        tma_load_2d(sbase + Gm::kBoxK, &tmV, 0, (int)row, full);
        if constexpr (FMT == kFmtNvfp4) {
          bulk_load(sbase + 2 * Gm::kBoxK, a.k_bscale + row * Gm::kSRow, Gm::kBoxS, full);
          bulk_load(sbase + 2 * Gm::kBoxK + Gm::kBoxS, a.v_bscale + row * Gm::kSRow,
                    Gm::kBoxS, full);
        }
        ++issued;
      }
      // no copy in flight at exit (bounded waits)
      for (int k = max(0, issued - kPfStages); k < issued; ++k)
        mbar_wait(smem_u32(&sm.full[k % kPfStages]), (k / kPfStages) & 1);
    }
    return;
  }
  if (warp >= nact) return;   // no query rows for this warp

  // ====================================================== consumer warps
  // score and output factors of this kv head (per-kv-head scales if given)
  const float qk_scale_log2 =
      a.k_hs ? (a.sm_scale * __ldg(a.k_hs + h)) * 1.4426950408889634f : a.qk_scale_log2;
  const float out_mult = a.v_hs ? __ldg(a.v_hs + h) : a.out_mult;
  const int rg = warp % nrg, kgi = warp / nrg;   // row group, key group
  // rows of this lane: g and g + 8 of the group's 16
  int qi[2], qh[2], pos[2];
  bool rv[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int row = r0 + 16 * rg + g + 8 * e;
    rv[e] = row < R;
    qi[e] = rv[e] ? row / a.G : 0;      // query token
    qh[e] = rv[e] ? row % a.G : 0;      // head within the kv head's group
    pos[e] = L - a.q_len + qi[e];       // its position (keys 0..pos)
    if (!rv[e]) pos[e] = -1;
  }
  // Q as the A operand: a0/a2 = row g, a1/a3 = row g + 8; head dims of
  // k-step j: (D/4) t + 4j + {0,1} (a0, a1) and + {2,3} (a2, a3).  Each row
  // is prescaled by its power of two; qsc[e] is its score scale.
  uint32_t qa[KS][4];
  float qsc[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const uint16_t* qp = static_cast<const uint16_t*>(a.q) +
                         (((size_t)b * a.q_len + qi[e]) * a.Hq + (size_t)h * a.G + qh[e]) * D +
                         (D / 4) * t;
    uint2 raw[KS];
    uint32_t mx2 = 0;
#pragma unroll
    for (int j = 0; j < KS; ++j) {
      raw[j] = rv[e] ? *reinterpret_cast<const uint2*>(qp + 4 * j) : make_uint2(0, 0);
      mx2 = __vmaxu2(mx2, __vmaxu2(raw[j].x & 0x7FFF7FFFu, raw[j].y & 0x7FFF7FFFu));
    }
    uint32_t mx = max(mx2 & 0xFFFFu, mx2 >> 16);
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const int ex = q_prescale_exp(mx);
    const float f = exp2i(ex);
#pragma unroll
    for (int j = 0; j < KS; ++j) {
      qa[j][e] = pack_f16x2(__uint_as_float(raw[j].x << 16) * f,
                            __uint_as_float(raw[j].x & 0xFFFF0000u) * f);
      qa[j][e + 2] = pack_f16x2(__uint_as_float(raw[j].y << 16) * f,
                                __uint_as_float(raw[j].y & 0xFFFF0000u) * f);
    }
    qsc[e] = scale_pow2(qk_scale_log2, -ex);
  }

  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  bool aborted = false;

  for (int j = kgi; j < nboxes; j += nkg) {
    const int st = j % kPfStages;
    bool got = true;
    if (lane == 0) got = wait_or_abort(smem_u32(&sm.full[st]), (j / kPfStages) & 1, abort_flag);
    if (!__all_sync(0xffffffffu, got)) {
      aborted = true;
      break;
    }
    __syncwarp();
    const uint32_t sbase = ring + st * Gm::kStage;
    const uint32_t boxK = sbase, boxV = sbase + Gm::kBoxK;
    const uint32_t boxKs = sbase + 2 * Gm::kBoxK, boxVs = boxKs + Gm::kBoxS;
    const int k0 = j * kBoxTokens;
    const int nvalid = min(kBoxTokens, kend - k0);

    // S = Q K^T: n-tile u covers keys k0 + 8u + {2t, 2t+1} in this lane;
    // x[u][0..1] row g, x[u][2..3] row g + 8
    float x[2][4];
    {
      uint32_t kg[KS][2], kg8[KS][2];
      k_frag<FMT, D>(boxK, boxKs, g, t, kg);
      k_frag<FMT, D>(boxK, boxKs, g + 8, t, kg8);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < KS; kk += 2) {
          const uint32_t(&kb)[KS][2] = u ? kg8 : kg;
          mma_f16(s0, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], kb[kk][0], kb[kk][1]);
          mma_f16(s1, qa[kk + 1][0], qa[kk + 1][1], qa[kk + 1][2], qa[kk + 1][3],
                  kb[kk + 1][0], kb[kk + 1][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = k0 + 8 * u + 2 * t + (e & 1);
          const int r = e >> 1;
          const float v = (s0[e] + s1[e]) * qsc[r];
          x[u][e] = key <= pos[r] ? v : -INFINITY;   // causal (and past the end)
        }
      }
    }
    // online softmax of rows g (r = 0) and g + 8 (r = 1), lazy reference max
    bool need = false;
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e) need |= x[u][e] > m[e >> 1] + kLazyMax;
    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float mx = fmaxf(fmaxf(x[0][2 * r], x[0][2 * r + 1]), fmaxf(x[1][2 * r], x[1][2 * r + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const bool mv = mx > m[r] + kLazyMax;
        const float alpha = mv ? ex2(m[r] - mx) : 1.f;
        m[r] = mv ? mx : m[r];
        l[r] *= alpha;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          o[n][2 * r] *= alpha;
          o[n][2 * r + 1] *= alpha;
        }
      }
    }
    float p[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float mr = m[e >> 1] == -INFINITY ? 0.f : m[e >> 1];
        p[u][e] = ex2(x[u][e] - mr);
        l[e >> 1] += p[u][e];
      }
    // P as the A operand (f16 high part + residual): a0 = row g, keys 2t..;
    // a1 = row g + 8; a2/a3 = the same rows, keys 8 + 2t..
    uint32_t ph[4], pl[4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const uint32_t hi = pack_f16x2(p[u][2 * r], p[u][2 * r + 1]);
        const float2 hf = unpack_f16x2(hi);
        ph[2 * u + r] = hi;
        pl[2 * u + r] = pack_f16x2(p[u][2 * r] - hf.x, p[u][2 * r + 1] - hf.y);
      }
    // O += P V: n-tile (i, c) holds value dim (D/8) g' + 2i + c in column g'
    uint32_t va[MT][4];
    v_frag<FMT, D>(boxV, boxVs, t, g, nvalid, va);
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      mma_f16(o[2 * i], ph[0], ph[1], ph[2], ph[3], va[i][0], va[i][2]);
      mma_f16(o[2 * i], pl[0], pl[1], pl[2], pl[3], va[i][0], va[i][2]);
      mma_f16(o[2 * i + 1], ph[0], ph[1], ph[2], ph[3], va[i][1], va[i][3]);
      mma_f16(o[2 * i + 1], pl[0], pl[1], pl[2], pl[3], va[i][1], va[i][3]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sm.empty[st]));   // this warp is done with the stage
  }
  if (aborted) {
    *abort_flag = 1;
    record_error(a.error_flag, 1);
  }

  // key groups 1.. of a row group hand their states (O fragments, m, lane
  // sums l) to key group 0 through shared memory, which rescales to the
  // common max and adds them
  if (nkg > 1) {
    float4* xo = reinterpret_cast<float4*>(dyn_smem + (ring - smem_u32(dyn_smem)) +
                                           kPfStages * Gm::kStage);
    const int slot_f4 = NT * 32 + 32;   // O fragments, then (m0, m1, l0, l1) per lane
    if (kgi > 0) {
      float4* my = xo + ((kgi - 1) * nrg + rg) * slot_f4;
#pragma unroll
      for (int n = 0; n < NT; ++n) my[n * 32 + lane] = make_float4(o[n][0], o[n][1], o[n][2], o[n][3]);
      my[NT * 32 + lane] = make_float4(m[0], m[1], l[0], l[1]);
    }
    asm volatile("bar.sync 1, %0;" ::"r"(nact * 32) : "memory");
    if (kgi > 0) return;
#pragma unroll 1
    for (int k = 1; k < nkg; ++k) {
      const float4* ot = xo + ((k - 1) * nrg + rg) * slot_f4;
      const float4 ml = ot[NT * 32 + lane];
      const float mo[2] = {ml.x, ml.y}, lo[2] = {ml.z, ml.w};
      float fa[2], fb[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float M = fmaxf(m[r], mo[r]);
        fa[r] = M == -INFINITY ? 0.f : ex2(m[r] - M);
        fb[r] = M == -INFINITY ? 0.f : ex2(mo[r] - M);
        l[r] = l[r] * fa[r] + lo[r] * fb[r];
        m[r] = M;
      }
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const float4 v = ot[n * 32 + lane];
        o[n][0] = o[n][0] * fa[0] + v.x * fb[0];
        o[n][1] = o[n][1] * fa[0] + v.y * fb[0];
        o[n][2] = o[n][2] * fa[1] + v.z * fb[1];
        o[n][3] = o[n][3] * fa[1] + v.w * fb[1];
      }
    }
  }

  // normalize and store: accumulator (row g or g + 8, columns 2t, 2t+1) of
  // n-tile (i, c) is value dim (D/8)(2t + q) + 2i + c for column 2t + q
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float v = l[r];
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    l[r] = v;
  }
  const float fac[2] = {l[0] > 0.f ? out_mult / l[0] : 0.f, l[1] > 0.f ? out_mult / l[1] : 0.f};
  const bool bad = aborted || *abort_flag != 0;   // any warp of the CTA gave up
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (!rv[r]) continue;
    const size_t orow = (((size_t)b * a.q_len + qi[r]) * a.Hq + (size_t)h * a.G + qh[r]) * D;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const int i = n >> 1, c = n & 1;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int dim = (D / 8) * (2 * t + q) + 2 * i + c;
        const float val = bad ? NAN : o[n][2 * r + q] * fac[r];
        if (a.out_dtype == 0) store_out_t<0>(a.out, a.out_scale, orow + dim, val);
        else if (a.out_dtype == 1) store_out_t<1>(a.out, a.out_scale, orow + dim, val);
        else store_out_t<2>(a.out, a.out_scale, orow + dim, val);
      }
    }
  }
}

template <int FMT, int D>
cudaError_t launch_prefill_t(const TensorMaps& m, const PartialArgs& a, cudaStream_t st) {
  // ring, plus the state exchange of the key groups (up to three O
  // fragment sets of 16 rows with their max and sums)
  const size_t xbytes = (size_t)(kPfConsumers - 1) * ((D / 8) * 32 + 32) * 16;
  const size_t smem = 1024 + (size_t)kPfStages * Geom<FMT, D>::kStage + xbytes;
  auto kern = prefill_kernel<FMT, D>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int tiles = (a.q_len * a.G + kPfRows - 1) / kPfRows;
  return launch_pdl(kern, dim3(tiles, a.batch * a.Hkv), dim3(kPfThreads), smem, st, m.k16, m.v16,
                    a);
}

}  // namespace

cudaError_t launch_prefill(int fmt, int D, const TensorMaps& m, const PartialArgs& a,
                           cudaStream_t st) {
  if (fmt == kFmtFp8 && D == 128) return launch_prefill_t<kFmtFp8, 128>(m, a, st);
  if (fmt == kFmtFp8 && D == 64) return launch_prefill_t<kFmtFp8, 64>(m, a, st);
  if (fmt == kFmtNvfp4 && D == 128) return launch_prefill_t<kFmtNvfp4, 128>(m, a, st);
  if (fmt == kFmtNvfp4 && D == 64) return launch_prefill_t<kFmtNvfp4, 64>(m, a, st);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
