// MLA absorbed decode over an NVFP4 latent cache (sm_103a).
//
// Model-Optimizer PR 714 (Testing: module printout) quantizes the MLA latent
// cache kv_c (512 wide, after kv_a_layernorm) with an NVFP4 quantizer
// (kv_c_bmm_quantizer) and leaves the query unquantized (q_bmm_quantizer
// disabled); a tensor-parallel rank holds 16 query heads (q_b_proj 3072 =
// 16 x 192).  Absorbed decode attends all 16 heads to one latent "kv head":
//   S_i = sm_scale (q_lat . kv^_c,i + q_pe . k_pe,i),  V_i = kv^_c,i
// with kv^_c the dequantized latent (e2m1 * block scale * global scale) and
// k_pe the bf16 rope key (64 wide).  The split-KV scheme is the same as the
// GQA kernel's (Model-Optimizer PR 1832 notes).
//
// GB300 design: four warps per CTA each own a 128-dim slice of the latent
// (and one 16-dim slice of the rope key).  Per 16-token box:
//  * each warp streams its own slice with TMA (3-D tensor maps: a 16 x 64 B
//    code box and a 16 x 32 B rope box) plus the box's block-scale rows by a
//    1-D bulk copy, through a private 4-deep mbarrier ring;
//  * each warp computes a partial S^T = K Q^T over its slice on mma.sync
//    (f16 latent fragments decoded from E2M1 * E4M3 exactly, bf16 rope
//    fragments as stored); the four partials are summed through a small
//    double-buffered shared-memory exchange (one CTA barrier per box);
//  * every warp then runs the same softmax update (bitwise identical) and
//    accumulates O^T = V^T P^T for its own 128 value dims, so the output
//    needs no cross-warp merge.  P enters the MMA as f16 (N(0,1)-scale
//    values keep its rounding far inside the tolerance; see the design notes).

#include "kvq_attn.cuh"

namespace kvq {
namespace {

constexpr int kMlaLat = 512;
constexpr int kMlaRope = 64;
constexpr int kMlaHeads = 16;
constexpr int kMlaQkDim = kMlaLat + kMlaRope;
constexpr int kSliceDims = kMlaLat / kDecodeWarps;   // 128 latent dims per warp
constexpr int kScaleRow = kMlaLat / 16;              // 32 block-scale bytes per token
constexpr int kMlaStages = 4;
// per-warp stage: [codes 16 x 64 B][scale rows 16 x 32 B][rope 16 x 32 B]
constexpr int kMlaCodeOff = 0, kMlaScaleOff = 1024, kMlaRopeOff = 1536, kMlaStage = 2048;
constexpr int kMlaRing = kDecodeWarps * kMlaStages * kMlaStage;   // 32 KB
// partial-score exchange: [2 box parities][4 warps][8 fragment regs][32 lanes]
constexpr int kMlaSxFloats = 2 * kDecodeWarps * 8 * 32;
constexpr int kMlaSmem = 1024 + kMlaRing + kMlaSxFloats * 4 + kMaxGroup * (kMaxFusedSplits + 1) * 4;

struct MlaSmem {
  uint64_t full[kDecodeWarps][kMlaStages];
  int abort_flag;
  int pages[kPageCache];
  float lse[kMlaHeads];
};

// Column swizzle of the output buffer [head][512]: XOR-ing the low four bits
// of d with (lane group / 2, head pair) makes the fragment stores and the
// row-wise reads conflict-free.
__device__ __forceinline__ int mla_swz(int head, int d) {
  return d ^ (((d >> 5) & 3) | (((head >> 1) & 3) << 2));
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__global__ void __launch_bounds__(kDecodeThreads, 2)
    mla_partial_kernel(const __grid_constant__ CUtensorMap tmKv,
                       const __grid_constant__ CUtensorMap tmPe, const PartialArgs a) {
  using Gs = Geom<kFmtNvfp4, kSliceDims>;   // a warp's slice looks like an NVFP4 D=128 row
  constexpr int KS = kSliceDims / 16;       // 8 latent k-steps per warp
  constexpr int MT = kSliceDims / 16;       // 8 value m-tiles per warp

  extern __shared__ uint8_t dyn_smem[];
  __shared__ MlaSmem sm;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int b = blockIdx.x;
  const int split = blockIdx.y;

  const uint32_t ring = (smem_u32(dyn_smem) + 1023u) & ~1023u;
  float* sx = reinterpret_cast<float*>(dyn_smem + (ring - smem_u32(dyn_smem)) + kMlaRing);
  float* wbuf = sx + kMlaSxFloats;

  const int cap = min(a.max_pages * a.ps, a.max_kv_len);
  // only barrier setup before the grid-dependency wait
  if (threadIdx.x == 0) sm.abort_flag = 0;
  if (lane == 0) {
    for (int i = 0; i < kMlaStages; ++i) mbar_init(smem_u32(&sm.full[warp][i]), 1);
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tmap(&tmKv);
    prefetch_tmap(&tmPe);
  }
  // overlap mode (a.fresh > 0): only the loads of boxes that hold the last
  // a.fresh positions wait for the preceding append
  if (a.fresh == 0) griddep_wait();

  int L = a.seq_lens[b];
  if (L > cap || L < 0) {
    if (threadIdx.x == 0) record_error(a.error_flag, 2);
    L = L < 0 ? 0 : cap;
  }
  long c = ((long)L + a.num_splits - 1) / a.num_splits;
  c = (c + 15) / 16 * 16;
  const int cstart = (int)min((long)split * c, (long)L);
  const int cend = (int)min((long)cstart + c, (long)L);
  const int nboxes = (cend - cstart + kBoxTokens - 1) / kBoxTokens;   // all warps, all boxes
  const int fresh_box = a.fresh == 0 ? 0 : (max(L - a.fresh, cstart) - cstart) / kBoxTokens;
  bool dep_done = a.fresh == 0;

  const int32_t* bt = a.block_table + (size_t)b * a.max_pages;
  const int p0 = cstart / a.ps;
  const int npages = cend > cstart ? (cend - 1) / a.ps - p0 + 1 : 0;
  for (int i = threadIdx.x; i < min(npages, kPageCache); i += kDecodeThreads) {
    int pg = __ldg(bt + p0 + i);
    if (pg < 0 || pg >= a.num_pages) {
      record_error(a.error_flag, 4);
      pg = 0;
    }
    sm.pages[i] = pg;
  }
  __syncthreads();
  volatile int* abort_flag = &sm.abort_flag;

  // this warp's slice of box j: codes, all block-scale rows, rope slice
  auto issue = [&](int j) {
    const int tok = cstart + j * kBoxTokens;
    const int pidx = tok / a.ps;
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
    const long row = (long)page * a.ps + (tok % a.ps);
    if (!dep_done && j >= fresh_box) {
      griddep_wait();
      dep_done = true;
    }
    const int st = j % kMlaStages;
    const uint32_t full = smem_u32(&sm.full[warp][st]);
    const uint32_t sbase = ring + (warp * kMlaStages + st) * kMlaStage;
    mbar_arrive_expect_tx(full, 16 * 64 + 16 * kScaleRow + 16 * 32);
    tma_load_3d(sbase + kMlaCodeOff, &tmKv, 0, warp, (int)row, full);
    bulk_load(sbase + kMlaScaleOff, a.k_bscale + row * kScaleRow, 16 * kScaleRow, full);
    tma_load_3d(sbase + kMlaRopeOff, &tmPe, 0, warp, (int)row, full);
  };
  int issued = 0;
  if (lane == 0)
    for (; issued < min(nboxes, kMlaStages); ++issued) issue(issued);

  // Q^T fragments: latent dims 128 w + 32 t + 4 j + {0..3} (permuted like
  // the K fragments) and rope dims 512 + 16 w + 4 t + {0..3} (bf16 as is)
  uint32_t qb[KS][2][2], qr[2][2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const uint16_t* qh = a.q + ((size_t)b * kMlaHeads + g + 8 * hh) * kMlaQkDim;
    const uint16_t* qp = qh + kSliceDims * warp + 32 * t;
#pragma unroll
    for (int j = 0; j < KS; ++j) {
      const uint2 v = *reinterpret_cast<const uint2*>(qp + 4 * j);
      qb[j][hh][0] = pack_f16x2(bf16_bits_to_f32(v.x & 0xFFFFu), bf16_bits_to_f32(v.x >> 16));
      qb[j][hh][1] = pack_f16x2(bf16_bits_to_f32(v.y & 0xFFFFu), bf16_bits_to_f32(v.y >> 16));
    }
    const uint2 r = *reinterpret_cast<const uint2*>(qh + kMlaLat + 16 * warp + 4 * t);
    qr[hh][0] = r.x;
    qr[hh][1] = r.y;
  }

  float o[MT][2][4];
#pragma unroll
  for (int i = 0; i < MT; ++i)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) o[i][hh][0] = o[i][hh][1] = o[i][hh][2] = o[i][hh][3] = 0.f;
  float m[2][2], l[2][2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) m[hh][0] = m[hh][1] = -INFINITY, l[hh][0] = l[hh][1] = 0.f;
  bool aborted = false;

  for (int j = 0; j < nboxes; ++j) {
    const int st = j % kMlaStages;
    // Every warp takes part in the per-box barrier, so a failed wait does
    // not leave the loop: the warp skips its work and keeps step.
    if (!aborted) {
      bool got = true;
      if (lane == 0)
        got = wait_or_abort(smem_u32(&sm.full[warp][st]), (j / kMlaStages) & 1, abort_flag);
      aborted = !__all_sync(0xffffffffu, got);
      __syncwarp();
    }
    const int tbase = cstart + j * kBoxTokens;
    const int nvalid = min(kBoxTokens, cend - tbase);
    const uint32_t sbase = ring + (warp * kMlaStages + st) * kMlaStage;
    const uint32_t boxK = sbase + kMlaCodeOff;
    const uint32_t boxS = sbase + kMlaScaleOff + 8 * warp;   // this slice's 8 blocks of a row
    float* sxp = sx + (j & 1) * (kDecodeWarps * 8 * 32);

    if (!aborted) {
      // ---- partial scores of this warp's slice (log2 domain, scaled)
      uint32_t kg[KS][2], kg8[KS][2];
      k_frag<kFmtNvfp4, kSliceDims, kScaleRow>(boxK, boxS, g, t, kg);
      k_frag<kFmtNvfp4, kSliceDims, kScaleRow>(boxK, boxS, g + 8, t, kg8);
      const uint2 rg = lds64(sbase + kMlaRopeOff + g * 32 + 8 * t);
      const uint2 rg8 = lds64(sbase + kMlaRopeOff + (g + 8) * 32 + 8 * t);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        float sp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < KS; kk += 2) {
          mma_f16(s0, kg[kk][0], kg8[kk][0], kg[kk][1], kg8[kk][1], qb[kk][hh][0], qb[kk][hh][1]);
          mma_f16(s1, kg[kk + 1][0], kg8[kk + 1][0], kg[kk + 1][1], kg8[kk + 1][1],
                  qb[kk + 1][hh][0], qb[kk + 1][hh][1]);
        }
        mma_bf16(sp, rg.x, rg8.x, rg.y, rg8.y, qr[hh][0], qr[hh][1]);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          sxp[(warp * 8 + 4 * hh + e) * 32 + lane] =
              (s0[e] + s1[e]) * a.qk_scale_log2 + sp[e] * a.pe_scale_log2;
      }
    }
    __syncthreads();   // the four slice partials of this box are in shared memory
    if (!aborted) {
      float x[2][4];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < kDecodeWarps; ++w) v += sxp[(w * 8 + 4 * hh + e) * 32 + lane];
          x[hh][e] = (g + 8 * (e >> 1) < nvalid) ? v : -INFINITY;
        }
      // ---- softmax update with a lazily moving reference max (identical in
      // every warp: same inputs, same operations)
      bool need = false;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 4; ++e) need |= x[hh][e] > m[hh][e & 1] + 8.0f;
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float mx = fmaxf(x[hh][e], x[hh][e + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const bool mv = mx > m[hh][e] + 8.0f;
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
      uint32_t pb[2][2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float b0 = m[hh][0] == -INFINITY ? 0.f : m[hh][0];
        const float b1 = m[hh][1] == -INFINITY ? 0.f : m[hh][1];
        const float p0 = ex2(x[hh][0] - b0), p1 = ex2(x[hh][1] - b1);
        const float p2 = ex2(x[hh][2] - b0), p3 = ex2(x[hh][3] - b1);
        l[hh][0] += p0 + p2;
        l[hh][1] += p1 + p3;
        pb[hh][0] = movmatrix_trans(pack_f16x2(p0, p1));
        pb[hh][1] = movmatrix_trans(pack_f16x2(p2, p3));
      }
      // ---- O^T += V^T P^T over this warp's 128 value dims (V = the latent)
      uint32_t va[MT][4];
      v_frag<kFmtNvfp4, kSliceDims, kScaleRow>(boxK, boxS, t, g, nvalid, va);
#pragma unroll
      for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          mma_f16(o[i][hh], va[i][0], va[i][1], va[i][2], va[i][3], pb[hh][0], pb[hh][1]);
      __syncwarp();
      if (lane == 0 && issued < nboxes) {
        fence_proxy_async_shared();
        issue(issued++);
      }
    }
  }
  if (aborted) {
    *abort_flag = 1;
    record_error(a.error_flag, 1);
  }
  if (lane == 0) {
    const int done = aborted ? 0 : nboxes;
    for (int k = max(done, issued - kMlaStages); k < issued; ++k)
      mbar_wait(smem_u32(&sm.full[warp][k % kMlaStages]), (k / kMlaStages) & 1);
  }
  __syncwarp();
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = l[hh][e];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      l[hh][e] = v;
    }
  __syncthreads();
  if (!dep_done && threadIdx.x == 0) griddep_wait();   // the grid ends after the append
  const bool bad = *abort_flag != 0;
  // normalized O of this warp's dims -> shared memory obuf[head][512] (the ring
  // is drained), then coalesced stores of the partials
  float* obuf = reinterpret_cast<float*>(dyn_smem + (ring - smem_u32(dyn_smem)));
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int head = 2 * t + (e & 1) + 8 * hh;
      const float li = l[hh][e & 1];
      const float f = (li > 0.f) ? a.out_mult / li : 0.f;
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        const int d = kSliceDims * warp + 16 * g + 2 * i + (e >> 1);
        obuf[head * kMlaLat + mla_swz(head, d)] = bad ? NAN : o[i][hh][e] * f;
      }
    }
  if (warp == 0 && g == 0) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float mm = m[hh][e], li = l[hh][e];
        sm.lse[2 * t + e + 8 * hh] = bad ? NAN : (mm == -INFINITY || li == 0.f) ? -INFINITY
                                                                               : (mm + log2f(li)) * kLn2;
      }
  }
  __syncthreads();
  const size_t part_row = (size_t)b * kMlaHeads;
  for (int i = threadIdx.x; i < kMlaHeads * kMlaLat; i += kDecodeThreads) {
    const int head = i / kMlaLat, d = i % kMlaLat;
    a.part_o[((part_row + head) * a.num_splits + split) * kMlaLat + d] =
        obuf[head * kMlaLat + mla_swz(head, d)];
  }
  if (threadIdx.x < kMlaHeads)
    a.part_lse[(part_row + threadIdx.x) * a.num_splits + split] = sm.lse[threadIdx.x];
  if (a.counters) fused_combine(a, b, part_row, wbuf);
}

}  // namespace

cudaError_t launch_mla_partial(const CUtensorMap& tkv, const CUtensorMap& tpe,
                               const PartialArgs& a, cudaStream_t st) {
  static_assert(kMlaHeads * kMlaLat * 4 <= kMlaRing, "the output buffer must fit in the ring");
  cudaError_t e = cudaFuncSetAttribute(mla_partial_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kMlaSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(mla_partial_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  return launch_pdl(mla_partial_kernel, dim3(a.batch, a.num_splits), dim3(kDecodeThreads),
                    (size_t)kMlaSmem, st, tkv, tpe, a);
}

}  // namespace kvq
