// MLA absorbed decode over an NVFP4 latent cache on the 5th-generation tensor
// cores (sm_103a: tcgen05 MMAs with accumulators in tensor memory).
//
// Model-Optimizer PR 714 (Testing: module printout) quantizes the MLA latent
// cache kv_c (512 wide, after kv_a_layernorm) with an NVFP4 quantizer
// (kv_c_bmm_quantizer) and leaves the query unquantized (q_bmm_quantizer
// disabled); a tensor-parallel rank holds 16 query heads (q_b_proj 3072 =
// 16 x 192).  Absorbed decode attends all 16 heads to one latent "kv head":
//   S_i = sm_scale (q_lat . kv^_c,i + q_pe . k_pe,i),  V_i = kv^_c,i
// with kv^_c the dequantized latent (e2m1 * block scale * global scale) and
// k_pe the bf16 rope key (64 wide).  The split-KV scheme is the GQA kernel's
// (Model-Optimizer PR 1832 notes).
//
// GB300 design.  One CTA per SM runs one chunk in tiles of 128 tokens with
// warp-specialized roles that hand work over through mbarriers:
//  * TMA copies bring a tile's latent codes (128-byte swizzled boxes) and
//    block scales (1-D bulk copies) into a raw buffer, and its rope keys
//    straight into one of two bf16 operand tiles (the same swizzled layout);
//    the O^T issuing thread issues those of the first tile (it is idle
//    until the first P^T), lane 0 of the last decode warp those of every
//    later tile once the previous tile has been decoded;
//  * six decode warps turn the tile, once, into an f16 [token][dim] tile
//    (E2M1 x E4M3 -> f16 is exact) in the 128-byte-swizzled layout that is
//    the K-major A operand of S^T = K Q^T and, read MN-major, the A operand
//    of O^T = V^T P^T.  They decode it one 128-dim block at a time, each
//    block as soon as the O^T MMAs of the previous tile have finished
//    reading that block, so that decoding overlaps the tensor pipe;
//  * the MMAs are tcgen05.mma (kind::f16, M = 128 tokens or value dims,
//    N = 16 heads): S^T of the latent (f16) block by block as the blocks are
//    decoded and of the rope part (bf16) into two tensor-memory accumulators
//    (their scales differ), and O^T of four 128-dim blocks into a third,
//    each block committed on its own barrier.  One thread issues S^T,
//    another O^T;
//  * four softmax warps (one per tensor-memory lane quarter) read S^T (one
//    token per thread, all 16 heads), run the softmax with a lazily moving
//    reference max, rescale O in tensor memory when it moves and write P^T
//    (f16) as the B operand of the O^T MMA.
// A 128-token tile fills the M = 128 rows of every S^T MMA (a 64-token tile
// left half of them empty): 68 MMAs per 128 tokens instead of 104.  The
// f16 tile is single buffered; rope tiles, S^T accumulators and P^T are
// double buffered.  The softmax and decode loops start with a dry pass of
// their code (nothing waited for, nothing handed over, the state unchanged)
// while tile 0 is loaded: after an L2 flush their first real pass would
// otherwise fetch the unrolled instructions from DRAM on the critical path.
// With 2..8 splits the CTAs of a request form a cluster and merge their
// partials through distributed shared memory.  Every wait is bounded; a
// timeout sets an error bit and the partials become NaN.

#include <atomic>

#include "kvq_attn.cuh"

namespace kvq {
namespace {

constexpr int kMlaLat = 512;
constexpr int kMlaRope = 64;
constexpr int kMlaHeads = 16;
constexpr int kMlaQkDim = kMlaLat + kMlaRope;
constexpr int kT = 128;             // tokens per tile
constexpr int kBoxes = kT / kBoxTokens;
constexpr int kSoftWarps = 4;       // warps 0-3: softmax, one per lane quarter
constexpr int kDecWarps = 6;        // warps 4-9: decode
constexpr int kDecoders = 32 * kDecWarps;
constexpr int kWorkers = 32 * kSoftWarps + kDecoders;
constexpr int kSWarp = kWorkers / 32, kOWarp = kSWarp + 1;   // S^T issue, O^T issue
constexpr int kThreads = kWorkers + 64;
constexpr int kBlocks = kMlaLat / 128;   // 128-dim blocks (two 64-dim atom columns)
constexpr int kTmemCols = 128;      // S lat [2] @0,16 | S rope [2] @32,48 | O^T 4 x 16 @64
constexpr int kColSLat = 0, kColSPe = 32, kColO = 64;

// shared-memory map (bytes from the 1024-aligned base); every MMA operand
// tile starts on a 1024-byte boundary (the 128-byte swizzle period)
constexpr int kColBytes = kT * 128;                           // one 64-dim column, 16 KB
constexpr int kTileBytes = kT * kMlaLat * 2;                  // f16 latent tile, 128 KB
constexpr int kOffTile = 0;
constexpr int kHalfBytes = kT * 128;                          // codes of 256 dims, 16 KB
constexpr int kRawCodes = 2 * kHalfBytes;                     // [half][128 rows x 128 B]
constexpr int kRawScales = kT * (kMlaLat / 16);               // 4 KB block scales
constexpr int kOffRaw = kOffTile + kTileBytes;                // one raw tile
constexpr int kPeBytes = kT * kMlaRope * 2;                   // bf16 rope tile, 16 KB
constexpr int kOffPe = kOffRaw + kRawCodes + kRawScales;      // two rope operand tiles
constexpr int kOffQLat = kOffPe + 2 * kPeBytes;               // f16 [16][512], 16 KB
constexpr int kOffQPe = kOffQLat + kMlaHeads * kMlaLat * 2;   // bf16 [16][64], 2 KB
constexpr int kPBytes = kMlaHeads * kT * 2;                   // f16 P^T [16][128], 4 KB
constexpr int kOffP = kOffQPe + kMlaHeads * kMlaRope * 2;     // two P^T tiles
constexpr int kSmemUsed = kOffP + 2 * kPBytes;
constexpr int kSmemBytes = kSmemUsed + 1024;                  // alignment slack
static_assert(kOffRaw % 1024 == 0 && (kOffRaw + kRawCodes) % 1024 == 0 && kOffPe % 1024 == 0 &&
                  kOffQLat % 1024 == 0 && kOffQPe % 1024 == 0 && kOffP % 1024 == 0,
              "operand tiles on the swizzle period");
static_assert(kRawCodes + kRawScales >= kMaxGroup * (kMaxFusedSplits + 1) * 4,
              "combine weights fit in the raw buffer");

struct MlaSmem {
  uint64_t raw_full;               // codes and scales of a tile landed
  uint64_t pe_full[2];             // rope keys of a tile landed (per rope buffer)
  uint64_t dec_blk[kBlocks];       // decode warps: 128-dim block of the tile written
  uint64_t s_done[2];              // S^T MMAs of a tile completed
  uint64_t o_blk[kBlocks];         // O^T MMAs of a 128-dim block completed
  uint64_t p_ready[2];             // P^T written and O rescaled: O^T MMAs may go
  uint64_t comb_full;              // fused combine: partials landed
  uint32_t tmem;                   // tensor-memory base address
  int abort_flag;
  int need[kSoftWarps];            // softmax warps: the reference max must move
  float wmax[kSoftWarps][kMlaHeads];   // per-warp tile maxima
  float lsum[kSoftWarps][kMlaHeads];   // per-warp denominators (end)
  float m[kMlaHeads];              // final reference max (end)
  float fac[kMlaHeads];            // partial's factor per head: value scale / denominator (end)
  uint32_t qmax[kMlaHeads];        // largest |q_lat| per head (bf16 magnitude bits)
  float qfac[kMlaHeads];           // latent score scale per head (log2 domain)
  int pages[kPageCache];
};
static_assert(kSmemBytes + sizeof(MlaSmem) <= 232448, "shared memory of one CTA");

// ----------------------------------------------------------------- tcgen05
// Shared-memory matrix descriptor: start, leading/stride byte offsets (16-byte
// units), descriptor version 1, 128-byte swizzle.  K-major operands: SBO =
// distance of 8-row groups; MN-major: LBO = distance of 64-element columns
// along M/N, SBO = distance of 8-row groups along K.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor, kind::f16: D f32, A/B f16 (0) or bf16 (1), A K-major
// (0) or MN-major (1), B K-major, N = 16, M = 128.
__host__ __device__ constexpr uint32_t idesc(uint32_t ab_fmt, uint32_t a_mn) {
  return (1u << 4) | (ab_fmt << 7) | (ab_fmt << 10) | (a_mn << 15) | ((16u >> 3) << 17) |
         ((128u >> 4) << 24);
}
constexpr uint32_t kIdF16 = idesc(0, 0), kIdBf16 = idesc(1, 0), kIdF16MnA = idesc(0, 1);

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                    bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"((uint32_t)acc)
      : "memory");
}
// arrives on `bar` once every MMA this thread issued before has completed
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 lanes x 16 columns of 32 bits: thread i of the warp gets lane (base + i)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// byte offset of 16-bit element (row r, col c < 64) in a 128-byte-swizzled
// column of 8-row atoms (atom stride 1 KB)
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((((c >> 3) ^ r) & 7) << 4) + (c & 7) * 2);
}

// Bounded wait by the calling thread; a timeout raises the CTA's abort flag.
__device__ __forceinline__ void wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (!mbar_wait(bar, parity)) *abort_flag = 1;
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_tc_kernel(const __grid_constant__ CUtensorMap tmCodes,
                  const __grid_constant__ CUtensorMap tmPe,
                  const __grid_constant__ CUtensorMap tmCodes64,
                  const __grid_constant__ CUtensorMap tmPe64, const PartialArgs a) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ MlaSmem sm;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x, split = blockIdx.y;
  const uint32_t base = (smem_u32(dyn_smem) + 1023u) & ~1023u;
  uint8_t* gbase = dyn_smem + (base - smem_u32(dyn_smem));
  volatile int* abort_flag = &sm.abort_flag;
  const int dt = tid - 32 * kSoftWarps;   // decode thread 0..kDecoders-1 (decode warps)
  const bool decoder = dt >= 0 && dt < kDecoders;

  // ---- setup that reads no input: barriers, tensor memory
  if (tid == 0) {
    mbar_init(smem_u32(&sm.raw_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.pe_full[i]), 1);
      mbar_init(smem_u32(&sm.s_done[i]), 1);
      mbar_init(smem_u32(&sm.p_ready[i]), 1);
    }
    for (int i = 0; i < kBlocks; ++i) {
      mbar_init(smem_u32(&sm.dec_blk[i]), kDecoders);
      mbar_init(smem_u32(&sm.o_blk[i]), 1);
    }
    mbar_init(smem_u32(&sm.comb_full), 1);
    sm.abort_flag = 0;
    for (int h = 0; h < kMlaHeads; ++h) sm.qmax[h] = 0u;
    fence_barrier_init();
    prefetch_tmap(&tmCodes);
    prefetch_tmap(&tmPe);
    prefetch_tmap(&tmCodes64);
    prefetch_tmap(&tmPe64);
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sm.tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // overlap mode (a.fresh > 0): only loads of tiles holding the last a.fresh
  // positions wait for the preceding append
  if (a.fresh == 0) griddep_wait();

  // Q (decode warps): every load first, before the block table, so that the
  // two DRAM trips after an L2 flush overlap
  constexpr int kQItems = kMlaHeads * (kMlaQkDim / 8);
  constexpr int kQPer = (kQItems + kDecoders - 1) / kDecoders;
  uint4 qv[kQPer];
  if (decoder) {
    const uint16_t* qg = static_cast<const uint16_t*>(a.q) + (size_t)b * kMlaHeads * kMlaQkDim;
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int i = dt + k * kDecoders;
      if (i < kQItems)
        qv[k] = *reinterpret_cast<const uint4*>(qg + (size_t)(i / (kMlaQkDim / 8)) * kMlaQkDim +
                                                (i % (kMlaQkDim / 8)) * 8);
    }
  }

  // one-page requests: the page index does not depend on the length, so its
  // load overlaps the length's
  const int32_t* bt = a.block_table + (size_t)b * a.max_pages;
  int pg_single = 0;
  if (a.max_pages == 1 && tid == 0) pg_single = __ldg(bt);

  // ---- chunk of this split
  int L = a.seq_lens[b];
  const int cap = min(a.max_pages * a.ps, a.max_kv_len);
  if (L > cap || L < 0) {
    if (tid == 0) record_error(a.error_flag, 2);
    L = L < 0 ? 0 : cap;
  }
  long c = ((long)L + a.num_splits - 1) / a.num_splits;
  c = (c + 15) / 16 * 16;
  const int cstart = (int)min((long)split * c, (long)L);
  const int cend = (int)min((long)cstart + c, (long)L);
  const int ntok = cend - cstart;
  const int nt = (ntok + kT - 1) / kT;
  const int fresh_tok = a.fresh == 0 ? 0x7fffffff : max(L - a.fresh, cstart) - cstart;
  bool dep_done = a.fresh == 0;   // issuer: has waited for the preceding kernel

  const int p0 = cstart / a.ps;
  const int npages = cend > cstart ? (cend - 1) / a.ps - p0 + 1 : 0;
  for (int i = tid; i < min(npages, kPageCache); i += kThreads) {
    int pg = a.max_pages == 1 ? pg_single : __ldg(bt + p0 + i);
    if (pg < 0 || pg >= a.num_pages) {
      record_error(a.error_flag, 4);
      pg = 0;
    }
    sm.pages[i] = pg;
  }

  tc_fence_before();
  __syncthreads();   // page cache and tensor-memory address ready
  tc_fence_after();
  const uint32_t tmem = sm.tmem;

  auto cache_row = [&](int tok) -> long {
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
    return (long)page * a.ps + (tok % a.ps);
  };

  // Descriptors are built once; per MMA only the start-address field moves
  // (16-byte units, no carry out of 14 bits: every shared address is below
  // 256 KB).
  const uint64_t dq = sdesc(base + kOffQLat, 16, 1024);
  const uint64_t dqpe = sdesc(base + kOffQPe, 16, 1024);
  const uint64_t dk = sdesc(base + kOffTile, 16, 1024);   // K-major tile

  // Copies of tile x (tile 0 by the O^T thread, later ones by lane 0 of the
  // last decode warp): codes and scales
  // into the raw buffer, rope keys into rope tile x % 2.  Each 64-token half
  // inside one page moves as four copies (64-row boxes), otherwise as four
  // per 16-token box.  Raw layout: codes [half][row][128 B] (128-byte
  // swizzle), scales [row][32 B]; rope tile [row][128 B] (128-byte swizzle).
  auto issue_raw = [&](int x) {
    if (!dep_done && x * kT + kT > fresh_tok) {
      griddep_wait();
      dep_done = true;
    }
    const int nb = min(kBoxes, (ntok - x * kT + kBoxTokens - 1) / kBoxTokens);
    const uint32_t st = base + kOffRaw;
    const uint32_t pe = base + kOffPe + (x & 1) * kPeBytes;
    const uint32_t bar = smem_u32(&sm.raw_full), pbar = smem_u32(&sm.pe_full[x & 1]);
    mbar_arrive_expect_tx(bar, nb * kBoxTokens * (kMlaLat / 2 + kMlaLat / 16));
    mbar_arrive_expect_tx(pbar, nb * kBoxTokens * kMlaRope * 2);
    for (int sub = 0; sub < 2; ++sub) {
      const int nbs = min(4, nb - 4 * sub);
      if (nbs <= 0) break;
      const int tok0 = cstart + x * kT + 64 * sub;
      const long row0 = cache_row(tok0);
      const uint32_t o = 8192 * sub;   // 64 rows of 128 bytes
      if (nbs == 4 && tok0 / a.ps == (tok0 + 63) / a.ps) {
        tma_load_3d(st + o, &tmCodes64, 0, 0, (int)row0, bar);
        tma_load_3d(st + kHalfBytes + o, &tmCodes64, 0, 1, (int)row0, bar);
        bulk_load(st + kRawCodes + 64 * sub * (kMlaLat / 16), a.k_bscale + row0 * (kMlaLat / 16),
                  64 * (kMlaLat / 16), bar);
        tma_load_2d(pe + o, &tmPe64, 0, (int)row0, pbar);
        continue;
      }
      for (int k = 0; k < nbs; ++k) {
        const long row = k == 0 ? row0 : cache_row(tok0 + k * kBoxTokens);
        tma_load_3d(st + o + k * 2048, &tmCodes, 0, 0, (int)row, bar);
        tma_load_3d(st + kHalfBytes + o + k * 2048, &tmCodes, 0, 1, (int)row, bar);
        bulk_load(st + kRawCodes + (64 * sub + k * kBoxTokens) * (kMlaLat / 16),
                  a.k_bscale + row * (kMlaLat / 16), kBoxTokens * (kMlaLat / 16), bar);
        tma_load_2d(pe + o + k * 2048, &tmPe, 0, (int)row, pbar);
      }
    }
  };

  if (warp == kSWarp) {
    // ============================================== S^T issue (one thread)
    if (lane == 0) {
      const uint64_t dpe0 = sdesc(base + kOffPe, 16, 1024);
      const uint64_t dpe1 = sdesc(base + kOffPe + kPeBytes, 16, 1024);
      int s_issued = 0;
      for (int x = 0; x < nt && !*abort_flag; ++x) {
        // S^T buffer x % 2 was read by the softmax of x - 2, which precedes
        // O^T x - 2 and so the decode of x - 1 and x
        const uint32_t dl = tmem + kColSLat + 16 * (x & 1), dp = tmem + kColSPe + 16 * (x & 1);
        for (int blk = 0; blk < kBlocks; ++blk) {
          wait_bar(smem_u32(&sm.dec_blk[blk]), x & 1, abort_flag);
          if (*abort_flag) break;
          tc_fence_after();
#pragma unroll
          for (int k8 = 0; k8 < 8; ++k8) {
            const int kk = 8 * blk + k8;   // 16-dim K-step: column kk / 4 of the tile
            mma(dl, dk + (uint64_t)(((kk >> 2) * kColBytes + (kk & 3) * 32) >> 4),
                dq + (uint64_t)(((kk >> 2) * 2048 + (kk & 3) * 32) >> 4), kIdF16, kk > 0);
          }
        }
        if (*abort_flag) break;
        wait_bar(smem_u32(&sm.pe_full[x & 1]), (x >> 1) & 1, abort_flag);
        if (*abort_flag) break;
        tc_fence_after();
        const uint64_t dpe = (x & 1) ? dpe1 : dpe0;
#pragma unroll
        for (int kk = 0; kk < kMlaRope / 16; ++kk)
          mma(dp, dpe + (uint64_t)(kk * 2), dqpe + (uint64_t)(kk * 2), kIdBf16, kk > 0);
        mma_commit(smem_u32(&sm.s_done[x & 1]));
        ++s_issued;
      }
      // every MMA of this thread has completed at exit (bounded waits)
      for (int x = max(0, s_issued - 2); x < s_issued; ++x)
        mbar_wait(smem_u32(&sm.s_done[x & 1]), (x >> 1) & 1);
      if (s_issued < nt) *abort_flag = 1;
    }
    __syncwarp();
  } else if (warp == kOWarp) {
    // ============================================== O^T issue (one thread)
    if (lane == 0) {
      // the copies of tile 0: this thread is idle until its first P^T, and
      // the decode warps convert Q meanwhile
      if (nt > 0) issue_raw(0);
      const uint64_t dv = sdesc(base + kOffTile, kColBytes, 1024);   // MN-major tile
      const uint64_t dpt0 = sdesc(base + kOffP, 16, 1024);
      const uint64_t dpt1 = sdesc(base + kOffP + kPBytes, 16, 1024);
      int o_issued = 0;
      for (int x = 0; x < nt; ++x) {
        // P^T x written and O rescaled (which implies S^T x done)
        wait_bar(smem_u32(&sm.p_ready[x & 1]), (x >> 1) & 1, abort_flag);
        if (*abort_flag) break;
        tc_fence_after();
        const uint64_t dpt = (x & 1) ? dpt1 : dpt0;
        for (int i = 0; i < kBlocks; ++i) {
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            mma(tmem + kColO + 16 * i,
                dv + (uint64_t)(((2 * i) * kColBytes + (2 * kk) * 1024) >> 4),
                dpt + (uint64_t)(((kk >> 2) * 2048 + (kk & 3) * 32) >> 4), kIdF16MnA,
                x > 0 || kk > 0);
          mma_commit(smem_u32(&sm.o_blk[i]));   // block i of the tile free for x + 1
        }
        ++o_issued;
      }
      bool ok = true;
      if (o_issued > 0)
        ok = mbar_wait(smem_u32(&sm.o_blk[kBlocks - 1]), (o_issued - 1) & 1);
      if (!ok || o_issued < nt) *abort_flag = 1;
    }
    __syncwarp();
  } else if (decoder) {
    // ============================================================ decode
    // lane 0 of the last decode warp issues the copies of tile y + 1 when
    // every decode thread is done with tile y (tile 0: the O^T thread)
    const bool tma_thread = warp == kWorkers / 32 - 1 && lane == 0;
    // The latent part of each head is scaled by its power of two 2^e
    // (q_prescale_exp of the head's largest |q_lat|) before the f16
    // conversion, so that the bf16 query keeps its full range; 2^-e goes
    // into the head's score scale.  The rope part stays bf16 (exact).
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int i = dt + k * kDecoders;
      if (i >= kQItems) break;
      const int h = i / (kMlaQkDim / 8), d = (i % (kMlaQkDim / 8)) * 8;
      if (d < kMlaLat) {
        const uint4 v = qv[k];
        const uint32_t m2 = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                     __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
        const uint32_t mx = max(m2 & 0xFFFFu, m2 >> 16);
        if (mx) atomicMax(&sm.qmax[h], mx);
      }
    }
    asm volatile("bar.sync 3, %0;" ::"n"(kDecoders) : "memory");   // decode warps only
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int i = dt + k * kDecoders;
      if (i >= kQItems) break;
      const int h = i / (kMlaQkDim / 8), d = (i % (kMlaQkDim / 8)) * 8;
      const uint4 v = qv[k];
      if (d < kMlaLat) {
        const float fs = exp2i(q_prescale_exp(sm.qmax[h]));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t f[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          f[j] = pack_f16x2(__uint_as_float(w[j] << 16) * fs,
                            __uint_as_float(w[j] & 0xFFFF0000u) * fs);
        sts128(base + kOffQLat + (d >> 6) * 2048 + swz(h, d & 63), f[0], f[1], f[2], f[3]);
      } else {
        sts128(base + kOffQPe + swz(h, d - kMlaLat), v.x, v.y, v.z, v.w);
      }
    }
    if (dt < kMlaHeads) sm.qfac[dt] = scale_pow2(a.qk_scale_log2, -q_prescale_exp(sm.qmax[dt]));
    fence_proxy_async_shared();   // Q: generic stores -> operand of the async MMAs
    // the softmax warps read the score scales after this barrier; the first
    // S^T MMAs read Q after the first block barrier
    asm volatile("bar.arrive 2, %0;" ::"n"(kDecoders + 32 * kSoftWarps) : "memory");

    // Decode of 128-dim block blk of tile x.  A unit is (token, 64-dim
    // column, half) = 32 dims; eight consecutive threads take the eight
    // tokens of an atom, so that the swizzled loads and stores spread over
    // all banks.  Rows past the chunk are zero (finite operands for the
    // masked tokens of the O^T MMA).
    auto decode_block = [&](int x, int blk) {
      const uint32_t st = base + kOffRaw;
      const int nvalid = x < 0 ? kT : min(kT, ntok - x * kT);
      // this thread's units u = dt + k kDecoders (up to kUnits): every load
      // first, then the conversions and stores, so the loads overlap
      constexpr int kUnits = (kT * 4 + kDecoders - 1) / kDecoders;
      uint4 v[kUnits];
      uint32_t sc[kUnits];
#pragma unroll
      for (int k = 0; k < kUnits; ++k) {
        const int u = dt + k * kDecoders;
        const int p = u & 7, rest = u >> 3;
        const int db = 2 * blk + ((rest >> 1) & 1), half = rest & 1;
        const int r = (rest >> 2) * 8 + p;
        v[k] = make_uint4(0u, 0u, 0u, 0u);
        sc[k] = 0u;
        if (u < kT * 4 && r < nvalid) {
          v[k] = lds128(st + (db >> 2) * kHalfBytes + r * 128 +
                        (((((db & 3) * 2 + half) ^ r) & 7) << 4));
          sc[k] = lds16(st + kRawCodes + r * (kMlaLat / 16) + db * 4 + half * 2);
        }
      }
#pragma unroll
      for (int k = 0; k < kUnits; ++k) {
        const int u = dt + k * kDecoders;
        if (u >= kT * 4) break;
        const int p = u & 7, rest = u >> 3;
        const int db = 2 * blk + ((rest >> 1) & 1), half = rest & 1;
        const int r = (rest >> 2) * 8 + p;
        // rows past the chunk: zero codes and scales decode to zeros
        const uint32_t s2 = e4m3x2_to_f16x2(sc[k]);
        const uint32_t s_lo = __byte_perm(s2, 0, 0x1010), s_hi = __byte_perm(s2, 0, 0x3232);
        const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
        uint32_t o[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t e0, e1, e2, e3;
          e2m1x8_to_f16x2x4(w[j], e0, e1, e2, e3);
          const uint32_t sj = j < 2 ? s_lo : s_hi;
          o[j][0] = hmul2(e0, sj);
          o[j][1] = hmul2(e1, sj);
          o[j][2] = hmul2(e2, sj);
          o[j][3] = hmul2(e3, sj);
        }
        const uint32_t row_base =
            base + kOffTile + db * kColBytes + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          sts128(row_base + ((((half * 4 + j) ^ r) & 7) << 4), o[j][0], o[j][1], o[j][2],
                 o[j][3]);
      }
      fence_proxy_async_shared();   // generic stores -> operands of the async MMAs
      if (x >= 0) mbar_arrive(smem_u32(&sm.dec_blk[blk]));
    };

    int issued = nt > 0 ? 1 : 0;
    // x = -1 is a dry pass: one block of whatever the raw buffer holds is
    // decoded into the tile buffer (rewritten by tile 0 before any MMA reads
    // it), with no wait and no arrival, so that the decode code is fetched
    // while tile 0's codes are still on their way
    for (int x = nt > 0 ? -1 : 0; x < nt && !*abort_flag; ++x) {
      if (x >= 0) wait_bar(smem_u32(&sm.raw_full), x & 1, abort_flag);
#pragma unroll 1
      for (int blk = 0; blk < (x < 0 ? 1 : kBlocks) && !*abort_flag; ++blk) {
        // block blk of the tile buffer was last read by O^T x - 1 (and S^T
        // x - 1, which completed before it)
        if (x > 0) wait_bar(smem_u32(&sm.o_blk[blk]), (x - 1) & 1, abort_flag);
        decode_block(x, blk);
      }
      // the raw buffer is free once every decode thread is done with tile x
      if (x >= 0 && tma_thread && issued < nt) {
        wait_bar(smem_u32(&sm.dec_blk[kBlocks - 1]), x & 1, abort_flag);
        if (!*abort_flag) issue_raw(issued++);
      }
    }
    if (tma_thread) {
      if (!dep_done) griddep_wait();   // the grid ends after the append it overlapped
      // no copy in flight at exit (bounded waits)
      if (issued > 0) {
        mbar_wait(smem_u32(&sm.raw_full), (issued - 1) & 1);
        mbar_wait(smem_u32(&sm.pe_full[(issued - 1) & 1]), ((issued - 1) >> 1) & 1);
      }
    }
  }

  // softmax state (warps 0-3: one token per thread, all 16 heads)
  float m[kMlaHeads], l[kMlaHeads];
#pragma unroll
  for (int h = 0; h < kMlaHeads; ++h) m[h] = -INFINITY, l[h] = 0.f;
  if (warp < kSoftWarps) {
    // ============================================================ softmax
    float qf[kMlaHeads];
#pragma unroll
    for (int h = 0; h < kMlaHeads; ++h) qf[h] = 0.f;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
    // t = -1 is a dry pass of the loop's code while tile 0 is loaded and
    // decoded (after the L2 flush its first run would fetch the unrolled
    // instructions from DRAM when the first scores wait): every token is
    // masked, so m and l do not move, and nothing is handed over.
    for (int t = -1; t < nt; ++t) {
      if (t == 0) {
        asm volatile("bar.sync 2, %0;" ::"n"(kDecoders + 32 * kSoftWarps) : "memory");
#pragma unroll
        for (int h = 0; h < kMlaHeads; ++h) qf[h] = sm.qfac[h];
      }
      if (t >= 0) wait_bar(smem_u32(&sm.s_done[t & 1]), (t >> 1) & 1, abort_flag);
      tc_fence_after();
      uint32_t sl[16], sp[16];
      tmem_ld16(lane_addr + kColSLat + 16 * (t & 1), sl);
      tmem_ld16(lane_addr + kColSPe + 16 * (t & 1), sp);
      tmem_wait_ld();
      const int r = tid;   // token of the tile
      const bool valid = t >= 0 && r < ntok - t * kT && !*abort_flag;
      float xs[kMlaHeads];
      bool need = false;
#pragma unroll
      for (int h = 0; h < kMlaHeads; ++h) {
        xs[h] = valid ? __uint_as_float(sl[h]) * qf[h] + __uint_as_float(sp[h]) * a.pe_scale_log2
                      : -INFINITY;
        need |= xs[h] > m[h] + kLazyMax;
      }
      need = __any_sync(0xffffffffu, need);
      if (lane == 0) sm.need[warp] = need;
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kSoftWarps) : "memory");
      const bool any_need = t < 0 || (sm.need[0] | sm.need[1] | sm.need[2] | sm.need[3]);
      bool resc = false;
      float alpha[kMlaHeads];
      if (any_need) {
#pragma unroll
        for (int h = 0; h < kMlaHeads; ++h) {
          float mx = xs[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          if (lane == 0) sm.wmax[warp][h] = mx;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kSoftWarps) : "memory");
#pragma unroll
        for (int h = 0; h < kMlaHeads; ++h) {
          const float mx = fmaxf(fmaxf(sm.wmax[0][h], sm.wmax[1][h]),
                                 fmaxf(sm.wmax[2][h], sm.wmax[3][h]));
          const bool mv = mx > m[h] + kLazyMax;   // also the first finite tile
          alpha[h] = mv ? ex2(m[h] - mx) : 1.f;
          m[h] = mv ? mx : m[h];
          l[h] *= alpha[h];
          resc |= alpha[h] != 1.f;
        }
      }
      // identical in all softmax threads: the maxima come from shared memory
      const bool do_resc = any_need && resc && t > 0;
      const uint32_t pt = base + kOffP + (t & 1) * kPBytes + (r >> 6) * 2048;
#pragma unroll
      for (int h = 0; h < kMlaHeads; ++h) {
        const float pv = ex2(xs[h] - (m[h] == -INFINITY ? 0.f : m[h]));
        l[h] += pv;
        sts16(pt + swz(h, r & 63), __half_as_ushort(__float2half_rn(pv)));
      }
      if (do_resc) {
        // O of the tensor-memory lanes of this warp (value dims 128 i +
        // 32 w + lane), once O^T t - 1 has completed
        wait_bar(smem_u32(&sm.o_blk[kBlocks - 1]), (t - 1) & 1, abort_flag);
        tc_fence_after();
#pragma unroll 1
        for (int i = 0; i < kBlocks; ++i) {
          uint32_t v[16];
          tmem_ld16(lane_addr + kColO + 16 * i, v);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < kMlaHeads; ++h)
            v[h] = __float_as_uint(__uint_as_float(v[h]) * alpha[h]);
          tmem_st16(lane_addr + kColO + 16 * i, v);
        }
        tmem_wait_st();
      }
      fence_proxy_async_shared();
      tc_fence_before();
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kSoftWarps) : "memory");   // all of P^T and O
      if (tid == 0 && t >= 0) mbar_arrive(smem_u32(&sm.p_ready[t & 1]));   // O^T MMAs t may go
      if (*abort_flag) break;
    }
    // denominators over the tile's tokens; the reference max
#pragma unroll
    for (int h = 0; h < kMlaHeads; ++h) {
      float v = l[h];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) sm.lsum[warp][h] = v;
      if (tid == 0) sm.m[h] = m[h];
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool bad = *abort_flag != 0;
  if (bad && tid == 0) record_error(a.error_flag, 1);

  // ---- partials: warp w < 4 holds dims 128 i + 32 w + lane of every block i;
  // to global memory, or (cluster merge) to this CTA's shared memory:
  // [head][512] floats in the free tile buffer, the lse after them
  const size_t part_row = (size_t)b * kMlaHeads;
  const bool cl = a.cluster_merge != 0;
  float* own = reinterpret_cast<float*>(gbase + kOffTile);
  float* own_lse = own + kMlaHeads * kMlaLat;
  // one thread per head: the factor and the lse (this code runs cold, once
  // per CTA: one short sequence instead of sixteen per thread)
  if (tid < kMlaHeads) {
    const float lt = (sm.lsum[0][tid] + sm.lsum[1][tid]) + (sm.lsum[2][tid] + sm.lsum[3][tid]);
    sm.fac[tid] = bad ? NAN : lt > 0.f ? __fdividef(a.out_mult, lt) : 0.f;
    const float mm = sm.m[tid];
    const float lse =
        bad ? NAN : (mm == -INFINITY || lt == 0.f) ? -INFINITY : (mm + log2f(lt)) * kLn2;
    if (cl)
      own_lse[tid] = lse;
    else
      a.part_lse[(part_row + tid) * a.num_splits + split] = lse;
  }
  if (warp < kSoftWarps) {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kSoftWarps) : "memory");   // factors written
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
    // the four blocks' accumulators in one round trip
    uint32_t v[kBlocks][16];
    if (nt > 0 && !bad) {
#pragma unroll
      for (int i = 0; i < kBlocks; ++i) tmem_ld16(lane_addr + kColO + 16 * i, v[i]);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int i = 0; i < kBlocks; ++i)
#pragma unroll
        for (int h = 0; h < kMlaHeads; ++h) v[i][h] = 0u;
    }
    const size_t hstride = cl ? (size_t)kMlaLat : (size_t)a.num_splits * kMlaLat;
    float* po = (cl ? own : a.part_o + (part_row * a.num_splits + split) * kMlaLat) + 32 * warp + lane;
#pragma unroll
    for (int h = 0; h < kMlaHeads; ++h) {
      const float f = sm.fac[h];
#pragma unroll
      for (int i = 0; i < kBlocks; ++i) po[(size_t)h * hstride + 128 * i] = __uint_as_float(v[i][h]) * f;
    }
  }
  // ---- tensor memory back; then the fused combine
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
  // fused combine: through the cluster's shared memory, or with the
  // partials of the request (16 x s x 512 floats) staged in the tile buffer
  // (128 KB) and the weights in the raw buffer
  if (cl)
    fused_combine_cluster(a, part_row, kMlaHeads, base + kOffTile,
                          base + kOffTile + kMlaHeads * kMlaLat * 4,
                          reinterpret_cast<float*>(gbase + kOffRaw));
  else if (a.counters)
    fused_combine_staged<32, 4>(a, b, part_row, kMlaHeads, base + kOffTile,
                                reinterpret_cast<const float*>(gbase + kOffTile), kTileBytes,
                                reinterpret_cast<float*>(gbase + kOffRaw), smem_u32(&sm.comb_full));
}
}  // namespace

namespace {
// Clusters of s CTAs of this kernel that fit on the device at once (cached
// per device and s; 0 when the query fails).
int mla_max_clusters(int dev, int s) {
  constexpr int kDevs = 64;
  static std::atomic<int> cache[kDevs][kMaxClusterSplits + 1];
  if (dev < 0 || dev >= kDevs) return 0;
  const int c = cache[dev][s].load(std::memory_order_relaxed);
  if (c > 0) return c - 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(1, s);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)s;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, mla_tc_kernel, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  cache[dev][s].store(n + 1, std::memory_order_relaxed);
  return n;
}
}  // namespace

// The fused decode (arrival counters given) with 2..8 splits runs as
// clusters of the s splits of a request, whose partials then merge through
// distributed shared memory, when the clusters that fit at once cover the
// grid in no more waves than single CTAs would (one CTA per SM).
cudaError_t launch_mla_partial(const CUtensorMap& tcodes, const CUtensorMap& tpe,
                               const CUtensorMap& tcodes64, const CUtensorMap& tpe64,
                               const PartialArgs& a, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  PartialArgs args = a;
  args.cluster_merge = 0;
  const int s = a.num_splits;
  if (a.counters && s >= 2 && s <= kMaxClusterSplits) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        sms > 0) {
      const long maxc = mla_max_clusters(dev, s);
      if (maxc > 0 && (a.batch + maxc - 1) / maxc <= ((long)a.batch * s + sms - 1) / sms)
        args.cluster_merge = 1;
    } else {
      (void)cudaGetLastError();
    }
  }
  if (args.cluster_merge)
    return launch_pdl_cluster(mla_tc_kernel, dim3(a.batch, s), dim3(kThreads),
                              (size_t)kSmemBytes, s, st, tcodes, tpe, tcodes64, tpe64, args);
  return launch_pdl(mla_tc_kernel, dim3(a.batch, s), dim3(kThreads), (size_t)kSmemBytes, st,
                    tcodes, tpe, tcodes64, tpe64, args);
}

}  // namespace kvq
