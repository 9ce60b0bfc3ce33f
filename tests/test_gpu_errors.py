"""Device error bits of the decode kernels, raised by bad host inputs.

Wrong inputs must be reported, not silently absorbed (Model-Optimizer PR
673 fixes KV scales that silently defaulted to 1).  The decode kernels
check two inputs they read on the device and keep every access in bounds:
  * seq_lens[b] above the cache (max_kv_len, or the block table's
    capacity) is clamped and sets KVQ_DEVERR_SEQ_CLAMPED;
  * a block-table entry outside [0, num_pages) reads page 0 instead and
    sets KVQ_DEVERR_BAD_PAGE.
Each test makes one of them fire and checks the bit and the output, which
must be the oracle's on the clamped or page-0 reading.  No access leaves
the caller's buffers in either case, so nothing here can fault the GPU."""
import numpy as np
import pytest
import torch

import oracle
from kvq_testlib import Setup, assert_f32_close
from quantized_kv_cache_05_gb300 import build as kbuild
from quantized_kv_cache_05_gb300 import kvq, runtime, synth

pytestmark = pytest.mark.gpu

SEQ_CLAMPED, BAD_PAGE = 2, 4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kvq.lib()
    torch.cuda.init()


def run(S, s, seq_lens_t, fused):
    cfg = S.config(s, "f32")
    flag = torch.zeros(1, dtype=torch.int32, device=S.device)
    if fused:
        out = runtime.decode_fused(S.cache, S.q_t, seq_lens_t, cfg, None, flag)
    else:
        out = runtime.decode(S.cache, S.q_t, seq_lens_t, cfg, None, flag)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(flag.item())


def oracle_rows(S, bt):
    """Oracle (K^, V^) of every request as the decode reads them through the
    block table `bt`: physical page P holds the rows that the original table
    put there, and an entry outside [0, num_pages) reads page 0."""
    w, ps = S.w, S.ps
    owner = {}
    for b in range(w.B):
        for p in range(-(-int(w.seq_lens[b]) // ps)):
            owner[int(S.bt[b, p])] = (b, p)
    kv = {}
    for b in range(w.B):
        for h in range(w.Hkv):
            kv[(b, h)] = S.oracle_kv(b, h)
    npages = S.cache.num_pages

    def rows(b, h, L):
        kh0, vh0 = kv[(b, h)]
        K = np.zeros((L, kh0.shape[1]))
        V = np.zeros((L, vh0.shape[1]))
        for t in range(L):
            pg = int(bt[b, t // ps])
            if pg < 0 or pg >= npages:
                pg = 0
            if pg in owner:
                ob, op = owner[pg]
                src = op * ps + t % ps
                if src < int(w.seq_lens[ob]):
                    K[t], V[t] = kv[(ob, h)][0][src], kv[(ob, h)][1][src]
        return K, V
    return rows


def oracle_out(S, rows, lens):
    w = S.w
    q = S.q64()
    out = np.zeros((w.B, w.Hq, w.Dv))
    for b in range(w.B):
        for h in range(w.Hkv):
            K, V = rows(b, h, int(lens[b]))
            qs = q[b, h * w.G:(h + 1) * w.G][None]
            o, _ = oracle.decode_batch(qs, K[None, None], V[None, None], np.array([int(lens[b])]),
                                       w.sm_scale)
            out[b, h * w.G:(h + 1) * w.G] = o[0]
    return out


def gqa_setup(paged):
    w = synth.gqa_fp8(300)
    w.B, w.Hq, w.Hkv = 3, 8, 2
    w.seq_lens = np.array([300, 200, 77], np.int32)
    if paged:
        w.page_size, w.permute_pages = 16, True
    return Setup(w)


def mla_setup():
    w = synth.mla_nvfp4(B=2, L=160)
    w.seq_lens = np.array([160, 90], np.int32)
    w.page_size, w.permute_pages = 16, True
    return Setup(w)


@pytest.mark.parametrize("kind", ["gqa_contiguous", "gqa_paged", "mla_paged"])
@pytest.mark.parametrize("fused", [False, True], ids=["two_launch", "fused"])
def test_seq_len_clamped(kind, fused):
    """seq_lens[1] far above max_kv_len: the kernels read max_kv_len tokens
    (the cache rows never written are zero codes) and set the bit."""
    S = mla_setup() if kind == "mla_paged" else gqa_setup(kind == "gqa_paged")
    w = S.w
    lens = w.seq_lens.copy()
    lens[1] = 1 << 20
    cap = w.Lmax   # max_kv_len of the call (below the block table's capacity)
    seq_t = torch.from_numpy(lens).to(S.device)
    out, flag = run(S, 3, seq_t, fused)
    assert flag & SEQ_CLAMPED, flag
    assert not flag & BAD_PAGE, flag
    eff = np.minimum(lens, cap)
    # past its own pages request 1 reads what its block-table entries name
    # (the table is padded with page 0); oracle_rows follows the same table
    ref = oracle_out(S, oracle_rows(S, S.bt), eff)
    assert_f32_close(out, ref, f"{kind} clamped")


@pytest.mark.parametrize("kind", ["gqa_contiguous", "gqa_paged", "mla_paged"])
@pytest.mark.parametrize("bad", [-1, 1 << 30], ids=["negative", "past_end"])
def test_bad_page_reads_page_zero(kind, bad):
    S = mla_setup() if kind == "mla_paged" else gqa_setup(kind == "gqa_paged")
    bt = S.bt.copy()
    # request 1: its first page (contiguous) or its third page (paged)
    p = 0 if kind == "gqa_contiguous" else 2
    bt[1, p] = bad
    S.cache.block_table.copy_(torch.from_numpy(bt))
    for fused in (False, True):
        out, flag = run(S, 2, S.seq_lens_t, fused)
        assert flag == BAD_PAGE, flag
        ref = oracle_out(S, oracle_rows(S, bt), S.w.seq_lens)
        assert_f32_close(out, ref, f"{kind} bad page {bad} fused={fused}")


def test_good_inputs_leave_the_flag_clear():
    S = gqa_setup(True)
    for fused in (False, True):
        _, flag = run(S, 3, S.seq_lens_t, fused)
        assert flag == 0
