"""kvq_decode_noalloc, the allocation-free decode entry point.

Some callers cannot allocate device memory for scratch: their device memory
belongs to a host framework's fixed pool, or a memory budget forbids another
cudaMalloc.  kvq_decode_noalloc keeps the split partials and arrival counters
in the library's own static device buffer (4 MiB).  These tests call it
through the C ABI twice in a row and compare each result with kvq_decode
(caller-owned buffers) within the fp32 tolerance the other tests use; check
a request that fills the buffer exactly and refuse the next larger one; and
run it right after an append with fresh_tokens = 1 (accepted; the decode
then simply starts after the append).  This file is
collected last so that a run stopping at the first failure has already run
everything else; it also passes on its own in a fresh process.
"""
import math

import numpy as np
import pytest
import torch

from kvq_testlib import Setup, assert_f32_close, to_dev_bf16
from quantized_kv_cache_05_gb300 import build as kbuild
from quantized_kv_cache_05_gb300 import kvq, runtime, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kvq.lib()
    torch.cuda.init()


def _workloads():
    tiny = synth.tiny_fp8()
    gqa = synth.gqa_fp8(1000)
    paged = synth.paged_fp8_probs(B=4, lo=20, hi=400, seed=7)
    mla = synth.mla_nvfp4(B=2, L=250)
    return [(tiny, 2), (gqa, 0), (paged, 2), (mla, 3)]


@pytest.mark.parametrize("case", range(4), ids=["tiny_fp8", "gqa_fp8", "paged_probs", "mla"])
def test_noalloc_matches_kvq_decode_on_two_calls(case):
    w, s = _workloads()[case]
    S = Setup(w)
    if s == 0:
        s = runtime.auto_splits(w.B, w.Hkv, w.G, w.Lmax, w.fmt)
    cfg = S.config(s, "f32")
    ref = runtime.decode_fused(S.cache, S.q_t, S.seq_lens_t, cfg).clone()
    torch.cuda.synchronize()
    ref64 = ref.cpu().numpy().astype(np.float64)
    out = torch.empty_like(ref)
    p = cfg.params(S.seq_lens_t)
    for call in range(2):
        out.fill_(math.nan)
        st = kvq.kvq_decode_noalloc(S.cache.struct(), p, S.q_t, out)
        assert st == kvq.KVQ_OK, kvq.status_string(st)
        torch.cuda.synchronize()
        assert_f32_close(out.cpu().numpy(), ref64, f"{w.name} no-alloc call {call}")


def test_noalloc_refuses_requests_beyond_its_buffer():
    w = synth.gqa_fp8(1000)
    S = Setup(w)
    # 2 x 32 heads x 64 splits x 128 dims x 4 B = 2 MiB fits; batch 4 would not
    cfg = S.config(64, "f32")
    p = cfg.params(S.seq_lens_t)
    out = torch.empty((w.B, w.Hq, w.Dv), dtype=torch.float32, device="cuda")
    assert kvq.kvq_decode_noalloc(S.cache.struct(), p, S.q_t, out) == kvq.KVQ_OK
    p.batch = 4
    need = 4 * 32 * 64 * (128 + 1) * 4
    assert need > kvq.KVQ_NOALLOC_SCRATCH_BYTES
    assert kvq.kvq_decode_noalloc(S.cache.struct(), p, S.q_t, out) == kvq.KVQ_ERR_WORKSPACE


def _exact_fit_workload():
    """64 requests x 4 kv heads (MHA, head_dim 64), 63 splits: counters
    1 KiB + partial lse 63 KiB + partial o 4032 KiB = exactly 4 MiB."""
    w = synth.Workload("noalloc_fit", "fp8", 64, 4, 4, 64, np.full(64, 1008, np.int32))
    rows = w.B * w.Hq * 63
    need = 4 * w.B * w.Hkv + 4 * rows + 4 * rows * w.Dv
    assert need == kvq.KVQ_NOALLOC_SCRATCH_BYTES
    return w


def test_noalloc_exact_fit_and_one_more_request():
    w = _exact_fit_workload()
    S = Setup(w)
    cfg = S.config(63, "f32")
    ref = runtime.decode_fused(S.cache, S.q_t, S.seq_lens_t, cfg).clone()
    torch.cuda.synchronize()
    out = torch.full_like(ref, math.nan)
    p = cfg.params(S.seq_lens_t)
    assert kvq.kvq_decode_noalloc(S.cache.struct(), p, S.q_t, out) == kvq.KVQ_OK
    torch.cuda.synchronize()
    assert_f32_close(out.cpu().numpy(), ref.cpu().numpy().astype(np.float64), "exact fit")
    # one more request needs 4 B of counters and 63 rows of partials more
    p.batch = w.B + 1
    assert kvq.kvq_decode_noalloc(S.cache.struct(), p, S.q_t, out) == kvq.KVQ_ERR_WORKSPACE


def test_noalloc_after_append_with_fresh_tokens():
    """Append each request's last row (other values first, then the true
    row), then kvq_decode_noalloc with fresh_tokens = 1 on the same stream:
    the result equals kvq_decode's on the true cache."""
    w = synth.gqa_fp8(700)
    w.B, w.Hq, w.Hkv = 2, 8, 2
    w.seq_lens = np.array([700, 129], np.int32)
    S = Setup(w)
    cfg = S.config(3, "f32")
    ref = runtime.decode_fused(S.cache, S.q_t, S.seq_lens_t, cfg).clone()
    torch.cuda.synchronize()
    last = [int(L) - 1 for L in w.seq_lens]
    k_last = to_dev_bf16(np.stack([S.k[b][last[b]:last[b] + 1] for b in range(w.B)]))
    v_last = to_dev_bf16(np.stack([S.v[b][last[b]:last[b] + 1] for b in range(w.B)]))
    start = torch.tensor(last, dtype=torch.int32, device="cuda")
    c = S.cache.struct()
    # stale rows (sign-flipped) first, so that reading before the append shows
    kvq.check(kvq.kvq_quantize_append(c, -k_last, -v_last, None, start, w.B, 1))
    torch.cuda.synchronize()
    out = torch.full_like(ref, math.nan)
    p = cfg.params(S.seq_lens_t)
    p.fresh_tokens = 1
    kvq.check(kvq.kvq_quantize_append(c, k_last, v_last, None, start, w.B, 1))
    assert kvq.kvq_decode_noalloc(c, p, S.q_t, out) == kvq.KVQ_OK
    torch.cuda.synchronize()
    assert_f32_close(out.cpu().numpy(), ref.cpu().numpy().astype(np.float64), "fresh_tokens=1")
