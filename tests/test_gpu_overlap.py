"""Decode overlapping the append of its step (kvq_decode_params.fresh_tokens).

The last position of every request is first filled with other rows (the
negated K/V rows); then, back to back on one stream, the true rows are
appended and the decode runs with fresh_tokens = 1.  The decode reads every
other position without waiting for the append and the appended position
only after it, so its result must be the oracle's on the true rows.  Short
requests put the appended position in the first box of a chunk (the box a
CTA loads first)."""
import numpy as np
import pytest
import torch

from kvq_testlib import Setup, assert_e4m3_close, assert_f32_close, to_dev_bf16
from quantized_kv_cache_05_gb300 import build as kbuild
from quantized_kv_cache_05_gb300 import kvq, runtime, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kvq.lib()
    torch.cuda.init()


def last_rows(S, rows, negate=False):
    """[B][1][...] bf16 device tensor of each request's last row (zeros for
    empty requests); negate flips the sign bits."""
    w = S.w
    out = []
    for b in range(w.B):
        L = int(w.seq_lens[b])
        r = rows[b][L - 1:L] if L > 0 else np.zeros((1,) + rows[b].shape[1:], np.uint16)
        r = np.ascontiguousarray(r, np.uint16)
        if negate:
            r = r ^ np.uint16(0x8000)
        out.append(r)
    return to_dev_bf16(np.stack(out), S.device)


def overlapped_step(S, s, out="f32", out_scale=1.0, fused=True):
    w = S.w
    start = torch.tensor([int(L) - 1 for L in w.seq_lens], dtype=torch.int32, device=S.device)
    k, v = last_rows(S, S.k), (last_rows(S, S.v) if S.v else None)
    kpe = last_rows(S, S.kpe) if S.kpe else None
    ks, vs = last_rows(S, S.k, True), (last_rows(S, S.v, True) if S.v else None)
    kpes = last_rows(S, S.kpe, True) if S.kpe else None
    S.cache.append(ks, vs, start, kpes)
    torch.cuda.synchronize()
    cfg = S.config(s, out, out_scale)
    cfg.fresh_tokens = 1
    flag = torch.zeros(1, dtype=torch.int32, device=S.device)
    S.cache.append(k, v, start, kpe)
    if fused:
        ws = runtime.FusedWorkspace(cfg, w.Hkv, S.device)
        res = runtime.decode_fused(S.cache, S.q_t, S.seq_lens_t, cfg, ws, flag)
    else:
        res = runtime.decode(S.cache, S.q_t, S.seq_lens_t, cfg, None, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    return res


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("s", [1, 3])
def test_overlap_gqa_fp8_short_requests(fused, s):
    w = synth.gqa_fp8(64)
    w.B = 24
    w.seq_lens = np.array([1, 2, 15, 16, 17, 31, 33, 47, 64, 5, 9, 40] * 2, np.int32)
    w.seq_lens[5] = 0
    S = Setup(w)
    ref, _ = S.oracle_decode()
    out = overlapped_step(S, s, fused=fused)
    assert_f32_close(out.cpu().numpy(), ref, f"overlap fp8 s={s}")


def test_overlap_nvfp4_long():
    S = Setup(synth.nvfp4(1000))
    s = runtime.auto_splits(S.w.B, S.w.Hkv, S.w.G, S.w.Lmax, "nvfp4")
    ref, _ = S.oracle_decode(s=s)
    out = overlapped_step(S, s)
    assert_f32_close(out.cpu().numpy(), ref, "overlap nvfp4")


def test_overlap_paged_fp8_probs():
    S = Setup(synth.paged_fp8_probs(B=6, lo=20, hi=300, seed=3))
    for s in (1, 2):
        ref, _ = S.oracle_decode(mode=1, s=s)
        out_scale = float(np.float32(np.float32(np.nanmax(np.abs(ref))) / np.float32(448.0)))
        out = overlapped_step(S, s, "e4m3", out_scale)
        assert_e4m3_close(out.cpu().numpy(), ref, out_scale, f"overlap paged s={s}")


def test_overlap_mla():
    w = synth.mla_nvfp4(B=3, L=200)
    w.seq_lens = np.array([200, 1, 77], np.int32)
    S = Setup(w)
    for s in (1, 4):
        ref, _ = S.oracle_decode(s=s)
        out = overlapped_step(S, s)
        assert_f32_close(out.cpu().numpy(), ref, f"overlap mla s={s}")
