"""Per-kv-head ("attn_head") static scales on the GPU vs the oracle.

compressed-tensors PR 436 adds the "attn_head" strategy (one static FP8
scale per attention head; its GSM8K table has a KV-FP8-Head row).  The cache
takes optional device arrays of per-kv-head scales for K and V.  These tests
calibrate them with the amax kernel per head (equal to the oracle's), append
through the C ABI (codes bit-exact against the oracle's per-head quantizer)
and decode (fp32 output within 2e-3 and cosine 0.9999 of the oracle on the
per-head dequantized cache).  The kv heads get different magnitudes (powers
of two), so per-head and per-tensor codes differ."""
import numpy as np
import pytest
import torch

from kvq_testlib import Setup, assert_f32_close
from quantized_kv_cache_05_gb300 import build as kbuild
from quantized_kv_cache_05_gb300 import kvq, runtime, synth

pytestmark = pytest.mark.gpu

SKEW = (0, -7, 3, -2)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kvq.lib()
    torch.cuda.init()


def gqa(head_scales=True, fmt="fp8", paged=False, probs=False):
    w = synth.gqa_fp8(700) if fmt == "fp8" else synth.nvfp4(700)
    w.B, w.Hq, w.Hkv = 2, 16, 4
    w.seq_lens = np.array([700, 233], np.int32)
    w.head_scales, w.head_exp = head_scales, SKEW
    if paged:
        w.page_size, w.permute_pages = 16, True
    w.prob_fp8 = probs
    return w


def check_codes(S):
    w = S.w
    for b in range(w.B):
        for h in range(w.Hkv):
            for which in ("k", "v"):
                codes, bs = S.oracle_codes(which, b, h)
                assert np.array_equal(S.gpu_rows(which, b, h), codes), (which, b, h)
                if bs is not None:
                    assert np.array_equal(S.gpu_rows(which + "s", b, h), bs), (which, b, h)


def fused(S, s):
    cfg = S.config(s, "f32")
    flag = torch.zeros(1, dtype=torch.int32, device=S.device)
    out = runtime.decode_fused(S.cache, S.q_t, S.seq_lens_t, cfg, None, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_head_scales_codes_and_decode(fmt):
    S = Setup(gqa(True, fmt))
    assert len(set(S.k_head.tolist())) == len(SKEW)   # one scale per head, all different
    check_codes(S)
    ref, _ = S.oracle_decode()
    w = S.w
    for s in (1, 3, 0):
        s = s or runtime.auto_splits(w.B, w.Hkv, w.G, w.Lmax, w.fmt)
        out, _ = S.gpu_decode(s)
        assert_f32_close(out.cpu().numpy(), ref, f"{fmt} head scales s={s}")
        assert_f32_close(fused(S, s), ref, f"{fmt} head scales fused s={s}")


def test_head_scales_change_the_codes():
    """The same skewed cache with one scale per tensor stores other codes for
    the small heads (and the same for the head that sets the tensor's amax)."""
    Sh = Setup(gqa(True))
    St = Setup(gqa(False))
    check_codes(St)
    big = int(np.argmax(SKEW))
    for h in range(4):
        a, b = Sh.gpu_rows("k", 0, h), St.gpu_rows("k", 0, h)
        if h == big:
            assert np.array_equal(a, b)
        else:
            assert not np.array_equal(a, b)


def test_head_scales_paged_fp8_probs():
    S = Setup(gqa(True, "fp8", paged=True, probs=True))
    check_codes(S)
    for s in (1, 2):
        ref, _ = S.oracle_decode(mode=1, s=s)
        out, _ = S.gpu_decode(s)
        assert_f32_close(out.cpu().numpy(), ref, f"paged probs head scales s={s}")
        assert_f32_close(fused(S, s), ref, f"paged probs head scales fused s={s}")
