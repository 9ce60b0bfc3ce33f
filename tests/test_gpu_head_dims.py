"""NVFP4 decode at head_dim 64, 128 and 256.

The NVFP4 quantizer works on any head_dim that is a multiple of the 16-element
block (Model-Optimizer PR 714, Testing: block_sizes={-1: 16}); the decode
kernels take 64, 128 and 256.  Each case appends a ragged batch (codes and
block scales bit-exact against the oracle), then decodes it through the C ABI
with several split counts, two launches and fused, with exact and with FP8
probabilities, against the oracle on the same dequantized cache."""
import numpy as np
import pytest
import torch

from kvq_testlib import Setup, assert_f32_close
from quantized_kv_cache_05_gb300 import build as kbuild
from quantized_kv_cache_05_gb300 import kvq, runtime, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kvq.lib()
    torch.cuda.init()


def workload(D, hq, hkv, probs=False, paged=False):
    w = synth.nvfp4(600)
    w.D, w.B, w.Hq, w.Hkv = D, 3, hq, hkv
    w.seq_lens = np.array([600, 251, 17], np.int32)
    w.prob_fp8 = probs
    if paged:
        w.page_size, w.permute_pages = 16, True
    return w


def check_codes(S):
    w = S.w
    for b in range(w.B):
        for h in range(w.Hkv):
            codes, bs = S.oracle_codes("k", b, h)
            assert np.array_equal(S.gpu_rows("k", b, h), codes), ("k", b, h)
            assert np.array_equal(S.gpu_rows("ks", b, h), bs), ("ks", b, h)
            codes, bs = S.oracle_codes("v", b, h)
            assert np.array_equal(S.gpu_rows("v", b, h), codes), ("v", b, h)
            assert np.array_equal(S.gpu_rows("vs", b, h), bs), ("vs", b, h)


def fused(S, s):
    cfg = S.config(s, "f32")
    flag = torch.zeros(1, dtype=torch.int32, device=S.device)
    out = runtime.decode_fused(S.cache, S.q_t, S.seq_lens_t, cfg, None, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("D", [64, 256])
@pytest.mark.parametrize("hq,hkv", [(8, 2), (16, 1)], ids=["G4", "G16"])
def test_nvfp4_head_dim(D, hq, hkv):
    S = Setup(workload(D, hq, hkv, paged=(D == 64)))
    check_codes(S)
    ref, _ = S.oracle_decode()
    w = S.w
    for s in (1, 3, 0):
        s = s or runtime.auto_splits(w.B, w.Hkv, w.G, w.Lmax, w.fmt)
        out, _ = S.gpu_decode(s)
        assert_f32_close(out.cpu().numpy(), ref, f"D={D} G={w.G} s={s}")
        assert_f32_close(fused(S, s), ref, f"D={D} G={w.G} fused s={s}")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_nvfp4_head_dim_fp8_probs(D):
    S = Setup(workload(D, 8, 2, probs=True, paged=True))
    for s in (1, 3):
        ref, _ = S.oracle_decode(mode=1, s=s)
        out, _ = S.gpu_decode(s)
        assert_f32_close(out.cpu().numpy(), ref, f"D={D} probs s={s}")
        assert_f32_close(fused(S, s), ref, f"D={D} probs fused s={s}")
