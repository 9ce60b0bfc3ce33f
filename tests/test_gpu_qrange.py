"""The decode takes the whole bf16 range of q.

The query is unquantized bf16 (Model-Optimizer PR 714, Testing: the
q_bmm_quantizer is disabled).  The kernels feed it to f16 tensor-core
operands after a per-head power-of-two prescale, so magnitudes far outside
f16's range (above 65504 or below 2^-14) must still give the oracle's
result.  The cases pair scaled queries with keys scaled the other way, so
that the scores stay O(1) and the softmax is not one-hot: a wrong magnitude
anywhere changes the output, and an overflow in the f16 conversion gives
NaN.  Heads of one kv-head group get different magnitudes (the prescale is
per head), and one case mixes huge and tiny elements inside one head."""
import numpy as np
import pytest
import torch

from kvq_testlib import Setup, assert_f32_close
from quantized_kv_cache_05_gb300 import build as kbuild
from quantized_kv_cache_05_gb300 import kvq, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kvq.lib()
    torch.cuda.init()


def scaled_bits(bits: np.ndarray, mult) -> np.ndarray:
    """bf16 bits times a power of two (or an array of them), exactly."""
    x = synth.bf16_to_f32(bits).astype(np.float64) * mult
    out = synth.f32_to_bf16(x.astype(np.float32))
    assert np.array_equal(synth.bf16_to_f32(out).astype(np.float64), x), "inexact scaling"
    return out


def rescale(w, q_head_exp, k_exp, elem_mix=False):
    """Scale query head h by 2^q_head_exp[h % len] and every key (MLA: the
    latent and the rope keys) by 2^k_exp.  With elem_mix, every other query
    element of each head is additionally scaled by 2^-40."""
    q0, kv0, kpe0 = w.q, w.kv_rows, w.kpe_rows
    e = np.array([q_head_exp[h % len(q_head_exp)] for h in range(w.Hq)], np.float64)

    def q():
        m = np.broadcast_to((2.0 ** e)[None, :, None], (w.B, w.Hq, w.Dqk)).copy()
        if elem_mix:
            m[:, :, 1::2] *= 2.0 ** -40
        return scaled_bits(q0(), m)

    def kv_rows(tensor, b, t0=0, t1=None):
        r = kv0(tensor, b, t0, t1)
        return scaled_bits(r, 2.0 ** k_exp) if tensor == synth.T_K else r

    def kpe_rows(b, t0=0, t1=None):
        return scaled_bits(kpe0(b, t0, t1), 2.0 ** k_exp)

    w.q, w.kv_rows, w.kpe_rows = q, kv_rows, kpe_rows
    return w


def small_gqa(fmt):
    w = synth.gqa_fp8(600) if fmt == "fp8" else synth.nvfp4(600)
    w.B, w.Hq, w.Hkv = 2, 8, 2
    w.seq_lens = np.array([600, 251], np.int32)
    return w


CASES = {
    # |q| up to ~2^22 (beyond f16's 65504), keys ~2^-20: scores O(1)
    "huge_q": ([20, 22, 18, 20, 21, 19, 20, 17], -20, False),
    # |q| ~2^-20 (f16 subnormal or zero before the prescale), keys ~2^20
    "tiny_q": ([-20, -22, -18, -20, -21, -19, -24, -20], 20, False),
    # per-head magnitudes spanning 2^-30 .. 2^30 in one group, keys 2^-2
    "mixed_heads": ([30, -30, 0, 2, 15, -15, 16, -2], -2, False),
    # inside each head, huge and tiny elements side by side
    "mixed_elements": ([20, 20, 20, 20, 20, 20, 20, 20], -20, True),
}


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("case", list(CASES))
def test_gqa_q_range(fmt, case):
    qe, ke, mix = CASES[case]
    S = Setup(rescale(small_gqa(fmt), qe, ke, mix))
    ref, _ = S.oracle_decode()
    for s in (1, 3):
        out, _ = S.gpu_decode(s)
        assert_f32_close(out.cpu().numpy(), ref, f"{fmt} {case} s={s}")


@pytest.mark.parametrize("case", ["huge_q", "tiny_q"])
def test_fp8_probs_q_range(case):
    qe, ke, mix = CASES[case]
    w = synth.paged_fp8_probs(B=3, lo=40, hi=400, seed=13)
    S = Setup(rescale(w, qe, ke, mix))
    for s in (1, 2):
        ref, _ = S.oracle_decode(mode=1, s=s)
        out, _ = S.gpu_decode(s)
        assert_f32_close(out.cpu().numpy(), ref, f"probs {case} s={s}")


@pytest.mark.parametrize("case", ["huge_q", "tiny_q", "mixed_heads"])
def test_mla_q_range(case):
    """In MLA the values are the latent itself, so scaling the latent by 2^k
    scales the outputs too: both sides are compared in the values' own units
    (times 2^-k, exact)."""
    qe, ke, mix = CASES[case]
    w = synth.mla_nvfp4(B=2, L=200)
    w.seq_lens = np.array([200, 77], np.int32)
    S = Setup(rescale(w, qe, ke, mix))
    ref, _ = S.oracle_decode()
    unit = 2.0 ** -ke
    for s in (1, 2):
        out, _ = S.gpu_decode(s)
        assert_f32_close(out.cpu().numpy().astype(np.float64) * unit, ref * unit,
                         f"mla {case} s={s}")
