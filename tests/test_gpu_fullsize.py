"""Full-size workloads in the launch configuration the benchmark times
(kvq_decode, split count from kvq_auto_splits, the workload's output type),
checked against the oracle on sampled (request, kv head) groups: codes and
block scales bit-exact, outputs within the comparison rules."""
import numpy as np
import pytest
import torch

from kvq_testlib import Setup, assert_bf16_close, assert_e4m3_close, assert_f32_close, bf16_bits
from quantized_kv_cache_05_gb300 import build as kbuild
from quantized_kv_cache_05_gb300 import kvq, runtime, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kvq.lib()
    torch.cuda.init()


def sampled_pairs(w):
    bs = sorted({0, w.B // 2, w.B - 1})
    hs = sorted({0, w.Hkv - 1})
    return [(b, h) for b in bs for h in hs][:4]


def run_fullsize(w, out):
    S = Setup(w)
    s = runtime.auto_splits(w.B, w.Hkv, w.G, w.Lmax, w.fmt)
    pairs = sampled_pairs(w)
    # bit-exact cache contents for the sampled groups
    for b, h in pairs:
        for which in (["k"] if w.mla else ["k", "v"]):
            codes, bs = S.oracle_codes(which, b, h)
            assert np.array_equal(S.gpu_rows(which, b, h), codes), (which, b, h)
            if bs is not None:
                assert np.array_equal(S.gpu_rows(which + "s", b, h), bs), (which, b, h)
    mode = 1 if w.prob_fp8 else 0
    ref, _ = S.oracle_decode(mode=mode, s=s, heads=pairs)
    out_scale = 1.0
    if out == "e4m3":
        m = np.nanmax(np.abs(ref))
        out_scale = float(np.float32(np.float32(m) / np.float32(448.0)))
    cfg = S.config(s, out, out_scale)
    ws = runtime.FusedWorkspace(cfg, w.Hkv, S.device)
    flag = torch.zeros(1, dtype=torch.int32, device=S.device)
    res = runtime.decode_fused(S.cache, S.q_t, S.seq_lens_t, cfg, ws, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    if out == "f32":
        assert_f32_close(res.cpu().numpy(), ref, f"{w.name} s={s}")
    elif out == "bf16":
        assert_bf16_close(bf16_bits(res), ref, f"{w.name} s={s}")
    else:
        flips = assert_e4m3_close(res.cpu().numpy(), ref, out_scale, f"{w.name} s={s}")
        assert flips <= max(2, int(np.sum(~np.isnan(ref))) // 1000)
    assert not ws.counters.any()


def test_gqa_fp8_32k():
    run_fullsize(synth.gqa_fp8(32768), "bf16")


def test_nvfp4_32k():
    run_fullsize(synth.nvfp4(32768), "f32")


def test_paged_fp8_probs_full():
    run_fullsize(synth.paged_fp8_probs(), "e4m3")


def test_mla_full():
    run_fullsize(synth.mla_nvfp4(), "f32")
