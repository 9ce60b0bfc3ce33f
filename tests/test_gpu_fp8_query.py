"""FP8 query on the GPU vs the oracle.

compressed-tensors PR 436 calibrates a query observer next to K and V
("QKV-FP8-Tensor" / "QKV-FP8-Head"); vLLM PR 15734 quantizes QK in the
attention loop.  The query scale comes from the amax kernel (per tensor or
per query head), kvq_quantize_fp8 makes the E4M3 codes (bit-exact against
the oracle), and the decode takes them with q_fp8 = 1: with an FP8 cache the
scores run on E4M3 x E4M3 MMAs from the cached bytes, with an NVFP4 cache on
f16.  Outputs must match the oracle on the dequantized query within 2e-3
and cosine 0.9999."""
import numpy as np
import pytest
import torch

import oracle
from kvq_testlib import Setup, assert_e4m3_close, assert_f32_close, to_dev_bf16
from quantized_kv_cache_05_gb300 import build as kbuild
from quantized_kv_cache_05_gb300 import kvq, runtime, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kvq.lib()
    torch.cuda.init()


def gpu_q_codes(S, per_head):
    """(codes tensor, q scale float, head-scale tensor or None, oracle
    dequantized q) through the product path, checked against the oracle."""
    w = S.w
    fmt = kvq.KVQ_FP8_E4M3
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    codes = torch.empty((w.B, w.Hq, w.D), dtype=torch.uint8, device="cuda")
    if per_head:
        hs = []
        for h in range(w.Hq):
            x = to_dev_bf16(np.ascontiguousarray(S.q[:, h]))
            kvq.check(kvq.kvq_amax_bf16(x, x.numel(), amax))
            st, sc = kvq.kvq_tensor_scale(fmt, float(amax.item()))
            kvq.check(st)
            hs.append(sc)
        hs = np.array(hs, np.float32)
        assert np.array_equal(hs, oracle.fp8_head_scales(S.q))   # q [B][Hq][D]: rows = B
        hs_t = torch.from_numpy(hs).cuda()
        kvq.check(kvq.kvq_quantize_fp8(S.q_t, S.q_t.numel(), 0.0, hs_t, w.D, w.Hq, codes))
        ref_codes, deq = oracle.fp8_query(S.q, hs)
        qs = 1.0
    else:
        kvq.check(kvq.kvq_amax_bf16(S.q_t, S.q_t.numel(), amax))
        st, qs = kvq.kvq_tensor_scale(fmt, float(amax.item()))
        kvq.check(st)
        assert qs == oracle.fp8_tensor_scale(oracle.amax_bf16(S.q))
        kvq.check(kvq.kvq_quantize_fp8(S.q_t, S.q_t.numel(), qs, None, 0, 0, codes))
        ref_codes, deq = oracle.fp8_query(S.q, qs)
        hs_t = None
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), ref_codes)
    return codes, qs, hs_t, deq


def oracle_out(S, qdeq, mode=0, s=1):
    w = S.w
    out = np.zeros((w.B, w.Hq, w.Dv))
    for b in range(w.B):
        for h in range(w.Hkv):
            kh, vh = S.oracle_kv(b, h)
            qq = qdeq[b, h * w.G:(h + 1) * w.G][None]
            o, _ = oracle.decode_batch(qq, kh[None, None], vh[None, None],
                                       np.array([int(w.seq_lens[b])]), w.sm_scale, mode=mode,
                                       s=s, prob_scale=w.prob_scale)
            out[b, h * w.G:(h + 1) * w.G] = o[0]
    return out


def run(S, codes, qs, hs, s, fused, out="f32", out_scale=1.0):
    cfg = S.config(s, out, out_scale)
    cfg.q_fp8, cfg.q_scale, cfg.q_head_scale = True, qs, hs
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    if fused:
        o = runtime.decode_fused(S.cache, codes, S.seq_lens_t, cfg, None, flag)
    else:
        o = runtime.decode(S.cache, codes, S.seq_lens_t, cfg, None, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    return o.cpu().numpy()


CASES = {
    "gqa_fp8_d128": lambda: _gqa("fp8", 128, 16, 4),
    "gqa_fp8_d64_g16": lambda: _gqa("fp8", 64, 16, 1),
    "nvfp4_d128": lambda: _gqa("nvfp4", 128, 8, 2),
}


def _gqa(fmt, D, hq, hkv):
    w = synth.gqa_fp8(600) if fmt == "fp8" else synth.nvfp4(600)
    w.D, w.B, w.Hq, w.Hkv = D, 2, hq, hkv
    w.seq_lens = np.array([600, 97], np.int32)
    return w


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("per_head", [False, True], ids=["q_tensor", "q_head"])
def test_fp8_query_decode(case, per_head):
    S = Setup(CASES[case]())
    codes, qs, hs, deq = gpu_q_codes(S, per_head)
    ref = oracle_out(S, deq)
    for s in (1, 3):
        for fused in (False, True):
            got = run(S, codes, qs, hs, s, fused)
            assert_f32_close(got, ref, f"{case} per_head={per_head} s={s} fused={fused}")


def test_fp8_query_paged_fp8_probs_e4m3_out():
    w = synth.paged_fp8_probs(B=4, lo=30, hi=500, seed=17)
    S = Setup(w)
    codes, qs, hs, deq = gpu_q_codes(S, False)
    for s in (1, 2):
        ref = oracle_out(S, deq, mode=1, s=s)
        assert_f32_close(run(S, codes, qs, hs, s, False), ref, f"probs s={s}")
        out_scale = float(np.float32(np.float32(np.max(np.abs(ref))) / np.float32(448.0)))
        got = run(S, codes, qs, hs, s, True, "e4m3", out_scale)
        assert_e4m3_close(got, ref, out_scale, f"probs e4m3 out s={s}")


def test_fp8_query_differs_from_bf16_query():
    """The FP8-query result is the oracle's on the dequantized query, which
    is measurably not the bf16-query result (the query really is quantized)."""
    S = Setup(CASES["gqa_fp8_d128"]())
    codes, qs, hs, deq = gpu_q_codes(S, False)
    got = run(S, codes, qs, hs, 1, False)
    exact, _ = S.oracle_decode()
    assert np.max(np.abs(got - exact)) > 1e-3
