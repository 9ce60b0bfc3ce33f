"""Causal prefill attention over the quantized cache (kvq_prefill) vs the
oracle.

Model-Optimizer PR 1832 times a prefill attention kernel next to split-KV
decode.  Each request's cache holds L tokens, the last Tq of them the new
ones; query i (position L - Tq + i) attends to keys 0 .. L - Tq + i.  The
oracle runs exact attention per query prefix on its own dequantized cache;
fp32 outputs must be within 2e-3 and cosine 0.9999, bf16 within one step.
Cases: Tq = 1 (the decode shape the pages compare), Tq spanning several
query tiles, GQA 4:1 and 16:1, FP8 and NVFP4 caches, paged and ragged
requests, a request shorter than its query count."""
import numpy as np
import pytest
import torch

import oracle
from kvq_testlib import Setup, assert_bf16_close, assert_f32_close, bf16_bits, to_dev_bf16
from quantized_kv_cache_05_gb300 import build as kbuild
from quantized_kv_cache_05_gb300 import kvq, runtime, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kvq.lib()
    torch.cuda.init()


def queries(w, Tq):
    """[B][Tq][Hq][D] bf16 from the query stream (offset past the decode q)."""
    n = w.B * Tq * w.Hq * w.D
    return synth.fill_bf16(w.seed, synth.T_Q, n, offset=1 << 24).reshape(w.B, Tq, w.Hq, w.D)


def oracle_prefill(S, q, Tq):
    w = S.w
    out = np.zeros((w.B, Tq, w.Hq, w.Dv))
    qf = synth.bf16_to_f32(q).astype(np.float64)
    for b in range(w.B):
        L = int(w.seq_lens[b])
        for h in range(w.Hkv):
            kh, vh = S.oracle_kv(b, h)
            for g in range(w.G):
                hq = h * w.G + g
                n = min(Tq, L)            # queries with a position >= 0
                if n == 0:
                    continue
                o, _ = oracle.prefill_attention(qf[b, Tq - n:, hq], kh, vh, w.sm_scale)
                out[b, Tq - n:, hq] = o
    return out


def run(S, q, Tq, out="f32"):
    cfg = S.config(1, out)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = runtime.prefill(S.cache, to_dev_bf16(q), S.seq_lens_t, cfg, Tq, error_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    return o


def workload(fmt, D, hq, hkv, lens, paged):
    w = synth.gqa_fp8(int(max(lens))) if fmt == "fp8" else synth.nvfp4(int(max(lens)))
    w.D, w.B, w.Hq, w.Hkv = D, len(lens), hq, hkv
    w.seq_lens = np.array(lens, np.int32)
    if paged:
        w.page_size, w.permute_pages = 16, True
    return w


@pytest.mark.parametrize("Tq", [1, 5, 37])
@pytest.mark.parametrize("fmt,D", [("fp8", 128), ("nvfp4", 64)])
def test_prefill(fmt, D, Tq):
    S = Setup(workload(fmt, D, 8, 2, [700, 233, 40], paged=(fmt == "nvfp4")))
    q = queries(S.w, Tq)
    ref = oracle_prefill(S, q, Tq)
    got = run(S, q, Tq).cpu().numpy()
    assert_f32_close(got, ref, f"{fmt} D={D} Tq={Tq}")


def test_prefill_many_heads_and_tiles_bf16():
    """16 query heads per kv head and 9 new tokens: 144 rows, three tiles."""
    S = Setup(workload("fp8", 64, 16, 1, [300, 129], paged=True))
    q = queries(S.w, 9)
    ref = oracle_prefill(S, q, 9)
    got = run(S, q, 9, "bf16")
    assert_bf16_close(bf16_bits(got), ref, "G=16 Tq=9 bf16")


def test_prefill_request_shorter_than_queries():
    """A request of 3 tokens with 5 queries: the two queries before position 0
    attend to nothing and give 0."""
    S = Setup(workload("fp8", 128, 8, 2, [300, 3], paged=False))
    q = queries(S.w, 5)
    ref = oracle_prefill(S, q, 5)
    got = run(S, q, 5).cpu().numpy()
    assert np.all(got[1, :2] == 0)
    assert_f32_close(got, ref, "short request")


def test_prefill_single_query_equals_decode():
    """With one new token the prefill output is the decode output."""
    S = Setup(workload("fp8", 128, 8, 2, [1000, 517], paged=False))
    q = queries(S.w, 1)
    pf = run(S, q, 1).cpu().numpy()[:, 0]
    cfg = S.config(4, "f32")
    dec = runtime.decode(S.cache, to_dev_bf16(q[:, 0]), S.seq_lens_t, cfg).cpu().numpy()
    assert np.max(np.abs(pf - dec)) <= 1e-4
