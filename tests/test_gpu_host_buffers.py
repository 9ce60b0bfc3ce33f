"""Per-step inputs and the decode output in pinned host memory.

The append reads k_new / v_new and the decode reads q from page-locked host
memory and writes the output there, in place; the results must be identical
to the run with the same values in device memory (the cache stays in device
memory either way)."""
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


def step(S, s, q, k, v, kpe, out, start):
    """append of one row per request, then kvq_decode (fresh_tokens = 1)."""
    cfg = S.config(s, "f32")
    cfg.fresh_tokens = 1
    ws = runtime.FusedWorkspace(cfg, S.w.Hkv, S.device)
    c = S.cache.struct()
    kvq.check(kvq.kvq_quantize_append(c, k, v, kpe, start, S.w.B, 1, None))
    p = cfg.params(S.seq_lens_t)
    kvq.check(kvq.kvq_decode(c, p, q, ws.part_o, ws.part_lse, ws.counters, out, None))
    torch.cuda.synchronize()


@pytest.mark.parametrize("mk", [lambda: synth.gqa_fp8(300), lambda: synth.mla_nvfp4(B=2, L=200)],
                         ids=["gqa_fp8", "mla"])
def test_host_inputs_and_output_match_device(mk):
    S = Setup(mk())
    w = S.w
    start = torch.tensor([int(L) - 1 for L in w.seq_lens], dtype=torch.int32, device=S.device)
    last = lambda rows: torch.from_numpy(
        np.stack([rows[b][int(w.seq_lens[b]) - 1:int(w.seq_lens[b])] for b in range(w.B)])
        .view(np.int16)).view(torch.bfloat16)
    k = last(S.k)
    v = last(S.v) if S.v else None
    kpe = last(S.kpe) if S.kpe else None
    s = runtime.auto_splits(w.B, w.Hkv, w.G, w.Lmax, w.fmt)
    shape = (w.B, w.Hq, w.Dv)

    dev = lambda x: x.to(S.device) if x is not None else None
    out_d = torch.empty(shape, dtype=torch.float32, device=S.device)
    step(S, s, S.q_t, dev(k), dev(v), dev(kpe), out_d, start)

    pin = lambda x: x.contiguous().pin_memory() if x is not None else None
    q_h = pin(S.q_t.cpu())
    out_h = torch.full(shape, float("nan"), dtype=torch.float32).pin_memory()
    step(S, s, q_h, pin(k), pin(v), pin(kpe), out_h, start)

    assert torch.equal(out_h, out_d.cpu())
    ref, _ = S.oracle_decode(s=s)
    assert_f32_close(out_h.numpy(), ref, f"{w.name} host buffers")
