"""The decode's division by the prob scale, over every probability.

With FP8 probabilities (vLLM PR 15734: softmax(QK^T) quantized to FP8 with
prob_output_scale) each weight p in [0, 1] becomes E4M3(fl32(p /
prob_scale)).  The kernels divide with a precomputed reciprocal and one
fused correction when the host's check accepts the prob scale, else with the
IEEE division.  kvq_encode_prob_e4m3 runs that same device code elementwise;
here it runs on every fp32 p in (0, 1] (0x00000001 .. 0x3F800000) for the
workloads' prob scale fl32(1/448) and for other scales, and every code must
equal the oracle's E4M3(fl32(p / prob_scale))."""
import numpy as np
import pytest
import torch

import oracle
from quantized_kv_cache_05_gb300 import build as kbuild
from quantized_kv_cache_05_gb300 import kvq

pytestmark = pytest.mark.gpu

SCALES = [float(np.float32(1.0 / 448.0)), float(np.float32(1.0 / 240.0)),
          float(np.float32(0.00311)), 2.0 ** -8]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kvq.lib()
    torch.cuda.init()


@pytest.mark.parametrize("prob_scale", SCALES)
def test_prob_quantizer_every_probability(prob_scale):
    chunk = 1 << 27
    last = 0x3F800000                      # 1.0f
    out = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    used = None
    total = 0
    for start in range(1, last + 1, chunk):
        n = min(chunk, last + 1 - start)
        p = torch.arange(start, start + n, dtype=torch.int32, device="cuda").view(torch.float32)
        st, used = kvq.kvq_encode_prob_e4m3(p, out, n, prob_scale)
        kvq.check(st)
        torch.cuda.synchronize()
        bad, first = oracle.count_probq_mismatch(start, prob_scale, out[:n].cpu().numpy())
        assert bad == 0, f"{bad} codes differ, first p pattern {first:#010x}"
        total += n
        del p
    assert total == last
    assert used == 1, "the reciprocal path was expected for this prob scale"
