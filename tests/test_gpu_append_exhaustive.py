"""Quantize-on-append over every finite bf16 input, bit-exact vs the oracle.

The append kernels divide by the scale with a reciprocal and one fused
correction, and fall back to the IEEE division wherever the quotient could be
an E4M3 (E2M1) rounding boundary or next to one.  The codes must therefore be
those of E4M3(fl32(x / scale)) (compressed-tensors PR 436 per-tensor FP8) and
of the NVFP4 block quantizer (Model-Optimizer PR 714: E2M1 in blocks of 16,
E4M3 block scales, fp32 global scale) for every input.  Every finite bf16 bit
pattern (65,280 of them) is appended as K and, in another order, as V, at
several scales, including ones that make quotients overflow or underflow."""
import numpy as np
import pytest
import torch

import oracle
from kvq_testlib import to_dev_bf16
from quantized_kv_cache_05_gb300 import build as kbuild
from quantized_kv_cache_05_gb300 import kvq, runtime

pytestmark = pytest.mark.gpu

D = 128
SCALES = [1.0, float(np.float32(1 / 3)), float(np.float32(7.53125 / 448)),
          float(np.float32(0.0123)), float(np.float32(2.5e-5)), float(np.float32(3e4))]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kvq.lib()
    torch.cuda.init()


def all_finite_bf16(order: int) -> np.ndarray:
    """Every finite bf16 pattern, zero-padded to whole rows of D; order 0 is
    ascending, order 1 a seeded shuffle (mixes magnitudes inside NVFP4
    blocks)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = ((bits >> 7) & 0xFF) != 0xFF
    x = bits[finite]
    if order == 1:
        x = x[np.random.default_rng(7).permutation(x.size)]
    pad = (-x.size) % D
    return np.concatenate([x, np.zeros(pad, np.uint16)]).reshape(-1, D)


def append_all(fmt: str, scale: float):
    k = all_finite_bf16(0)
    v = all_finite_bf16(1)
    T = k.shape[0]
    ps = -(-T // 16) * 16
    bt = torch.zeros((1, 1), dtype=torch.int32)
    cache = runtime.QuantizedKVCache(fmt, 1, ps, 1, D, bt, scale, scale)
    kt = to_dev_bf16(k[None, :, None, :])
    vt = to_dev_bf16(v[None, :, None, :])
    start = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache.append(kt, vt, start)
    torch.cuda.synchronize()
    return cache, k, v, T


@pytest.mark.parametrize("scale", SCALES)
def test_fp8_append_every_bf16(scale):
    cache, k, v, T = append_all("fp8", scale)
    for name, x, got in (("K", k, cache.k_codes), ("V", v, cache.v_codes)):
        want = oracle.fp8_quantize(x, scale)
        have = got.cpu().numpy()[0, 0, :T]
        bad = np.argwhere(have != want)
        assert bad.size == 0, (name, scale, len(bad), x[tuple(bad[0])], have[tuple(bad[0])],
                               want[tuple(bad[0])])


@pytest.mark.parametrize("scale", SCALES)
def test_nvfp4_append_every_bf16(scale):
    cache, k, v, T = append_all("nvfp4", scale)
    for name, x, codes, scales in (("K", k, cache.k_codes, cache.k_bscale),
                                   ("V", v, cache.v_codes, cache.v_bscale)):
        wc, ws = oracle.nvfp4_quantize(x, scale)
        assert np.array_equal(scales.cpu().numpy()[0, 0, :T], ws), (name, scale, "block scales")
        have = codes.cpu().numpy()[0, 0, :T]
        bad = np.argwhere(have != wc)
        assert bad.size == 0, (name, scale, len(bad))
