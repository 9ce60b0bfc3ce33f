"""Pins of the FP8-query path of the oracle.

compressed-tensors PR 436 calibrates a query observer next to the K and V
ones ("QKV-FP8-Tensor" and "QKV-FP8-Head" rows of its GSM8K table); vLLM PR
15734 runs QK quantization in the attention loop.  The oracle quantizes q
with the pinned E4M3 quantizer and scores with the dequantized query.  The
pins: a query already on the scaled grid is unchanged (so FP8-query
attention equals exact attention), per-head scales act per query head, and
an off-grid query moves the scores by at most the E4M3 half step."""
import numpy as np

from quantized_kv_cache_05_gb300 import synth

RNG = np.random.default_rng(11)


def test_grid_query_round_trips(orc):
    codes = RNG.integers(0, 256, size=(2, 4, 32)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x7E
    codes[:, :, 0] = 0x7E                      # 448 in every head: scale = s exactly
    s = 2.0 ** -5
    q = synth.f32_to_bf16((orc.e4m3_decode(codes) * s).astype(np.float32))
    assert orc.fp8_tensor_scale(orc.amax_bf16(q)) == s
    c, deq = orc.fp8_query(q, s)
    assert np.array_equal(c, codes)
    assert np.array_equal(deq, synth.bf16_to_f32(q).astype(np.float64))


def test_per_head_query_scales(orc):
    """Heads 0..3 on grids scaled by 1, 2^-8, 4, 2^-3: per-head scales keep
    every code; the per-tensor scale (4) flushes head 1 to the subnormal end."""
    hs = np.array([1.0, 2.0 ** -8, 4.0, 2.0 ** -3], np.float32)
    codes = RNG.integers(0x08, 0x7F, size=(3, 4, 16)).astype(np.uint8)   # normal codes
    codes[0, :, 0] = 0x7E
    q = synth.f32_to_bf16((orc.e4m3_decode(codes) * hs[None, :, None]).astype(np.float32))
    assert np.array_equal(orc.fp8_head_scales(np.ascontiguousarray(q)), hs)
    c, deq = orc.fp8_query(q, hs)
    assert np.array_equal(c, codes)
    ct, _ = orc.fp8_query(q, 4.0)
    assert np.array_equal(ct[:, 2], codes[:, 2])
    assert np.mean(ct[:, 1] != codes[:, 1]) > 0.9


def test_fp8_query_attention_error_bound(orc):
    """Scores from the dequantized query differ from exact scores by at most
    sm_scale * sum_d |q_d - q^_d| |k_d|, with |q - q^| within half an E4M3
    step (relative 2^-4 for normal values)."""
    D, L = 64, 50
    q = synth.f32_to_bf16(RNG.standard_normal((1, 1, D)).astype(np.float32))
    k = RNG.standard_normal((L, D))
    v = RNG.standard_normal((L, D))
    s = orc.fp8_tensor_scale(orc.amax_bf16(q))
    _, qh = orc.fp8_query(q, s)
    qf = synth.bf16_to_f32(q).astype(np.float64)[0, 0]
    err = np.abs(qf - qh[0, 0])
    assert np.all(err <= np.maximum(np.abs(qf) * 2.0 ** -4, 2.0 ** -10 * s) + 1e-30)
    sm = 1.0 / np.sqrt(D)
    _, l_exact = orc.attention_exact(qf, k, v, sm)
    _, l_q = orc.attention_exact(qh[0, 0], k, v, sm)
    bound = sm * (err @ np.abs(k).max(axis=0))
    assert abs(l_exact - l_q) <= bound + 1e-12
