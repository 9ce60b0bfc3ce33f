"""Pins of the oracle's per-kv-head ("attn_head") scales.

compressed-tensors PR 436 adds the "attn_head" strategy (one static scale per
attention head, minmax observer) next to the per-tensor one, and its GSM8K
table has a KV-FP8-Head row.  For the KV cache the head is the kv head: head
h's scale is the per-tensor formula on head h's own amax, and each element is
quantized with its head's scale.  The pins below do not re-run the oracle's
arithmetic: they build inputs whose codes are known by construction (grid
values times power-of-two scales), check the head amax against a numpy
reduction, and show the per-head and per-tensor codes differ where they must.
A transposed head index, a scale applied to the wrong head or a per-tensor
amax would fail them."""
import numpy as np
import pytest

from quantized_kv_cache_05_gb300 import synth

RNG = np.random.default_rng(3)


def bf16(x):
    out = synth.f32_to_bf16(np.asarray(x, np.float32))
    assert np.array_equal(synth.bf16_to_f32(out), np.asarray(x, np.float32)), "not exact in bf16"
    return out


def test_head_amax_is_the_per_head_max(orc):
    x = RNG.standard_normal((37, 5, 64)).astype(np.float32)
    x[:, 3] *= 100.0
    x[11, 1, 7] = -9.5                    # a negative extreme in head 1
    xb = synth.f32_to_bf16(x)
    want = np.max(np.abs(synth.bf16_to_f32(xb)), axis=(0, 2))
    assert np.array_equal(orc.head_amax_bf16(xb), want)


@pytest.fixture(scope="module")
def grid_heads(orc):
    """Three kv heads of E4M3 grid values times power-of-two scales s_h =
    1, 2^-6, 8; each head holds its largest value 448 s_h, so its scale is
    s_h exactly."""
    scales = np.array([1.0, 2.0 ** -6, 8.0], np.float32)
    codes = RNG.integers(0, 256, size=(40, 3, 32)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x7E            # no NaN codes
    codes[0, :, 0] = 0x7E                           # +448 in every head
    vals = orc.e4m3_decode(codes) * scales[None, :, None]
    return bf16(vals), codes, scales


def test_fp8_head_scales_and_codes_by_construction(orc, grid_heads):
    x, codes, scales = grid_heads
    s = orc.fp8_head_scales(x)
    assert np.array_equal(s, scales)
    assert np.array_equal(orc.fp8_quantize_heads(x, s), codes)


def test_fp8_per_head_differs_from_per_tensor(orc, grid_heads):
    x, codes, scales = grid_heads
    st = orc.fp8_tensor_scale(orc.amax_bf16(x))     # 448 * 8 / 448 = 8
    assert st == 8.0
    per_tensor = orc.fp8_quantize(x, st)
    # head 2 has the tensor's scale: same codes; head 1 (64x smaller) loses
    # its codes to the subnormal end of the grid
    assert np.array_equal(per_tensor[:, 2], codes[:, 2])
    assert np.mean(per_tensor[:, 1] != codes[:, 1]) > 0.5
    # and per-head quantization with one common scale is per-tensor quantization
    assert np.array_equal(orc.fp8_quantize_heads(x, np.full(3, st, np.float32)), per_tensor)


def test_fp8_heads_index_order(orc, grid_heads):
    """Scales given in another head order give other codes: the scale of
    head h applies to head h."""
    x, codes, scales = grid_heads
    wrong = orc.fp8_quantize_heads(x, scales[::-1].copy())
    assert not np.array_equal(wrong[:, 0], codes[:, 0])
    assert np.array_equal(wrong[:, 1], codes[:, 1])   # the middle head keeps its scale


def test_nvfp4_heads_by_construction(orc):
    """NVFP4 blocks of E2M1 values times an E4M3 block scale times the head's
    global scale g_h (powers of two); every block holds its 6 (so bamax / 6 =
    dsc g_h) and head h holds 6 * 448 * g_h (so amax_h / 2688 = g_h)."""
    gs = np.array([2.0 ** -4, 1.0, 2.0 ** 5], np.float32)
    rows, H, D = 24, 3, 64
    e2m1 = RNG.integers(0, 16, size=(rows, H, D)).astype(np.uint8)
    e2m1[..., ::16] = 0x7                         # +6 in every block
    sc = RNG.integers(0x08, 0x7F, size=(rows, H, D // 16)).astype(np.uint8)   # normal scales
    sc[0, :, 0] = 0x7E                            # 448 in every head
    dsc = orc.e4m3_decode(sc)
    vals = orc.e2m1_decode(e2m1) * np.repeat(dsc, 16, axis=2) * gs[None, :, None]
    x = bf16(vals)
    g = orc.nvfp4_head_scales(x)
    assert np.array_equal(g, gs)
    codes, bscales = orc.nvfp4_quantize_heads(x, g)
    assert np.array_equal(bscales, sc)
    want = (e2m1[..., 0::2] | (e2m1[..., 1::2] << 4)).astype(np.uint8)
    assert np.array_equal(codes, want)
    # the per-tensor global scale (2688 * 32 / 2688 = 32) changes the small
    # heads' block scales
    gt = orc.nvfp4_global_scale(orc.amax_bf16(x))
    assert gt == 32.0
    _, bs_t = orc.nvfp4_quantize(x, gt)
    assert np.array_equal(bs_t[:, 2], sc[:, 2])
    assert not np.array_equal(bs_t[:, 0], sc[:, 0])


def test_per_head_error_is_smaller_on_skewed_heads(orc):
    """With kv heads of very different ranges, a head far below the tensor's
    range falls into the subnormal end of the per-tensor grid, while its own
    scale keeps E4M3's relative precision; the largest head has the tensor's
    scale either way."""
    x = RNG.standard_normal((64, 4, 64)).astype(np.float32)
    x *= np.array([1.0, 1e-3, 30.0, 0.05], np.float32)[None, :, None]
    xb = synth.f32_to_bf16(x)
    xf = synth.bf16_to_f32(xb).astype(np.float64)
    s_h = orc.fp8_head_scales(xb)
    s_t = orc.fp8_tensor_scale(orc.amax_bf16(xb))
    err_h = np.abs(orc.e4m3_decode(orc.fp8_quantize_heads(xb, s_h)) * s_h[None, :, None] - xf)
    err_t = np.abs(orc.e4m3_decode(orc.fp8_quantize(xb, s_t)) * s_t - xf)
    assert err_h[:, 1].mean() < 0.3 * err_t[:, 1].mean()
    assert np.array_equal(err_h[:, 2], err_t[:, 2])
