"""Pins of the oracle's static scales and quantizers (FP8 per tensor, NVFP4).

Closed forms: tensors built on the code grid times a power-of-two scale must
reproduce their codes exactly; NVFP4 blocks built as e2m1 * dsc * g with one
element at +-6 must reproduce codes and block scale; an all-zero block gives
zero codes; the element at the tensor amax always lands on block scale 448 and
element code 6 (checked on the amax values printed on the Model-Optimizer PR
714 page).
"""
import numpy as np
import pytest

from conftest import read_golden
from quantized_kv_cache_05_gb300 import synth

E2M1_POS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def bf16(x):
    return synth.f32_to_bf16(np.asarray(x, np.float32))


def test_scale_formulas(orc):
    assert orc.fp8_tensor_scale(448.0) == 1.0
    assert orc.fp8_tensor_scale(896.0) == 2.0
    assert orc.fp8_tensor_scale(0.0) == 1.0
    assert orc.fp8_tensor_scale(7.53125) == float(np.float32(7.53125) / np.float32(448))
    assert orc.nvfp4_global_scale(2688.0) == 1.0
    assert orc.nvfp4_global_scale(0.0) == 1.0
    assert orc.nvfp4_global_scale(7.53125) == float(np.float32(7.53125) / np.float32(2688))


def test_amax(orc):
    x = bf16([0.5, -3.0, 2.0, -0.0])
    assert orc.amax_bf16(x) == 3.0


def test_fp8_grid_roundtrip(orc):
    # every finite code value times a power-of-two scale quantizes back to it
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = orc.e4m3_decode(codes)
    for scale in [1.0, 0.25, 2.0 ** -6, 8.0]:
        x = bf16(vals * scale)
        assert np.array_equal(synth.bf16_to_f32(x), (vals * scale).astype(np.float32))
        got = orc.fp8_quantize(x, scale)
        # -0.0 and +0.0 keep their sign
        assert np.array_equal(got, codes), scale
        back = orc.fp8_dequant(got, scale)
        assert np.array_equal(back, vals * scale)


def test_fp8_divides_not_multiplies(orc):
    # x / scale and x * (1/scale) differ for scale = 3/448 at some x; the
    # oracle must follow the division.  Find such an x and check the code.
    scale = float(np.float32(3.0) / np.float32(448.0))
    inv = np.float32(1.0) / np.float32(scale)
    xs = synth.bf16_to_f32(np.arange(0x3C00, 0x4300, dtype=np.uint16))
    div = (xs / np.float32(scale)).astype(np.float32)
    mul = (xs * inv).astype(np.float32)
    diff = np.nonzero(div != mul)[0]
    assert diff.size > 0
    for i in diff[:50]:
        code = orc.fp8_quantize(synth.f32_to_bf16(xs[i:i + 1]), scale)[0]
        assert code == orc.e4m3_encode(div[i:i + 1])[0]


def test_fp8_saturates(orc):
    x = bf16([1000.0, -1000.0, 448.0])
    assert list(orc.fp8_quantize(x, 1.0)) == [0x7E, 0xFE, 0x7E]


def nvfp4_block(e2m1_vals, dsc, g):
    return bf16(np.array(e2m1_vals, np.float64) * dsc * g)


@pytest.mark.parametrize("dsc_code", [0x01, 0x08, 0x30, 0x38, 0x55, 0x7E])
@pytest.mark.parametrize("g", [1.0, 2.0 ** -4, 2.0 ** 3])
def test_nvfp4_closed_form_block(orc, dsc_code, g):
    rng = np.random.default_rng(dsc_code)
    dsc = float(orc.e4m3_decode(np.array([dsc_code], np.uint8))[0])
    nibs = rng.integers(0, 16, size=16).astype(np.uint8)
    nibs[rng.integers(0, 16)] = 0x7 if rng.random() < 0.5 else 0xF   # one element at +-6
    vals = orc.e2m1_decode(nibs)
    x = nvfp4_block(vals, dsc, g)
    assert np.array_equal(synth.bf16_to_f32(x).astype(np.float64), vals * dsc * g)
    codes, sc = orc.nvfp4_quantize(x.reshape(1, 16), g)
    assert sc[0, 0] == dsc_code
    got = np.empty(16, np.uint8)
    got[0::2] = codes[0] & 0xF
    got[1::2] = codes[0] >> 4
    # +0 and -0 are both zero values; keep the sign the input had
    assert np.array_equal(got, nibs)
    back = orc.nvfp4_dequant(codes, sc, g)
    assert np.array_equal(back[0], vals * dsc * g)


def test_nvfp4_zero_block(orc):
    x = np.zeros((2, 32), np.uint16)
    x[1, 16:] = bf16(np.linspace(-1, 1, 16))
    codes, sc = orc.nvfp4_quantize(x, 0.5)
    assert np.all(codes[0] == 0) and np.all(sc[0] == 0)
    assert np.all(codes[1, :8] == 0) and sc[1, 0] == 0
    assert sc[1, 1] != 0


def test_nvfp4_underflowed_block_scale_gives_zero_codes(orc):
    # bamax/6/g below half the smallest E4M3 subnormal rounds the block scale
    # to 0; every element code is then 0.
    g = 1.0
    x = bf16(np.full(16, 2.0 ** -14))
    codes, sc = orc.nvfp4_quantize(x.reshape(1, 16), g)
    assert sc[0, 0] == 0 and np.all(codes == 0)


def test_nvfp4_element_scale_uses_quantized_block_scale(orc):
    """Elements divide by the quantized block scale, not by bamax/6/g.

    Block amax 5, g = 1: 5/6 = 0.8333 rounds to the E4M3 value 0.8125 (code
    0x35).  The element 0.205078125 (bf16 of 0.205) divided by 0.8125 is
    0.2524 -> E2M1 0.5 (code 1); divided by the unquantized 0.8333 it would
    be 0.2461 -> 0 (code 0).  The amax element 5 / 0.8125 = 6.15 saturates to
    6 (code 7)."""
    vals = np.zeros(16, np.float32)
    vals[0] = 5.0
    vals[1] = 0.205
    x = bf16(vals).reshape(1, 16)
    codes, sc = orc.nvfp4_quantize(x, 1.0)
    assert sc[0, 0] == 0x35
    assert orc.e4m3_decode(sc[0])[0] == 0.8125
    assert codes[0, 0] & 0xF == 0x7
    assert codes[0, 0] >> 4 == 0x1


@pytest.mark.parametrize("row", read_golden("mo714_amax.txt"), ids=lambda r: r[0])
def test_tensor_amax_element_maps_to_top_codes(orc, row):
    """The element equal to the tensor amax gets block scale 448 (0x7E) and
    element code +-6, for the calibrated amax values the page prints."""
    amax = float(np.float32(synth.bf16_to_f32(bf16([float(row[1])]))[0]))
    g = orc.nvfp4_global_scale(amax)
    blk = np.zeros(16, np.float32)
    blk[3] = amax
    blk[7] = -amax / 2
    codes, sc = orc.nvfp4_quantize(bf16(blk).reshape(1, 16), g)
    assert sc[0, 0] == 0x7E
    assert codes[0, 1] >> 4 == 0x7            # element 3 -> high nibble of byte 1
    # element 7 = -amax/2 -> -amax/2 / (448 g) = -3 up to fp32 rounding -> 0xD
    assert codes[0, 3] >> 4 == 0xD


def test_nvfp4_dequant_layout(orc):
    codes = np.array([[0x21] + [0] * 7], np.uint8)   # element 0 -> 0.5, element 1 -> 1.0
    sc = np.array([[0x38]], np.uint8)                # block scale 1.0
    out = orc.nvfp4_dequant(codes, sc, 2.0)
    assert out[0, 0] == 1.0 and out[0, 1] == 2.0 and np.all(out[0, 2:] == 0)
