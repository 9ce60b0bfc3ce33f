"""GPU quantize-on-append and encoders vs the oracle: bit-exact codes and
block scales, exhaustive over all 2^32 fp32 patterns for the encoders."""
import numpy as np
import pytest
import torch

import oracle
from kvq_testlib import Setup, to_dev_bf16
from quantized_kv_cache_05_gb300 import build as kbuild
from quantized_kv_cache_05_gb300 import kvq, runtime, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kvq.lib()
    torch.cuda.init()


@pytest.mark.parametrize("kind", [0, 1], ids=["e4m3", "e2m1"])
def test_device_encoder_exhaustive(kind):
    chunk = 1 << 28
    out = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    enc = kvq.kvq_encode_e4m3 if kind == 0 else kvq.kvq_encode_e2m1
    total = 0
    for start in range(0, 1 << 32, chunk):
        v = torch.arange(start, start + chunk, dtype=torch.int64, device="cuda")
        v = torch.where(v >= (1 << 31), v - (1 << 32), v).to(torch.int32)
        x = v.view(torch.float32)
        kvq.check(enc(x, out, chunk))
        torch.cuda.synchronize()
        bad, first = oracle.count_encode_mismatch(kind, start, out.cpu().numpy())
        assert bad == 0, f"{bad} mismatches in chunk {start:#x}, first {first:#010x}"
        total += chunk
        del v, x
    assert total == 1 << 32


def check_codes(S: Setup):
    w = S.w
    assert S.gpu_amax_k == oracle.amax_bf16(np.concatenate([x.reshape(-1) for x in S.k]))
    assert S.gpu_k_scale == S.k_scale and S.gpu_v_scale == S.v_scale
    for b in range(w.B):
        if int(w.seq_lens[b]) == 0:
            continue
        for h in range(w.Hkv):
            for which in (["k"] if w.mla else ["k", "v"]):
                codes, bs = S.oracle_codes(which, b, h)
                assert np.array_equal(S.gpu_rows(which, b, h), codes), (which, b, h)
                if bs is not None:
                    assert np.array_equal(S.gpu_rows(which + "s", b, h), bs), (which, b, h)
        if w.mla:
            assert np.array_equal(S.gpu_rows("kpe", b), S.kpe[b])


def test_append_fp8_tiny():
    check_codes(Setup(synth.tiny_fp8()))


def test_append_fp8_gqa_outliers():
    w = synth.gqa_fp8(1000)
    check_codes(Setup(w))


def test_append_fp8_paged_ragged():
    w = synth.paged_fp8_probs(B=5, lo=1, hi=300, seed=3)
    check_codes(Setup(w))


def test_append_nvfp4():
    check_codes(Setup(synth.nvfp4(1000)))


def test_append_nvfp4_mla_latent():
    check_codes(Setup(synth.mla_nvfp4(B=2, L=100)))


def _tiny_cache(fmt, D, g):
    bt = torch.zeros((1, 1), dtype=torch.int32)
    return runtime.QuantizedKVCache(fmt, 1, 16, 1, D, bt, g, g)


def test_nvfp4_corner_blocks():
    """Zero block, single non-zero, saturated block scale, underflowed block
    scale, +-6 saturation and signed zeros, against the oracle."""
    D, g = 128, 2.0 ** -6
    rows = np.zeros((16, D), np.float32)
    rows[1, 5] = 3.0                                # one non-zero in a block
    rows[2, :16] = 1e4                              # bamax/6/g >> 448: scale saturates
    rows[2, 16:32] = np.linspace(-1e4, 1e4, 16)
    rows[3, :16] = 2.0 ** -20                       # scale underflows to 0
    rows[4, :] = -1e-30                             # negative tiny values
    rows[5, :] = np.linspace(-7.0, 7.0, D) * g * 448
    rng = np.random.default_rng(0)
    rows[6:] = rng.standard_normal((10, D)) * rng.choice([1e-3, 1.0, 30.0], (10, 1))
    x = synth.f32_to_bf16(rows)
    c = _tiny_cache("nvfp4", D, g)
    kvq.check(kvq.kvq_quantize_append(c.struct(), to_dev_bf16(x[None, :, None, :]),
                                      to_dev_bf16(x[None, :, None, :]), None,
                                      torch.zeros(1, dtype=torch.int32, device="cuda"), 1, 16))
    codes, bs = oracle.nvfp4_quantize(x, g)
    assert np.array_equal(c.k_codes.cpu().numpy()[0, 0], codes)
    assert np.array_equal(c.k_bscale.cpu().numpy()[0, 0], bs)
    assert np.array_equal(c.v_codes.cpu().numpy()[0, 0], codes)
    assert bs[2, 0] == 0x7E and bs[3, 0] == 0x00


def test_fp8_saturation_and_zero_signs():
    D, s = 64, 0.5
    rows = np.zeros((16, D), np.float32)
    rows[0] = np.linspace(-1000, 1000, D)
    rows[1] = -1e-30
    rows[2, ::2] = -0.0
    rng = np.random.default_rng(1)
    rows[3:] = rng.standard_normal((13, D)) * 100
    x = synth.f32_to_bf16(rows)
    c = _tiny_cache("fp8", D, s)
    kvq.check(kvq.kvq_quantize_append(c.struct(), to_dev_bf16(x[None, :, None, :]),
                                      to_dev_bf16(x[None, :, None, :]), None,
                                      torch.zeros(1, dtype=torch.int32, device="cuda"), 1, 16))
    assert np.array_equal(c.k_codes.cpu().numpy()[0, 0], oracle.fp8_quantize(x, s))


def test_append_at_offsets_and_out_of_table():
    """start_pos offsets land in the right page rows; positions beyond the
    block table are skipped."""
    D, s = 128, 0.25
    bt = torch.tensor([[2, 0], [1, 3]], dtype=torch.int32)
    c = runtime.QuantizedKVCache("fp8", 4, 16, 1, D, bt, s, s)
    x = synth.fill_bf16(7, 1, 2 * 3 * D).reshape(2, 3, 1, D)
    start = torch.tensor([14, 30], dtype=torch.int32, device="cuda")   # 30, 31, 32(skipped)
    kvq.check(kvq.kvq_quantize_append(c.struct(), to_dev_bf16(x), to_dev_bf16(x), None, start, 2, 3))
    kc = c.k_codes.cpu().numpy()
    want = oracle.fp8_quantize(x, s)
    # request 0: positions 14, 15 -> page 2 rows 14, 15; 16 -> page 0 row 0
    assert np.array_equal(kc[2, 0, 14], want[0, 0, 0]) and np.array_equal(kc[2, 0, 15], want[0, 1, 0])
    assert np.array_equal(kc[0, 0, 0], want[0, 2, 0])
    # request 1: positions 30, 31 -> page 3 rows 14, 15; position 32 is outside the table
    assert np.array_equal(kc[3, 0, 14], want[1, 0, 0]) and np.array_equal(kc[3, 0, 15], want[1, 1, 0])
    touched = {(2, 14), (2, 15), (0, 0), (3, 14), (3, 15)}
    for p in range(4):
        for r in range(16):
            if (p, r) not in touched:
                assert not kc[p, 0, r].any()


def test_amax_kernel_unaligned_and_tail():
    x = synth.fill_bf16(5, 2, 10_001)
    t = to_dev_bf16(x)
    out = torch.empty(1, dtype=torch.float32, device="cuda")
    for off in (0, 1, 3):
        kvq.check(kvq.kvq_amax_bf16(t[off:], t.numel() - off, out))
        assert float(out.item()) == oracle.amax_bf16(x[off:])
    kvq.check(kvq.kvq_amax_bf16(t, 0, out))
    assert float(out.item()) == 0.0
