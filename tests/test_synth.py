"""The seeded input generator: determinism, slice consistency, recipe shape."""
import numpy as np

from quantized_kv_cache_05_gb300 import synth


def test_deterministic_and_sliceable():
    a = synth.fill_bf16(0, synth.T_K, 300_000)
    b = synth.fill_bf16(0, synth.T_K, 300_000)
    assert np.array_equal(a, b)
    c = synth.fill_bf16(0, synth.T_K, 1000, offset=123_456)
    assert np.array_equal(a[123_456:124_456], c)
    d = synth.fill_bf16(1, synth.T_K, 1000)
    assert not np.array_equal(a[:1000], d)
    e = synth.fill_bf16(0, synth.T_V, 1000)
    assert not np.array_equal(a[:1000], e)


def test_normal_statistics():
    x = synth.bf16_to_f32(synth.fill_bf16(3, 0, 1_000_000)).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert np.all(np.isfinite(x))


def test_outliers():
    n = 1_000_000
    base = synth.bf16_to_f32(synth.fill_bf16(0, 1, n))
    out = synth.bf16_to_f32(synth.fill_bf16(0, 1, n, elem_p=0.01, elem_mult=10.0))
    frac = np.mean(out != base)
    assert 0.008 < frac < 0.012
    m = np.zeros(64, np.uint8)
    m[[5, 9]] = 1
    ch = synth.bf16_to_f32(synth.fill_bf16(0, 1, 64 * 1000, D=64, chan_mask=m, chan_mult=20.0))
    ch = ch.reshape(1000, 64)
    assert ch[:, 5].std() > 10 and ch[:, 0].std() < 2


def test_workload_recipes():
    w = synth.tiny_fp8()
    assert (w.B, w.Hq, w.Hkv, w.D, w.Lmax) == (1, 4, 1, 64, 256)
    assert len(synth.pick_channels(0, 64, 2)) == 2
    p = synth.paged_fp8_probs()
    assert p.B == 64 and p.seq_lens.min() >= 512 and p.seq_lens.max() <= 8192
    bt, n = p.block_table()
    used = np.concatenate([bt[b, :-(-int(L) // 16)] for b, L in enumerate(p.seq_lens)])
    assert sorted(used.tolist()) == list(range(n))
    k = w.kv_rows(synth.T_K, 0, 10, 20)
    full = w.full(synth.T_K)
    assert np.array_equal(k, full[0, 10:20])
