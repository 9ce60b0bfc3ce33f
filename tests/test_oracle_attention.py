"""Pins of the oracle's attention, split partials, combine and FP8 paths.

Closed forms (constant keys give mean(V); one key gives that value; two keys
with a score gap of ln 3 give weights 3/4 and 1/4; a dominant key gives its
value), split invariance of partial + combine in fp64, brute force on tiny
inputs against an independently written formula (math.fsum softmax), the
chunk rule on hand-worked cases, the GQA head mapping, and the FP8-probability
reading on a hand-computed case.
"""
import math

import numpy as np
import pytest


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_constant_keys_give_mean_v(orc):
    L, D = 37, 16
    q = rnd(D, 1)
    k = np.tile(rnd(D, 2), (L, 1))
    v = rnd((L, D), 3)
    out, lse = orc.attention_exact(q, k, v, 0.25)
    assert np.allclose(out, v.mean(axis=0), rtol=0, atol=1e-14)
    s = 0.25 * float(q @ k[0])
    assert math.isclose(lse, s + math.log(L), rel_tol=0, abs_tol=1e-12)


def test_single_key_gives_its_value(orc):
    q, k, v = rnd(8, 1), rnd((1, 8), 2), rnd((1, 8), 3)
    out, lse = orc.attention_exact(q, k, v, 1.0)
    assert np.array_equal(out, v[0])
    assert math.isclose(lse, float(q @ k[0]), abs_tol=1e-14)


def test_two_keys_ln3_gap(orc):
    # q.k0 - q.k1 = ln 3 -> weights 3/4, 1/4
    q = np.array([1.0, 0.0])
    k = np.array([[math.log(3.0), 0.0], [0.0, 5.0]])
    v = np.array([[4.0, 0.0], [0.0, 8.0]])
    out, _ = orc.attention_exact(q, k, v, 1.0)
    assert np.allclose(out, [3.0, 2.0], atol=1e-14)


def test_dominant_key(orc):
    D, L = 16, 50
    q = np.zeros(D)
    q[3] = 1.0
    k = rnd((L, D), 4) * 0.01
    k[17, 3] = 1000.0
    v = rnd((L, D), 5)
    out, _ = orc.attention_exact(q, k, v, 1.0)
    assert np.allclose(out, v[17], atol=1e-12)


def test_empty_sequence(orc):
    out, lse = orc.attention_exact(np.ones(4), np.zeros((0, 4)), np.zeros((0, 4)), 1.0)
    assert lse == -math.inf and np.all(out == 0)


def brute(q, k, v, sm):
    """Independent direct formula: softmax with a log-sum-exp normalizer."""
    S = [sm * math.fsum(a * b for a, b in zip(q, row)) for row in k]
    m = max(S)
    lse = m + math.log(math.fsum(math.exp(s - m) for s in S))
    w = [math.exp(s - lse) for s in S]
    out = [math.fsum(w[i] * v[i][d] for i in range(len(S))) for d in range(len(v[0]))]
    return np.array(out), lse


@pytest.mark.parametrize("L", [1, 2, 3, 4])
@pytest.mark.parametrize("seed", range(5))
def test_bruteforce_tiny(orc, L, seed):
    D = 16
    q, k, v = rnd(D, seed), rnd((L, D), seed + 100) * 3, rnd((L, D), seed + 200)
    sm = 0.3
    out, lse = orc.attention_exact(q, k, v, sm)
    bo, bl = brute(q.tolist(), k.tolist(), v.tolist(), sm)
    assert np.allclose(out, bo, rtol=0, atol=1e-13)
    assert math.isclose(lse, bl, abs_tol=1e-13)


def test_chunk_rule(orc):
    # c = ceil(L/s) rounded up to 16; chunk j = [j c, min((j+1) c, L))
    assert [orc.chunk(256, 2, j) for j in range(2)] == [(0, 128), (128, 256)]
    assert [orc.chunk(100, 8, j) for j in range(8)] == [
        (0, 16), (16, 32), (32, 48), (48, 64), (64, 80), (80, 96), (96, 100), (100, 100)]
    assert [orc.chunk(1000, 3, j) for j in range(3)] == [(0, 336), (336, 672), (672, 1000)]
    assert orc.chunk(0, 4, 0) == (0, 0)
    assert orc.chunk(5, 4, 1) == (5, 5)


@pytest.mark.parametrize("s", range(1, 9))
def test_split_invariance(orc, s):
    L, D, Dv = 300, 32, 24
    q, k, v = rnd(D, 7), rnd((L, D), 8), rnd((L, Dv), 9)
    exact, lse = orc.attention_exact(q, k, v, 0.5)
    parts, lses = [], []
    for j in range(s):
        st, en = orc.chunk(L, s, j)
        o, l = orc.attention_partial(q, k, v, st, en, 0.5)
        parts.append(o)
        lses.append(l)
    got = orc.combine(np.array(parts), np.array(lses))
    assert np.allclose(got, exact, rtol=0, atol=1e-12)
    finite = [l for l in lses if l != -math.inf]
    m = max(finite)
    assert math.isclose(m + math.log(sum(math.exp(l - m) for l in finite)), lse,
                        abs_tol=1e-12)


def test_combine_skips_empty(orc):
    o = np.array([[1.0, 2.0], [0.0, 0.0], [3.0, 4.0]])
    lse = np.array([0.0, -math.inf, math.log(3.0)])
    assert np.allclose(orc.combine(o, lse), [2.5, 3.5], atol=1e-15)
    assert np.all(orc.combine(o, np.full(3, -math.inf)) == 0)


def test_gqa_head_mapping(orc):
    # query head hq reads kv head hq // G
    B, Hq, Hkv, L, D = 1, 6, 3, 20, 8
    q = rnd((B, Hq, D), 10)
    k = rnd((B, Hkv, L, D), 11)
    v = rnd((B, Hkv, L, D), 12)
    out, lse = orc.decode_batch(q, k, v, np.array([L]), 0.4)
    for hq in range(Hq):
        want, wl = orc.attention_exact(q[0, hq], k[0, hq // 2], v[0, hq // 2], 0.4)
        assert np.allclose(out[0, hq], want, atol=1e-14)
        other, _ = orc.attention_exact(q[0, hq], k[0, (hq // 2 + 1) % 3], v[0, (hq // 2 + 1) % 3],
                                       0.4)
        assert not np.allclose(out[0, hq], other, atol=1e-3)


def test_decode_batch_ragged(orc):
    B, H, Lc, D = 3, 2, 40, 8
    q = rnd((B, H, D), 13)
    k = rnd((B, H, Lc, D), 14)
    v = rnd((B, H, Lc, D), 15)
    lens = np.array([40, 1, 0])
    out, lse = orc.decode_batch(q, k, v, lens, 0.5)
    for b in range(B):
        for h in range(H):
            want, wl = orc.attention_exact(q[b, h], k[b, h, :lens[b]], v[b, h, :lens[b]], 0.5)
            assert np.allclose(out[b, h], want, atol=1e-14)
    assert np.all(out[2] == 0) and np.all(lse[2] == -math.inf)


# --------------------------------------------------------------------------
# FP8 probabilities (vLLM PR 15734: softmax(QK^T) quantized to FP8 with a
# prob scale) -- reading: p~ = exp(S - chunk max) in fp32, p_q =
# dec(E4M3(p~ / prob_scale)) * prob_scale multiplies V, the denominator sums p~.
# --------------------------------------------------------------------------

PS = float(np.float32(1.0) / np.float32(448.0))


def test_probq_constant_keys_mean(orc):
    L, D = 50, 16
    q = rnd(D, 20)
    k = np.tile(rnd(D, 21), (L, 1))
    v = rnd((L, D), 22)
    o, lse = orc.attention_partial_probq(q, k, v, 0, L, 0.3, PS)
    # p~ = 1 -> 1/PS = 448 exactly in fp32 -> code 0x7E -> p_q = 448 * PS
    pq = 448.0 * PS
    assert np.allclose(o, pq * v.mean(axis=0), atol=1e-13)


def test_probq_hand_case(orc):
    # two keys; score gap g with exp(-g) = 0.3: p~1 = fl32(0.3...) -> *448 =
    # 134.4 -> E4M3 128 -> p_q = 128 * PS; denominator uses p~
    g = -math.log(0.3)
    q = np.array([1.0])
    k = np.array([[g], [0.0]])
    v = np.array([[1.0, 0.0], [0.0, 1.0]])
    o, lse = orc.attention_partial_probq(q, k, v, 0, 2, 1.0, PS)
    p1 = float(np.float32(math.exp(-g)))
    assert abs(p1 - 0.3) < 1e-7
    want = np.array([448.0 * PS, 128.0 * PS]) / (1.0 + p1)
    assert np.allclose(o, want, atol=1e-14)
    assert math.isclose(lse, g + math.log(1.0 + p1), abs_tol=1e-12)
    # the unquantized answer differs visibly
    assert abs(o[1] - p1 / (1 + p1)) > 0.01


def test_probq_batch_uses_chunks(orc):
    B, H, L, D = 1, 1, 64, 8
    q = rnd((B, H, D), 30)
    k = rnd((B, H, L, D), 31)
    v = rnd((B, H, L, D), 32)
    for s in (1, 2, 4):
        out, lse = orc.decode_batch(q, k, v, np.array([L]), 0.5, mode=1, s=s, prob_scale=PS)
        parts, lses = [], []
        for j in range(s):
            st, en = orc.chunk(L, s, j)
            o, l = orc.attention_partial_probq(q[0, 0], k[0, 0], v[0, 0], st, en, 0.5, PS)
            parts.append(o)
            lses.append(l)
        assert np.allclose(out[0, 0], orc.combine(np.array(parts), np.array(lses)), atol=1e-14)
    exact, _ = orc.attention_exact(q[0, 0], k[0, 0], v[0, 0], 0.5)
    assert np.allclose(out[0, 0], exact, atol=0.1)     # same answer up to FP8 weights


@pytest.mark.parametrize("s", [1, 2, 3, 5])
def test_probq_powers_of_two_are_lossless(orc, s):
    """Weights 2^-n (0 <= n <= 14 below each chunk's max) quantize without
    loss: p~ / prob_scale = 1.75 * 2^(8 - n) is an E4M3 value, so the FP8
    probability mode equals exact attention up to the fp32 rounding of
    prob_scale itself (relative ~3e-8), for any split count.  A dropped or
    doubled prob_scale, a wrong chunk max or a broken chunk merge fails."""
    L, Dv = 40, 6
    rng = np.random.default_rng(41)
    n = rng.integers(0, 12, L)
    n[rng.integers(0, L)] = 0
    q = np.array([[[1.0]]])
    k = (-(n.astype(np.float64)) * math.log(2.0)).reshape(1, 1, L, 1)
    v = rng.standard_normal((1, 1, L, Dv))
    out, _ = orc.decode_batch(q, k, v, np.array([L]), 1.0, mode=1, s=s, prob_scale=PS)
    exact, _ = orc.attention_exact(q[0, 0], k[0, 0], v[0, 0], 1.0)
    w = np.exp2(-n.astype(np.float64))
    closed = (w[:, None] * v[0, 0]).sum(axis=0) / w.sum()
    assert np.allclose(exact, closed, rtol=0, atol=1e-12)
    assert np.allclose(out[0, 0], closed, rtol=0, atol=1e-7 * np.abs(v).max())


def test_fp8_output(orc):
    o = np.array([1.0, -2.0, 500.0, 0.0])
    assert list(orc.fp8_output(o, 1.0)) == [0x38, 0xC0, 0x7E, 0x00]
    assert list(orc.fp8_output(o, 0.5)) == [0x40, 0xC8, 0x7E, 0x00]
