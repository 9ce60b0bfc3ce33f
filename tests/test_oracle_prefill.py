"""Pins of the oracle's causal prefill attention.

Model-Optimizer PR 1832 compares split decode with a prefill attention kernel
(its latency tables' prefill column).  The oracle's prefill attention lets
query i of Tq new tokens (at position L - Tq + i of an L-token cache that
holds them) attend to keys [0, L - Tq + i].  Pins: the last query is the
decode attention over the whole cache; a key placed after a query's position
with a huge score leaves that query unchanged but takes over the later ones;
and a closed form (equal keys give the mean of each prefix's values)."""
import numpy as np

RNG = np.random.default_rng(21)


def test_last_query_is_decode(orc):
    L, Tq, D = 40, 6, 16
    q = RNG.standard_normal((Tq, D))
    k = RNG.standard_normal((L, D))
    v = RNG.standard_normal((L, D))
    out, lse = orc.prefill_attention(q, k, v, 0.25)
    o, l = orc.attention_exact(q[-1], k, v, 0.25)
    assert np.allclose(out[-1], o, atol=1e-14) and abs(lse[-1] - l) < 1e-12


def test_causal_mask(orc):
    """Key at position 37 aligned with every query and huge: queries at
    positions < 37 ignore it, queries at >= 37 return its value."""
    L, Tq, D = 40, 6, 16                 # queries at positions 34..39
    q = RNG.standard_normal((Tq, D))
    k = RNG.standard_normal((L, D)) * 0.01
    v = RNG.standard_normal((L, D))
    base, _ = orc.prefill_attention(q, k, v, 1.0)
    k2 = k.copy()
    k2[37] = 1e3 * q.sum(axis=0) / np.linalg.norm(q.sum(axis=0)) ** 2 * 50
    out, _ = orc.prefill_attention(q, k2, v, 1.0)
    for i in range(Tq):
        pos = L - Tq + i
        if pos < 37:
            assert np.array_equal(out[i], base[i]), i
        else:
            assert np.allclose(out[i], v[37], atol=1e-9), i


def test_equal_keys_give_prefix_means(orc):
    L, Tq, D = 30, 5, 8
    q = RNG.standard_normal((Tq, D))
    k = np.tile(RNG.standard_normal((1, D)), (L, 1))
    v = RNG.standard_normal((L, D))
    out, _ = orc.prefill_attention(q, k, v, 0.5)
    for i in range(Tq):
        n = L - Tq + i + 1
        assert np.allclose(out[i], v[:n].mean(axis=0), atol=1e-13)
