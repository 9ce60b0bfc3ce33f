"""GPU split-KV decode vs the oracle on the same dequantized cache.

Sizes span several pipeline stages and ragged tails; every split count of
the workloads plus uneven ones; partials checked chunk by chunk; edge cases:
empty sequences, one token, fewer tokens than splits, constant keys."""
import numpy as np
import pytest
import torch

import oracle
from kvq_testlib import (Setup, assert_bf16_close, assert_e4m3_close, assert_f32_close,
                         bf16_bits)
from quantized_kv_cache_05_gb300 import build as kbuild
from quantized_kv_cache_05_gb300 import kvq, runtime, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kvq.lib()
    torch.cuda.init()


def splits_of(w, s):
    if s == 0:
        return runtime.auto_splits(w.B, w.Hkv, w.G, w.Lmax, w.fmt)
    return s


@pytest.fixture(scope="module")
def tiny():
    return Setup(synth.tiny_fp8())


@pytest.mark.parametrize("s", [1, 2])
def test_tiny_fp8(tiny, s):
    ref, _ = tiny.oracle_decode()
    out, _ = tiny.gpu_decode(s)
    assert_f32_close(out.cpu().numpy(), ref, f"tiny s={s}")


@pytest.fixture(scope="module")
def gqa():
    return Setup(synth.gqa_fp8(1000))


@pytest.mark.parametrize("s", [1, 2, 3, 4, 8, 0])
def test_gqa_fp8_f32(gqa, s):
    ref, _ = gqa.oracle_decode()
    out, _ = gqa.gpu_decode(splits_of(gqa.w, s))
    assert_f32_close(out.cpu().numpy(), ref, f"gqa s={s}")


@pytest.mark.parametrize("s", [1, 8, 0])
def test_gqa_fp8_bf16_out(gqa, s):
    ref, _ = gqa.oracle_decode()
    out, _ = gqa.gpu_decode(splits_of(gqa.w, s), "bf16")
    assert_bf16_close(bf16_bits(out), ref, f"gqa bf16 s={s}")


def test_gqa_partials_per_chunk(gqa):
    s = 3
    w = gqa.w
    _, ws = gqa.gpu_decode(s)
    po = ws.part_o.cpu().numpy().reshape(w.B, w.Hq, s, w.Dv)
    pl = ws.part_lse.cpu().numpy().reshape(w.B, w.Hq, s)
    q = gqa.q64()
    for b in range(w.B):
        for kvh in (0, w.Hkv - 1):
            kh, vh = gqa.oracle_kv(b, kvh)
            L = int(w.seq_lens[b])
            for j in range(s):
                st, en = oracle.chunk(L, s, j)
                for hq in range(kvh * w.G, (kvh + 1) * w.G):
                    o, l = oracle.attention_partial(q[b, hq], kh, vh, st, en, w.sm_scale)
                    assert abs(pl[b, hq, j] - l) <= 1e-4 * max(1.0, abs(l)), (b, hq, j)
                    assert_f32_close(po[b, hq, j], o, f"partial b{b} h{hq} j{j}")


@pytest.fixture(scope="module")
def nv():
    return Setup(synth.nvfp4(1500))


@pytest.mark.parametrize("s", [1, 4, 7, 0])
def test_nvfp4(nv, s):
    ref, _ = nv.oracle_decode()
    out, _ = nv.gpu_decode(splits_of(nv.w, s))
    assert_f32_close(out.cpu().numpy(), ref, f"nvfp4 s={s}")


@pytest.fixture(scope="module")
def paged():
    return Setup(synth.paged_fp8_probs(B=6, lo=1, hi=700, seed=5))


@pytest.mark.parametrize("s", [1, 2, 5])
def test_paged_fp8_probs_f32(paged, s):
    ref, _ = paged.oracle_decode(mode=1, s=s)
    out, _ = paged.gpu_decode(s)
    assert_f32_close(out.cpu().numpy(), ref, f"paged probs s={s}")


@pytest.mark.parametrize("s", [1, 2])
def test_paged_fp8_probs_e4m3_out(paged, s):
    ref, _ = paged.oracle_decode(mode=1, s=s)
    out_scale = float(np.float32(np.float32(np.max(np.abs(ref))) / np.float32(448.0)))
    out, _ = paged.gpu_decode(s, "e4m3", out_scale)
    flips = assert_e4m3_close(out.cpu().numpy(), ref, out_scale, f"paged e4m3 s={s}")
    assert flips <= max(2, ref.size // 1000)


def test_paged_exact_probabilities_off():
    """The same paged MHA cache without FP8 probabilities matches exact
    attention."""
    w = synth.paged_fp8_probs(B=4, lo=17, hi=400, seed=9)
    w.prob_fp8 = False
    S = Setup(w)
    ref, _ = S.oracle_decode()
    out, _ = S.gpu_decode(2)
    assert_f32_close(out.cpu().numpy(), ref, "paged exact")


@pytest.mark.parametrize("hq,hkv,fmt", [(16, 1, "fp8"), (24, 2, "fp8"), (16, 2, "nvfp4"),
                                         (12, 1, "nvfp4")])
def test_large_groups(hq, hkv, fmt):
    """9..16 query heads per kv head (two head groups of the P.V MMA)."""
    w = synth.gqa_fp8(700) if fmt == "fp8" else synth.nvfp4(700)
    w.B, w.Hq, w.Hkv = 2, hq, hkv
    w.seq_lens = np.array([700, 333], np.int32)
    S = Setup(w)
    ref, _ = S.oracle_decode()
    for s in (1, 3):
        out, _ = S.gpu_decode(s)
        assert_f32_close(out.cpu().numpy(), ref, f"G={hq // hkv} {fmt} s={s}")


def test_large_groups_fp8_probs():
    w = synth.paged_fp8_probs(B=3, lo=40, hi=500, seed=11)
    w.Hq, w.Hkv = 16, 1
    S = Setup(w)
    for s in (1, 2):
        ref, _ = S.oracle_decode(mode=1, s=s)
        out, _ = S.gpu_decode(s)
        assert_f32_close(out.cpu().numpy(), ref, f"G=16 probs s={s}")


@pytest.mark.parametrize("shape", ["gqa4_d128", "gqa4_d64", "nvfp4_d128"])
def test_fp8_probs_shapes(shape):
    """FP8 probabilities beyond MHA: four query heads per kv head at head_dim
    128 and 64 with an FP8 cache, and with an NVFP4 cache; ragged lengths,
    several splits."""
    if shape == "gqa4_d128":
        w = synth.gqa_fp8(700)
        w.B, w.Hq, w.Hkv = 2, 8, 2
        w.seq_lens = np.array([700, 333], np.int32)
    elif shape == "gqa4_d64":
        w = synth.tiny_fp8(300)
        w.B = 3
        w.seq_lens = np.array([300, 77, 16], np.int32)
    else:
        w = synth.nvfp4(500)
        w.B, w.Hq, w.Hkv = 2, 8, 2
        w.seq_lens = np.array([500, 129], np.int32)
    w.prob_fp8 = True
    S = Setup(w)
    for s in (1, 3):
        ref, _ = S.oracle_decode(mode=1, s=s)
        out, _ = S.gpu_decode(s)
        assert_f32_close(out.cpu().numpy(), ref, f"{shape} probs s={s}")


def test_edge_lengths():
    """Lengths 0 (output 0), 1, 15, 16, 17 and fewer tokens than splits."""
    w = synth.gqa_fp8(64)
    w.seq_lens = np.array([0, 1, 15, 16, 17, 40], np.int32)
    w.B = 6
    w.page_size = 16
    S = Setup(w)
    ref, _ = S.oracle_decode()
    for s in (1, 3, 8):
        out, ws = S.gpu_decode(s)
        o = out.cpu().numpy()
        assert np.all(o[0] == 0)
        assert_f32_close(o, ref, f"edge s={s}")
        lse = ws.part_lse.cpu().numpy().reshape(w.B, w.Hq, s)
        assert np.all(np.isneginf(lse[0]))


def test_constant_keys_mean_values():
    """All keys equal: the output is the mean of the dequantized values."""
    w = synth.gqa_fp8(300)
    w.B = 1
    w.seq_lens = np.array([300], np.int32)
    S = Setup.__new__(Setup)
    Setup.__init__(S, w)
    # overwrite the cache's K codes with one row repeated
    kc = S.cache.k_codes
    kc[:] = kc[:, :, :1, :].clone() if kc.shape[2] > 0 else kc
    torch.cuda.synchronize()
    out, _ = S.gpu_decode(2)
    o = out.cpu().numpy()[0]
    for kvh in range(w.Hkv):
        vh = S.oracle_dequant("v", 0, kvh)
        mean = vh.mean(axis=0)
        for hq in range(kvh * w.G, (kvh + 1) * w.G):
            assert np.max(np.abs(o[hq] - mean)) <= 2e-3


def test_no_error_flag_and_repeatable(gqa):
    a, _ = gqa.gpu_decode(4)
    a = a.clone()
    b, _ = gqa.gpu_decode(4)
    assert torch.equal(a, b)


# --------------------------------------------------------------------------
# kvq_decode: partial + combine in one launch (last CTA merges)
# --------------------------------------------------------------------------

def fused(S, s, out="f32", out_scale=1.0, ws=None):
    cfg = S.config(s, out, out_scale)
    ws = ws or runtime.FusedWorkspace(cfg, S.w.Hkv, S.device)
    flag = torch.zeros(1, dtype=torch.int32, device=S.device)
    res = runtime.decode_fused(S.cache, S.q_t, S.seq_lens_t, cfg, ws, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    return res, ws


@pytest.mark.parametrize("s", [1, 3, 8, 0])
def test_fused_equals_two_launches(gqa, s):
    s = splits_of(gqa.w, s)
    a, _ = gqa.gpu_decode(s, "bf16")
    b, ws = fused(gqa, s, "bf16")
    assert torch.equal(a, b)
    # counters are back at zero: a second call on the same workspace agrees
    c, _ = fused(gqa, s, "bf16", ws=ws)
    assert torch.equal(a, c)
    assert not ws.counters.any()


def test_fused_vs_oracle_all_formats(tiny, nv, paged):
    ref, _ = tiny.oracle_decode()
    out, _ = fused(tiny, 2)
    assert_f32_close(out.cpu().numpy(), ref, "fused tiny")
    ref, _ = nv.oracle_decode()
    out, _ = fused(nv, splits_of(nv.w, 0))
    assert_f32_close(out.cpu().numpy(), ref, "fused nvfp4")
    for s in (1, 2):
        ref, _ = paged.oracle_decode(mode=1, s=s)
        out_scale = float(np.float32(np.float32(np.max(np.abs(ref))) / np.float32(448.0)))
        out, _ = fused(paged, s, "e4m3", out_scale)
        assert_e4m3_close(out.cpu().numpy(), ref, out_scale, f"fused paged e4m3 s={s}")


@pytest.fixture(scope="module")
def gqa4k():
    S = Setup(synth.gqa_fp8(4096))
    return S, S.oracle_decode()[0]


@pytest.mark.parametrize("s", [29, 30, 32, 33, 40, 57, 64])
def test_fused_many_splits(gqa4k, s):
    """Up to 32 splits the last CTA stages the partials of its 4 heads (2 KB
    a split) in shared memory with one copy; beyond that it merges from
    global memory.  Both paths give the two-launch result (fp32 sums in the
    same split order)."""
    S, ref = gqa4k
    a, _ = S.gpu_decode(s)
    b, ws = fused(S, s)
    assert_f32_close(b.cpu().numpy(), ref, f"fused s={s}")
    assert torch.allclose(a, b, rtol=4e-7, atol=1e-7)
    assert not ws.counters.any()


@pytest.mark.parametrize("fmt,s", [("fp8", 13), ("fp8", 20), ("fp8", 47), ("nvfp4", 57)])
def test_fused_many_splits_large_group(fmt, s):
    """16 query heads per kv head: 8 KB of partials per split, so beyond 13
    splits the last CTA merges from global memory with four heads' columns
    per thread."""
    w = synth.gqa_fp8(3000) if fmt == "fp8" else synth.nvfp4(3000)
    w.B, w.Hq, w.Hkv = 2, 16, 1
    w.seq_lens = np.array([3000, 1777], np.int32)
    S = Setup(w)
    ref, _ = S.oracle_decode()
    a, _ = S.gpu_decode(s)
    b, ws = fused(S, s)
    assert_f32_close(b.cpu().numpy(), ref, f"fused G=16 {fmt} s={s}")
    assert torch.allclose(a, b, rtol=4e-7, atol=1e-7)
    assert not ws.counters.any()


def test_fused_workspace_reuse_across_split_counts(gqa):
    """One scratch set (sized for 8 splits) serves calls with fewer splits.
    The fused merge sums the split weights sequentially and the combine
    kernel in a warp reduction, so fp32 outputs agree to a few ulps."""
    big = runtime.FusedWorkspace(gqa.config(8), gqa.w.Hkv, gqa.device)
    for s in (8, 3, 5, 8, 1):
        a, _ = gqa.gpu_decode(s)
        b, _ = fused(gqa, s, ws=big)
        assert torch.allclose(a, b, rtol=4e-7, atol=1e-7), s


# --------------------------------------------------------------------------
# MLA: 16 heads on one NVFP4 latent cache + bf16 rope keys
# --------------------------------------------------------------------------

@pytest.fixture(scope="module")
def mla():
    w = synth.mla_nvfp4(B=3, L=300)
    w.seq_lens = np.array([300, 37, 161], np.int32)
    return Setup(w)


@pytest.mark.parametrize("s", [1, 2, 5])
def test_mla_two_launch(mla, s):
    ref, _ = mla.oracle_decode()
    out, _ = mla.gpu_decode(s)
    assert_f32_close(out.cpu().numpy(), ref, f"mla s={s}")


@pytest.mark.parametrize("s", [1, 4, 5, 9])   # s > 4: the merge reads global memory
def test_mla_fused(mla, s):
    ref, _ = mla.oracle_decode()
    out, ws = fused(mla, s)
    assert_f32_close(out.cpu().numpy(), ref, f"mla fused s={s}")
    assert not ws.counters.any()


@pytest.mark.parametrize("s", [2, 3, 4, 5, 6, 7, 8, 9])
def test_mla_fused_equals_two_launches(mla, s):
    """The fused MLA decode (2..8 splits: clusters merging through
    distributed shared memory, whose item ranges split rows for 3, 5, 6
    and 7; 9: the last CTA's merge) gives the two-launch
    result bit for bit, in fp32, bf16 and E4M3, and leaves the counters at
    zero."""
    for out, scale in (("f32", 1.0), ("bf16", 1.0), ("e4m3", 0.01)):
        a, _ = mla.gpu_decode(s, out, scale)
        b, ws = fused(mla, s, out, scale)
        assert torch.equal(a, b), (s, out)
        assert not ws.counters.any()


def test_mla_fused_many_requests():
    """38 requests x 4 splits: more four-CTA clusters than fit on a GB300 at
    once (36), so the launcher keeps single CTAs and the last CTA's merge; the
    result is still the two-launch one bit for bit, and matches the oracle."""
    w = synth.mla_nvfp4(B=38, L=160)
    w.seq_lens = (np.arange(38, dtype=np.int32) * 7) % 161
    S = Setup(w)
    a, _ = S.gpu_decode(4, "bf16")
    b, ws = fused(S, 4, "bf16")
    assert torch.equal(a, b)
    assert not ws.counters.any()
    ref, _ = S.oracle_decode()
    out, _ = fused(S, 4)
    assert_f32_close(out.cpu().numpy(), ref, "mla 38 requests fused")


def test_mla_paged_bf16_out():
    w = synth.mla_nvfp4(B=2, L=200)
    w.seq_lens = np.array([200, 129], np.int32)
    w.page_size = 16
    w.permute_pages = True
    S = Setup(w)
    ref, _ = S.oracle_decode()
    for s in (1, 3):
        out, _ = S.gpu_decode(s, "bf16")
        assert_bf16_close(bf16_bits(out), ref, f"mla paged bf16 s={s}")


def test_mla_partials_per_chunk(mla):
    s = 3
    w = mla.w
    _, ws = mla.gpu_decode(s)
    po = ws.part_o.cpu().numpy().reshape(w.B, w.Hq, s, w.Dv)
    pl = ws.part_lse.cpu().numpy().reshape(w.B, w.Hq, s)
    q = mla.q64()
    for b in range(w.B):
        kh, vh = mla.oracle_kv(b, 0)
        L = int(w.seq_lens[b])
        for j in range(s):
            st, en = oracle.chunk(L, s, j)
            for hq in (0, 7, 15):
                o, l = oracle.attention_partial(q[b, hq], kh, vh, st, en, w.sm_scale)
                if en == st:
                    assert np.isneginf(pl[b, hq, j]) and not po[b, hq, j].any()
                    continue
                assert abs(pl[b, hq, j] - l) <= 1e-4 * max(1.0, abs(l)), (b, hq, j)
                assert_f32_close(po[b, hq, j], o, f"mla partial b{b} h{hq} j{j}")


@pytest.mark.parametrize("fmt,hq,hkv,d", [("fp8", 8, 8, 128), ("fp8", 16, 2, 64), ("nvfp4", 8, 8, 64),
                                          ("nvfp4", 8, 1, 128), ("fp8", 6, 2, 128)])
def test_six_warp_ctas(fmt, hq, hkv, d):
    """The six-warp CTAs (up to 8 query heads per kv head, head_dim <= 128):
    MHA, 8:1 and 3:1 groups, head_dim 64 and 128, ragged lengths whose box
    counts are not multiples of six warps (and shorter than six boxes), in the
    two-launch and the fused path."""
    w = synth.gqa_fp8(1500) if fmt == "fp8" else synth.nvfp4(1500)
    w.B, w.Hq, w.Hkv, w.D = 3, hq, hkv, d
    w.seq_lens = np.array([1500, 83, 997], np.int32)
    S = Setup(w)
    ref, _ = S.oracle_decode()
    for s in (1, 5, 0):
        s = splits_of(w, s)
        out, _ = S.gpu_decode(s)
        assert_f32_close(out.cpu().numpy(), ref, f"{fmt} {hq}:{hkv} D={d} s={s}")
        b, ws = fused(S, s)
        assert_f32_close(b.cpu().numpy(), ref, f"fused {fmt} {hq}:{hkv} D={d} s={s}")
        assert not ws.counters.any()
