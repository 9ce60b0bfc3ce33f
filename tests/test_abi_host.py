"""The C-ABI library loads, exports every symbol include/kvq.h declares, and
validates arguments on the host (no GPU needed: every call here is rejected
before any CUDA call, or is host-only)."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

from conftest import ROOT
from quantized_kv_cache_05_gb300 import build as kbuild
from quantized_kv_cache_05_gb300 import kvq


@pytest.fixture(scope="module")
def L():
    kbuild.build()
    return kvq.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(kvq.SIGNATURES), "binding covers exactly the header"


def test_status_strings(L):
    assert kvq.status_string(0) == "ok"
    assert "invalid" in kvq.status_string(1)
    assert kvq.status_string(99) == "unknown status"


def test_tensor_scale():
    assert kvq.kvq_tensor_scale(kvq.KVQ_FP8_E4M3, 448.0) == (0, 1.0)
    assert kvq.kvq_tensor_scale(kvq.KVQ_NVFP4, 2688.0) == (0, 1.0)
    assert kvq.kvq_tensor_scale(kvq.KVQ_FP8_E4M3, 0.0) == (0, 1.0)
    st, s = kvq.kvq_tensor_scale(kvq.KVQ_FP8_E4M3, 7.53125)
    assert st == 0
    # one IEEE fp32 division: 7.53125 / 448 rounded once to float
    assert s == float(np.float32(np.float32(7.53125) / np.float32(448.0)))
    for bad in [-1.0, math.nan, math.inf]:
        assert kvq.kvq_tensor_scale(kvq.KVQ_FP8_E4M3, bad)[0] == kvq.KVQ_ERR_INVALID
    assert kvq.kvq_tensor_scale(7, 1.0)[0] == kvq.KVQ_ERR_INVALID


def test_tensor_scale_matches_oracle(orc):
    import numpy as np
    for amax in [1e-3, 0.5, 3.0, 7.53125, 141.0, 1234.5, 3e4]:
        a = float(np.float32(amax))
        assert kvq.kvq_tensor_scale(kvq.KVQ_FP8_E4M3, a)[1] == orc.fp8_tensor_scale(a)
        assert kvq.kvq_tensor_scale(kvq.KVQ_NVFP4, a)[1] == orc.nvfp4_global_scale(a)


def test_auto_splits():
    f = kvq.kvq_auto_splits
    # 152 SMs, GQA 2 x 8 kv heads, two six-warp CTAs per SM: floor(2 * 152 / 16) = 19
    # (one wave of 304 CTAs)
    assert f(152, 2, 8, 4, 32768, 1) == (0, 19)
    assert f(152, 2, 8, 4, 8192, 1) == (0, 19)
    # short sequences: at least 128 tokens per chunk
    assert f(152, 2, 8, 4, 1024, 1) == (0, 8)
    assert f(152, 2, 8, 4, 100, 1) == (0, 1)
    # batch 1 x 8 kv heads: floor(304 / 8) = 38
    assert f(152, 1, 8, 4, 32768, 2) == (0, 38)
    assert f(152, 1, 8, 4, 16384, 2) == (0, 38)
    assert f(152, 1, 8, 4, 12288, 2) == (0, 38)
    # more than 32 splits of chunks under 256 tokens: max(32, ceil(L / 256))
    assert f(152, 1, 8, 4, 9216, 2) == (0, 36)
    assert f(152, 1, 8, 4, 8192, 2) == (0, 32)
    assert f(152, 1, 8, 4, 8192, 1) == (0, 32)
    assert f(152, 1, 8, 4, 2048, 2) == (0, 16)
    # more groups than one wave holds (1024 > 304): chunks of at most 2048 tokens
    # (ceil(8192 / 2048) = 4)
    assert f(152, 64, 16, 1, 8192, 1) == (0, 4)
    assert f(152, 64, 16, 1, 2048, 1) == (0, 1)
    assert f(152, 64, 16, 1, 2049, 1) == (0, 2)
    # groups that fit one wave fill it, whatever the length: floor(304 / 32) = 9,
    # floor(304 / 128) = 2, floor(304 / 64) = 4 (a partial second wave costs more)
    assert f(152, 4, 8, 4, 200000, 1) == (0, 9)
    assert f(152, 16, 8, 4, 8192, 1) == (0, 2)
    assert f(152, 8, 8, 4, 32768, 1) == (0, 4)
    # MLA shape (NVFP4, 16 heads on one kv head: one CTA per SM): floor(152 / 32) = 4
    assert f(152, 32, 1, 16, 4096, 2) == (0, 4)
    assert f(152, 128, 1, 16, 4096, 2) == (0, 1)
    # 16 FP8 heads on one kv head: two CTAs per SM, floor(304 / 32) = 9
    assert f(152, 32, 1, 16, 4096, 1) == (0, 9)
    assert f(152, 2, 1, 12, 32768, 1) == (0, 64)
    # clamp at 64
    assert f(152, 1, 1, 4, 1 << 20, 2) == (0, 64)
    assert f(0, 1, 1, 1, 10, 1)[0] == kvq.KVQ_ERR_INVALID
    assert f(152, 0, 1, 1, 10, 1)[0] == kvq.KVQ_ERR_INVALID


def test_workspace_bytes():
    assert kvq.kvq_partial_workspace_bytes(2, 32, 8, 128) == 2 * 32 * 8 * (128 + 1) * 4
    assert kvq.kvq_partial_workspace_bytes(-1, 1, 1, 1) == 0


def good_cache():
    c = kvq.kvq_cache()
    c.fmt, c.num_pages, c.page_size, c.num_kv_heads, c.head_dim = 1, 4, 16, 2, 128
    c.k_codes, c.v_codes = 0x10000, 0x20000
    c.k_scale = c.v_scale = 0.5
    c.block_table, c.max_pages_per_seq = 0x30000, 4
    return c


def good_params():
    p = kvq.kvq_decode_params()
    p.batch, p.num_q_heads, p.qk_dim, p.v_dim, p.num_splits = 1, 8, 128, 128, 2
    p.seq_lens, p.max_kv_len, p.sm_scale = 0x40000, 64, 0.088
    return p


@pytest.mark.parametrize("mutate", [
    lambda c, p: setattr(c, "fmt", 3),
    lambda c, p: setattr(c, "page_size", 24),
    lambda c, p: setattr(c, "page_size", 0),
    lambda c, p: setattr(c, "num_pages", 0),
    lambda c, p: setattr(c, "k_codes", None),
    lambda c, p: setattr(c, "k_codes", 0x10008),        # not 16-byte aligned
    lambda c, p: setattr(c, "v_codes", None),
    lambda c, p: setattr(c, "k_scale", math.nan),
    lambda c, p: setattr(c, "v_scale", 0.0),
    lambda c, p: setattr(c, "k_scale", -1.0),
    lambda c, p: setattr(c, "block_table", None),
    lambda c, p: setattr(p, "num_splits", 0),
    lambda c, p: setattr(p, "num_q_heads", 7),          # not a multiple of Hkv
    lambda c, p: setattr(p, "sm_scale", math.inf),
    lambda c, p: setattr(p, "prob_scale", -0.5),
    lambda c, p: setattr(p, "max_kv_len", 65),          # beyond 4 pages x 16
    lambda c, p: setattr(p, "seq_lens", None),
    lambda c, p: setattr(p, "qk_dim", 64),
    lambda c, p: setattr(p, "fresh_tokens", -1),
    lambda c, p: (setattr(c, "fmt", 2)),                 # NVFP4 without block scales
], ids=lambda f: "case")
def test_decode_partial_rejects_without_launch(L, mutate):
    c, p = good_cache(), good_params()
    mutate(c, p)
    st = kvq.kvq_decode_partial(c, p, 0x50000, 0x60000, 0x70000, None)
    assert st in (kvq.KVQ_ERR_INVALID, kvq.KVQ_ERR_UNSUPPORTED)


@pytest.mark.parametrize("mutate,want", [
    (lambda c, p: (setattr(c, "head_dim", 96), setattr(p, "qk_dim", 96), setattr(p, "v_dim", 96)),
     kvq.KVQ_ERR_UNSUPPORTED),
    (lambda c, p: setattr(p, "num_q_heads", 64), kvq.KVQ_ERR_UNSUPPORTED),   # G = 32
    (lambda c, p: (setattr(p, "prob_scale", 1 / 448), setattr(p, "num_splits", 1),
                   setattr(c, "max_pages_per_seq", 2000), setattr(p, "max_kv_len", 20000)),
     kvq.KVQ_ERR_UNSUPPORTED),                                               # scores too big
])
def test_decode_partial_unsupported(L, mutate, want):
    c, p = good_cache(), good_params()
    mutate(c, p)
    assert kvq.kvq_decode_partial(c, p, 0x50000, 0x60000, 0x70000, None) == want


def test_decode_null_outputs(L):
    c, p = good_cache(), good_params()
    assert kvq.kvq_decode_partial(c, p, None, 0x60000, 0x70000, None) == kvq.KVQ_ERR_INVALID
    assert kvq.kvq_decode_partial(c, p, 0x50008, 0x60000, 0x70000, None) == kvq.KVQ_ERR_INVALID
    assert kvq.kvq_decode_partial(None, p, 0x50000, 0x60000, 0x70000, None) == kvq.KVQ_ERR_INVALID
    assert kvq.kvq_decode_partial(c, None, 0x50000, 0x60000, 0x70000, None) == kvq.KVQ_ERR_INVALID


def test_decode_batch_zero_is_noop(L):
    c, p = good_cache(), good_params()
    p.batch = 0
    assert kvq.kvq_decode_partial(c, p, None, None, None, None) == kvq.KVQ_OK
    assert kvq.kvq_decode_combine(p, None, None, None, None) == kvq.KVQ_OK


def test_combine_rejects(L):
    p = good_params()
    assert kvq.kvq_decode_combine(p, None, 0x1000, 0x2000, None) == kvq.KVQ_ERR_INVALID
    p.out_dtype = 5
    assert kvq.kvq_decode_combine(p, 0x1000, 0x1000, 0x2000, None) == kvq.KVQ_ERR_INVALID
    p.out_dtype = kvq.KVQ_OUT_E4M3
    p.out_scale = 0.0
    assert kvq.kvq_decode_combine(p, 0x1000, 0x1000, 0x2000, None) == kvq.KVQ_ERR_INVALID


def test_append_rejects(L):
    c = good_cache()
    f = kvq.kvq_quantize_append
    assert f(c, None, 0x2000, None, 0x3000, 1, 1, None) == kvq.KVQ_ERR_INVALID
    assert f(c, 0x1000, None, None, 0x3000, 1, 1, None) == kvq.KVQ_ERR_INVALID
    assert f(c, 0x1000, 0x2000, 0x4000, 0x3000, 1, 1, None) == kvq.KVQ_ERR_INVALID  # kpe w/o MLA
    assert f(c, 0x1000, 0x2000, None, None, 1, 1, None) == kvq.KVQ_ERR_INVALID
    assert f(c, 0x1008, 0x2000, None, 0x3000, 1, 1, None) == kvq.KVQ_ERR_INVALID
    assert f(c, 0x1000, 0x2000, None, 0x3000, -1, 1, None) == kvq.KVQ_ERR_INVALID
    assert f(c, 0x1000, 0x2000, None, 0x3000, 0, 1, None) == kvq.KVQ_OK
    assert f(c, 0x1000, 0x2000, None, 0x3000, 1, 0, None) == kvq.KVQ_OK
    c.rope_dim = 64          # MLA needs k_pe, v_codes NULL, Hkv 1, NVFP4
    assert f(c, 0x1000, None, 0x4000, 0x3000, 1, 1, None) == kvq.KVQ_ERR_INVALID


def test_misc_rejects(L):
    assert kvq.kvq_amax_bf16(None, 10, 0x1000, None) == kvq.KVQ_ERR_INVALID
    assert kvq.kvq_amax_bf16(0x1000, 10, None, None) == kvq.KVQ_ERR_INVALID
    assert kvq.kvq_encode_e4m3(None, 0x1000, 4, None) == kvq.KVQ_ERR_INVALID
    assert kvq.kvq_encode_e2m1(0x1000, None, 4, None) == kvq.KVQ_ERR_INVALID
    assert kvq.kvq_encode_e4m3(None, None, 0, None) == kvq.KVQ_OK


def test_fused_decode_rejects(L):
    c, p = good_cache(), good_params()
    f = kvq.kvq_decode
    assert f(c, p, 0x50000, 0x60000, 0x70000, None, 0x80000, None) == kvq.KVQ_ERR_INVALID
    assert f(c, p, 0x50000, 0x60000, 0x70000, 0x90000, None, None) == kvq.KVQ_ERR_INVALID
    assert f(c, p, 0x50000, None, 0x70000, 0x90000, 0x80000, None) == kvq.KVQ_ERR_INVALID
    p.num_splits = 65
    assert f(c, p, 0x50000, 0x60000, 0x70000, 0x90000, 0x80000, None) == kvq.KVQ_ERR_UNSUPPORTED
    assert kvq.kvq_decode_partial(c, p, 0x50000, 0x60000, 0x70000, None) == kvq.KVQ_ERR_UNSUPPORTED
    assert kvq.kvq_decode_combine(p, 0x60000, 0x70000, 0x80000, None) == kvq.KVQ_ERR_UNSUPPORTED
    p.num_splits, p.batch = 2, 0
    assert f(c, p, None, None, None, None, None, None) == kvq.KVQ_OK


def test_prob_division_host_check():
    """n = 0 runs only the host check of the FP8-probability division: the
    reciprocal path is accepted for the workloads' prob scale fl32(1/448)
    and for other scales; invalid scales are refused."""
    import numpy as np
    for ps in [np.float32(1 / 448), np.float32(1 / 240), np.float32(0.00311), 2.0 ** -8]:
        assert kvq.kvq_encode_prob_e4m3(None, None, 0, float(ps)) == (kvq.KVQ_OK, 1)
    for bad in [0.0, -1.0, math.inf, math.nan]:
        assert kvq.kvq_encode_prob_e4m3(None, None, 0, bad)[0] == kvq.KVQ_ERR_INVALID


def nvfp4_cache(D):
    c = good_cache()
    c.fmt, c.head_dim = kvq.KVQ_NVFP4, D
    c.k_bscale, c.v_bscale = 0xA0000, 0xB0000
    return c


@pytest.mark.parametrize("D,want", [(40, kvq.KVQ_ERR_INVALID),        # D % 16 != 0
                                    (24, kvq.KVQ_ERR_INVALID),
                                    (96, kvq.KVQ_ERR_UNSUPPORTED),    # valid, no kernel
                                    (512, kvq.KVQ_ERR_UNSUPPORTED)])  # only as the MLA latent
def test_nvfp4_head_dims_refused_before_launch(L, D, want):
    """NVFP4 decode runs at head_dim 64, 128 and 256; a cache whose head_dim
    is not a multiple of 16 is invalid, other multiples are refused as
    unsupported -- in both cases before any launch."""
    c, p = nvfp4_cache(D), good_params()
    p.qk_dim = p.v_dim = D
    assert kvq.kvq_decode_partial(c, p, 0x50000, 0x60000, 0x70000, None) == want
    assert kvq.kvq_decode(c, p, 0x50000, 0x60000, 0x70000, 0x90000, 0x80000, None) == want


def test_head_scale_fields(L):
    """Per-kv-head scales replace the per-tensor ones (which may then be
    anything) and are refused for the MLA latent cache."""
    c, p = good_cache(), good_params()
    c.k_head_scale, c.v_head_scale = 0xC0000, 0xD0000
    c.k_scale = c.v_scale = 0.0
    c.head_dim, c.num_kv_heads = 96, 2   # an unsupported dim: refused after the scale checks
    p.qk_dim = p.v_dim = 96
    assert kvq.kvq_decode_partial(c, p, 0x50000, 0x60000, 0x70000, None) == kvq.KVQ_ERR_UNSUPPORTED
    c.k_head_scale = None                # back to the per-tensor k_scale = 0: invalid
    assert kvq.kvq_decode_partial(c, p, 0x50000, 0x60000, 0x70000, None) == kvq.KVQ_ERR_INVALID
    m = nvfp4_cache(512)
    m.num_kv_heads, m.v_codes, m.v_bscale, m.rope_dim, m.k_pe, m.v_is_k_latent = 1, None, None, 64, 0xE0000, 1
    m.k_head_scale = 0xC0000
    assert kvq.kvq_quantize_append(m, 0x1000, None, 0x4000, 0x3000, 1, 1, None) == kvq.KVQ_ERR_INVALID
