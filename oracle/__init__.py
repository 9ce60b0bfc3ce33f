"""Plain CPU oracle for quantized-KV decode attention -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never does, and shares no code with it.

The arithmetic lives in ``oracle.cpp`` (C++17, fp64); this module builds it
with g++ and exposes thin numpy wrappers.  Each wrapper's docstring names the
passage of the source pages it follows; ``oracle.cpp`` has the details.

Parity pins (what checks the oracle against something other than itself) are
in ``tests/test_oracle_*.py``.  The one reading with no independent pin is the
FP8-probability semantics of ``attention_partial_probq`` (parity unpinned:
the vLLM FP8-attention page only says that softmax(QK^T) is quantized to FP8
with a prob scale, not against which max).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.cpp into liboracle.so (g++, -O2, no FP contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", _LIB + ".tmp"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            _declare(L)
            _lib = L
    return _lib


_P = ctypes.c_void_p
_sz = ctypes.c_size_t
_i = ctypes.c_int
_f = ctypes.c_float
_d = ctypes.c_double
_u64 = ctypes.c_uint64


def _declare(L: ctypes.CDLL) -> None:
    sig = {
        "orc_e4m3_encode": (ctypes.c_uint8, [_f]),
        "orc_e4m3_decode": (_d, [ctypes.c_uint8]),
        "orc_e2m1_encode": (ctypes.c_uint8, [_f]),
        "orc_e2m1_decode": (_d, [ctypes.c_uint8]),
        "orc_e4m3_encode_n": (None, [_P, _sz, _P]),
        "orc_e2m1_encode_n": (None, [_P, _sz, _P]),
        "orc_count_encode_mismatch": (_u64, [_i, _u64, _u64, _P, _i, _P]),
        "orc_bruteforce_encode_check": (_u64, [_i, _u64, _u64, _i, _P]),
        "orc_count_probq_mismatch": (_u64, [_u64, _u64, _f, _P, _i, _P]),
        "orc_amax_bf16": (_f, [_P, _sz]),
        "orc_fp8_tensor_scale": (_f, [_f]),
        "orc_nvfp4_global_scale": (_f, [_f]),
        "orc_fp8_quantize": (None, [_P, _sz, _f, _P]),
        "orc_nvfp4_quantize": (None, [_P, _sz, _i, _f, _P, _P]),
        "orc_head_amax_bf16": (None, [_P, _sz, _i, _i, _P]),
        "orc_fp8_quantize_heads": (None, [_P, _sz, _i, _i, _P, _P]),
        "orc_nvfp4_quantize_heads": (None, [_P, _sz, _i, _i, _P, _P, _P]),
        "orc_fp8_dequant": (None, [_P, _sz, _f, _P]),
        "orc_nvfp4_dequant": (None, [_P, _P, _sz, _i, _f, _P]),
        "orc_chunk": (None, [_i, _i, _i, _P, _P]),
        "orc_attention_exact": (None, [_P, _P, _P, _i, _i, _i, _d, _P, _P]),
        "orc_attention_partial": (None, [_P, _P, _P, _i, _i, _i, _i, _d, _P, _P]),
        "orc_attention_partial_probq": (None, [_P, _P, _P, _i, _i, _i, _i, _d, _f, _P, _P]),
        "orc_combine": (None, [_P, _P, _i, _i, _P]),
        "orc_fp8_output": (None, [_P, _sz, _f, _P]),
        "orc_decode_batch": (None, [_P, _P, _P, _i, _i, _i, _i, _P, _i, _i, _d, _i, _i, _f,
                                    _P, _P, _i]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle wrappers need C-contiguous arrays"
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# --------------------------------------------------------------------------
# Codecs (E4M3 "FN" and E2M1; the pages name them "(4, 3)" and "(2, 1) bit"
# in the Model-Optimizer PR 714 module printout)
# --------------------------------------------------------------------------

def e4m3_encode(x) -> np.ndarray:
    """Round-to-nearest-even onto the E4M3 grid, saturating at +-448."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().orc_e4m3_encode_n(_ptr(x), x.size, _ptr(out))
    return out


def e4m3_decode(codes) -> np.ndarray:
    codes = np.asarray(codes, np.uint8)
    f = lib().orc_e4m3_decode
    return np.array([f(int(c)) for c in codes.ravel()], np.float64).reshape(codes.shape)


def e2m1_encode(x) -> np.ndarray:
    """Round-to-nearest-even onto the E2M1 grid, saturating at +-6 (nibbles)."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().orc_e2m1_encode_n(_ptr(x), x.size, _ptr(out))
    return out


def e2m1_decode(codes) -> np.ndarray:
    codes = np.asarray(codes, np.uint8)
    f = lib().orc_e2m1_decode
    return np.array([f(int(c)) for c in codes.ravel()], np.float64).reshape(codes.shape)


def count_encode_mismatch(kind: int, first: int, observed: np.ndarray,
                          nthreads: int | None = None) -> tuple[int, int]:
    """Compare observed codes for fp32 patterns [first, first+len) with the
    oracle encoder (kind 0 = E4M3, 1 = E2M1).  Returns (mismatches, first bad
    pattern or 2**64-1)."""
    observed = _c(observed, np.uint8)
    fb = ctypes.c_uint64(0)
    n = lib().orc_count_encode_mismatch(kind, first, observed.size, _ptr(observed),
                                        nthreads or default_threads(), ctypes.byref(fb))
    return int(n), int(fb.value)


def count_probq_mismatch(first: int, prob_scale: float, observed: np.ndarray,
                         nthreads: int | None = None) -> tuple[int, int]:
    """Compare observed codes for fp32 patterns [first, first+len), read as
    probabilities p, with E4M3(fl32(p / prob_scale)) (the FP8-probability
    step of vLLM PR 15734 as attention_partial_probq applies it).  Returns
    (mismatches, first bad pattern or 2**64-1)."""
    observed = _c(observed, np.uint8)
    fb = ctypes.c_uint64(0)
    n = lib().orc_count_probq_mismatch(first, observed.size, prob_scale, _ptr(observed),
                                       nthreads or default_threads(), ctypes.byref(fb))
    return int(n), int(fb.value)


def bruteforce_encode_check(kind: int, first: int, n: int,
                            nthreads: int | None = None) -> tuple[int, int]:
    """Nearest-value table search vs the encoder over fp32 patterns."""
    fb = ctypes.c_uint64(0)
    bad = lib().orc_bruteforce_encode_check(kind, first, n, nthreads or default_threads(),
                                            ctypes.byref(fb))
    return int(bad), int(fb.value)


# --------------------------------------------------------------------------
# Static scales (compressed-tensors PR 436 kv_cache_scheme: static, minmax,
# per tensor; Model-Optimizer PR 714 MaxCalibrator amax)
# --------------------------------------------------------------------------

def amax_bf16(x_bf16: np.ndarray) -> float:
    x = _c(x_bf16, np.uint16)
    return float(lib().orc_amax_bf16(_ptr(x), x.size))


def fp8_tensor_scale(amax: float) -> float:
    return float(lib().orc_fp8_tensor_scale(amax))


def nvfp4_global_scale(amax: float) -> float:
    return float(lib().orc_nvfp4_global_scale(amax))


# --------------------------------------------------------------------------
# Quantizers and dequantizers
# --------------------------------------------------------------------------

def fp8_quantize(x_bf16: np.ndarray, scale: float) -> np.ndarray:
    x = _c(x_bf16, np.uint16)
    out = np.empty(x.shape, np.uint8)
    lib().orc_fp8_quantize(_ptr(x), x.size, scale, _ptr(out))
    return out


def nvfp4_quantize(x_bf16: np.ndarray, g: float) -> tuple[np.ndarray, np.ndarray]:
    """x [..., D] bf16 -> (codes [..., D/2], block scales [..., D/16])."""
    x = _c(x_bf16, np.uint16)
    D = x.shape[-1]
    rows = x.size // D
    codes = np.empty(x.shape[:-1] + (D // 2,), np.uint8)
    sc = np.empty(x.shape[:-1] + (D // 16,), np.uint8)
    lib().orc_nvfp4_quantize(_ptr(x), rows, D, g, _ptr(codes), _ptr(sc))
    return codes, sc


# --------------------------------------------------------------------------
# Per-kv-head scales (compressed-tensors PR 436: "attn_head" strategy)
# --------------------------------------------------------------------------

def head_amax_bf16(x_bf16: np.ndarray) -> np.ndarray:
    """x [rows][H][D] bf16 -> amax [H] (float32): max |x| over each kv head."""
    x = _c(x_bf16, np.uint16)
    rows, H, D = x.shape
    out = np.empty(H, np.float32)
    lib().orc_head_amax_bf16(_ptr(x), rows, H, D, _ptr(out))
    return out


def fp8_head_scales(x_bf16: np.ndarray) -> np.ndarray:
    """Per-kv-head FP8 scales fl32(amax_h / 448) of x [rows][H][D]."""
    return np.array([fp8_tensor_scale(float(a)) for a in head_amax_bf16(x_bf16)], np.float32)


def nvfp4_head_scales(x_bf16: np.ndarray) -> np.ndarray:
    """Per-kv-head NVFP4 global scales fl32(amax_h / 2688) of x [rows][H][D]."""
    return np.array([nvfp4_global_scale(float(a)) for a in head_amax_bf16(x_bf16)], np.float32)


def fp8_quantize_heads(x_bf16: np.ndarray, scales) -> np.ndarray:
    """x [rows][H][D] -> codes, element [r][h][d] with scales[h]."""
    x = _c(x_bf16, np.uint16)
    rows, H, D = x.shape
    sc = _c(scales, np.float32)
    assert sc.size == H
    out = np.empty(x.shape, np.uint8)
    lib().orc_fp8_quantize_heads(_ptr(x), rows, H, D, _ptr(sc), _ptr(out))
    return out


def nvfp4_quantize_heads(x_bf16: np.ndarray, gs) -> tuple[np.ndarray, np.ndarray]:
    """x [rows][H][D] -> (codes [rows][H][D/2], block scales [rows][H][D/16]),
    head h with global scale gs[h]."""
    x = _c(x_bf16, np.uint16)
    rows, H, D = x.shape
    g = _c(gs, np.float32)
    assert g.size == H
    codes = np.empty((rows, H, D // 2), np.uint8)
    sc = np.empty((rows, H, D // 16), np.uint8)
    lib().orc_nvfp4_quantize_heads(_ptr(x), rows, H, D, _ptr(g), _ptr(codes), _ptr(sc))
    return codes, sc


# --------------------------------------------------------------------------
# FP8 query (compressed-tensors PR 436: "QKV-FP8-Tensor" / "QKV-FP8-Head",
# a query observer next to the K and V ones; vLLM PR 15734: QK quantization
# in the attention loop).  The query is quantized like K: E4M3(fl32(q / s))
# with a static scale per tensor or per query head, and the scores use the
# dequantized query.
# --------------------------------------------------------------------------

def fp8_query(q_bf16: np.ndarray, scales) -> tuple[np.ndarray, np.ndarray]:
    """q [B][Hq][D] bf16 and one scale (per tensor) or Hq scales (per query
    head) -> (E4M3 codes [B][Hq][D], dequantized q in float64)."""
    q = _c(q_bf16, np.uint16)
    sc = np.atleast_1d(np.asarray(scales, np.float32))
    if sc.size == 1:
        codes = fp8_quantize(q, float(sc[0]))
        return codes, fp8_dequant(codes, float(sc[0]))
    codes = fp8_quantize_heads(q, sc)
    deq = np.empty(q.shape, np.float64)
    for h in range(q.shape[1]):
        deq[:, h] = fp8_dequant(np.ascontiguousarray(codes[:, h]), float(sc[h]))
    return codes, deq


def fp8_dequant(codes: np.ndarray, scale: float) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().orc_fp8_dequant(_ptr(c), c.size, scale, _ptr(out))
    return out


def nvfp4_dequant(codes: np.ndarray, scales: np.ndarray, g: float) -> np.ndarray:
    c = _c(codes, np.uint8)
    s = _c(scales, np.uint8)
    D = c.shape[-1] * 2
    rows = c.size // (D // 2)
    out = np.empty(c.shape[:-1] + (D,), np.float64)
    lib().orc_nvfp4_dequant(_ptr(c), _ptr(s), rows, D, g, _ptr(out))
    return out


# --------------------------------------------------------------------------
# Attention (Model-Optimizer PR 1832: split-KV decode notes)
# --------------------------------------------------------------------------

def chunk(L: int, s: int, j: int) -> tuple[int, int]:
    st, en = ctypes.c_int(0), ctypes.c_int(0)
    lib().orc_chunk(L, s, j, ctypes.byref(st), ctypes.byref(en))
    return st.value, en.value


def attention_exact(q, k, v, sm_scale: float) -> tuple[np.ndarray, float]:
    q = _c(q, np.float64)
    k = _c(k, np.float64)
    v = _c(v, np.float64)
    L = k.shape[0]
    out = np.empty(v.shape[1], np.float64)
    lse = ctypes.c_double(0)
    lib().orc_attention_exact(_ptr(q), _ptr(k), _ptr(v), L, q.size, v.shape[1], sm_scale,
                              _ptr(out), ctypes.byref(lse))
    return out, lse.value


def attention_partial(q, k, v, start: int, end: int, sm_scale: float):
    q = _c(q, np.float64)
    k = _c(k, np.float64)
    v = _c(v, np.float64)
    out = np.empty(v.shape[1], np.float64)
    lse = ctypes.c_double(0)
    lib().orc_attention_partial(_ptr(q), _ptr(k), _ptr(v), start, end, q.size, v.shape[1],
                                sm_scale, _ptr(out), ctypes.byref(lse))
    return out, lse.value


def attention_partial_probq(q, k, v, start: int, end: int, sm_scale: float,
                            prob_scale: float):
    q = _c(q, np.float64)
    k = _c(k, np.float64)
    v = _c(v, np.float64)
    out = np.empty(v.shape[1], np.float64)
    lse = ctypes.c_double(0)
    lib().orc_attention_partial_probq(_ptr(q), _ptr(k), _ptr(v), start, end, q.size,
                                      v.shape[1], sm_scale, prob_scale, _ptr(out),
                                      ctypes.byref(lse))
    return out, lse.value


def prefill_attention(q, k, v, sm_scale: float) -> tuple[np.ndarray, np.ndarray]:
    """Causal attention of Tq new query tokens over a cache of L tokens that
    already holds them (Model-Optimizer PR 1832: the prefill kernel that its
    latency tables compare with split decode).  Query i sits at position
    L - Tq + i and attends to keys [0, L - Tq + i]: exact attention per query
    over that prefix.  q [Tq][Dqk], k [L][Dqk], v [L][Dv] (float64) ->
    (out [Tq][Dv], lse [Tq])."""
    q = _c(q, np.float64)
    k = _c(k, np.float64)
    v = _c(v, np.float64)
    Tq, L = q.shape[0], k.shape[0]
    assert Tq <= L, "the cache holds the new tokens"
    out = np.empty((Tq, v.shape[1]), np.float64)
    lse = np.empty(Tq, np.float64)
    for i in range(Tq):
        n = L - Tq + i + 1
        out[i], lse[i] = attention_exact(q[i], k[:n], v[:n], sm_scale)
    return out, lse


def combine(o_parts, lse) -> np.ndarray:
    o = _c(o_parts, np.float64)
    l = _c(lse, np.float64)
    s, Dv = o.shape
    out = np.empty(Dv, np.float64)
    lib().orc_combine(_ptr(o), _ptr(l), s, Dv, _ptr(out))
    return out


def fp8_output(o, out_scale: float) -> np.ndarray:
    o = _c(o, np.float64)
    out = np.empty(o.shape, np.uint8)
    lib().orc_fp8_output(_ptr(o), o.size, out_scale, _ptr(out))
    return out


def decode_batch(q, khat, vhat, seq_lens, sm_scale: float, mode: int = 0, s: int = 1,
                 prob_scale: float = 0.0, nthreads: int | None = None):
    """q [B][Hq][Dqk]; khat [B][Hkv][Lcap][Dqk]; vhat [B][Hkv][Lcap][Dv] (all
    float64); seq_lens [B].  mode 0 = exact attention, 1 = FP8-probability
    reading with s splits.  Returns (out [B][Hq][Dv], lse [B][Hq])."""
    q = _c(q, np.float64)
    khat = _c(khat, np.float64)
    vhat = _c(vhat, np.float64)
    sl = _c(seq_lens, np.int32)
    B, Hq, Dqk = q.shape
    _, Hkv, Lcap, _ = khat.shape
    Dv = vhat.shape[-1]
    out = np.empty((B, Hq, Dv), np.float64)
    lse = np.empty((B, Hq), np.float64)
    lib().orc_decode_batch(_ptr(q), _ptr(khat), _ptr(vhat), B, Hq, Hkv, Lcap, _ptr(sl), Dqk,
                           Dv, sm_scale, mode, s, prob_scale, _ptr(out), _ptr(lse),
                           nthreads or default_threads())
    return out, lse
