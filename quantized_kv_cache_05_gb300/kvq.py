"""Thin Python binding of the C ABI in include/kvq.h (ctypes).

Argument marshalling only: every step of quantize-on-append and split-KV
decode runs in the CUDA kernels of libkvq.so.  Functions keep the C names.
Tensor arguments may be torch tensors (their data_ptr() is passed) or raw
integer addresses.  A missing or unloadable libkvq.so raises; there is no
fallback path.

Streams: ``stream=None`` means torch's current CUDA stream when torch is
loaded with CUDA, else the legacy default stream.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Any, Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvq.so")

KVQ_OK, KVQ_ERR_INVALID, KVQ_ERR_UNSUPPORTED, KVQ_ERR_WORKSPACE, KVQ_ERR_CUDA = 0, 1, 2, 3, 4
KVQ_FP8_E4M3, KVQ_NVFP4 = 1, 2
KVQ_OUT_F32, KVQ_OUT_BF16, KVQ_OUT_E4M3 = 0, 1, 2
KVQ_DEVERR_WAIT_TIMEOUT, KVQ_DEVERR_SEQ_CLAMPED = 1, 2
KVQ_NOALLOC_SCRATCH_BYTES = 4 << 20

_i32 = ctypes.c_int32
_int = ctypes.c_int
_f = ctypes.c_float
_P = ctypes.c_void_p
_sz = ctypes.c_size_t


class kvq_cache(ctypes.Structure):
    _fields_ = [
        ("fmt", _i32), ("num_pages", _i32), ("page_size", _i32), ("num_kv_heads", _i32),
        ("head_dim", _i32), ("k_codes", _P), ("v_codes", _P), ("k_bscale", _P),
        ("v_bscale", _P), ("k_scale", _f), ("v_scale", _f), ("block_table", _P),
        ("max_pages_per_seq", _i32), ("rope_dim", _i32), ("k_pe", _P), ("v_is_k_latent", _i32),
        ("k_head_scale", _P), ("v_head_scale", _P),
    ]


class kvq_decode_params(ctypes.Structure):
    _fields_ = [
        ("batch", _i32), ("num_q_heads", _i32), ("qk_dim", _i32), ("v_dim", _i32),
        ("num_splits", _i32), ("seq_lens", _P), ("max_kv_len", _i32), ("sm_scale", _f),
        ("prob_scale", _f), ("out_dtype", _i32), ("out_scale", _f), ("error_flag", _P),
        ("fresh_tokens", _i32), ("q_fp8", _i32), ("q_scale", _f), ("q_head_scale", _P),
    ]


# name -> (restype, argtypes); the exported surface of include/kvq.h
SIGNATURES = {
    "kvq_status_string": (ctypes.c_char_p, [_int]),
    "kvq_tensor_scale": (_int, [_int, _f, ctypes.POINTER(_f)]),
    "kvq_amax_bf16": (_int, [_P, _sz, _P, _P]),
    "kvq_quantize_append": (_int, [ctypes.POINTER(kvq_cache), _P, _P, _P, _P, _int, _int, _P]),
    "kvq_auto_splits": (_int, [_int, _int, _int, _int, _int, _int, ctypes.POINTER(_int)]),
    "kvq_partial_workspace_bytes": (_sz, [_int, _int, _int, _int]),
    "kvq_decode_partial": (_int, [ctypes.POINTER(kvq_cache), ctypes.POINTER(kvq_decode_params),
                                  _P, _P, _P, _P]),
    "kvq_decode_combine": (_int, [ctypes.POINTER(kvq_decode_params), _P, _P, _P, _P]),
    "kvq_decode": (_int, [ctypes.POINTER(kvq_cache), ctypes.POINTER(kvq_decode_params), _P, _P,
                          _P, _P, _P, _P]),
    "kvq_decode_noalloc": (_int, [ctypes.POINTER(kvq_cache), ctypes.POINTER(kvq_decode_params),
                                  _P, _P, _P]),
    "kvq_encode_e4m3": (_int, [_P, _P, _sz, _P]),
    "kvq_encode_e2m1": (_int, [_P, _P, _sz, _P]),
    "kvq_encode_prob_e4m3": (_int, [_P, _P, _sz, _f, ctypes.POINTER(_int), _P]),
    "kvq_quantize_fp8": (_int, [_P, _sz, _f, _P, _int, _int, _P, _P]),
    "kvq_prefill": (_int, [ctypes.POINTER(kvq_cache), ctypes.POINTER(kvq_decode_params), _int,
                           _P, _P, _P]),
}

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """Load libkvq.so (built by quantized_kv_cache_05_gb300.build)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _addr(x: Any) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"expected a tensor or an address, got {type(x)}")


def _ref(x):
    return None if x is None else ctypes.byref(x)


def _stream(s: Any) -> Optional[int]:
    if s is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return torch.cuda.current_stream().cuda_stream
        except Exception:  # pragma: no cover - torch without CUDA
            pass
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def check(status: int, what: str = "kvq") -> None:
    if status != KVQ_OK:
        raise KvqError(status, what)


def status_string(s: int) -> str:
    return lib().kvq_status_string(s).decode()


def kvq_tensor_scale(fmt: int, amax: float) -> tuple[int, float]:
    out = _f(0.0)
    st = lib().kvq_tensor_scale(fmt, amax, ctypes.byref(out))
    return st, float(out.value)


def kvq_amax_bf16(x, n: int, amax_out, stream=None) -> int:
    return lib().kvq_amax_bf16(_addr(x), n, _addr(amax_out), _stream(stream))


def kvq_quantize_append(cache: kvq_cache, k_new, v_new, kpe_new, start_pos, batch: int,
                        n_tokens: int, stream=None) -> int:
    return lib().kvq_quantize_append(_ref(cache), _addr(k_new), _addr(v_new),
                                     _addr(kpe_new), _addr(start_pos), batch, n_tokens,
                                     _stream(stream))


def kvq_auto_splits(num_sms: int, batch: int, num_kv_heads: int, q_per_kv: int,
                    max_kv_len: int, fmt: int) -> tuple[int, int]:
    out = _int(0)
    st = lib().kvq_auto_splits(num_sms, batch, num_kv_heads, q_per_kv, max_kv_len, fmt,
                               ctypes.byref(out))
    return st, int(out.value)


def kvq_partial_workspace_bytes(batch: int, num_q_heads: int, num_splits: int,
                                v_dim: int) -> int:
    return int(lib().kvq_partial_workspace_bytes(batch, num_q_heads, num_splits, v_dim))


def kvq_decode_partial(cache: kvq_cache, params: kvq_decode_params, q, part_o, part_lse,
                       stream=None) -> int:
    return lib().kvq_decode_partial(_ref(cache), _ref(params), _addr(q),
                                    _addr(part_o), _addr(part_lse), _stream(stream))


def kvq_decode_combine(params: kvq_decode_params, part_o, part_lse, out, stream=None) -> int:
    return lib().kvq_decode_combine(_ref(params), _addr(part_o), _addr(part_lse),
                                    _addr(out), _stream(stream))


def kvq_decode(cache: kvq_cache, params: kvq_decode_params, q, part_o, part_lse, counters,
               out, stream=None) -> int:
    return lib().kvq_decode(_ref(cache), _ref(params), _addr(q), _addr(part_o), _addr(part_lse),
                            _addr(counters), _addr(out), _stream(stream))


def kvq_decode_noalloc(cache: kvq_cache, params: kvq_decode_params, q, out, stream=None) -> int:
    """kvq_decode with the library's own static scratch buffer: for callers
    that cannot allocate device memory for split partials (see kvq.h)."""
    return lib().kvq_decode_noalloc(_ref(cache), _ref(params), _addr(q), _addr(out),
                                    _stream(stream))


def kvq_encode_e4m3(x, out, n: int, stream=None) -> int:
    return lib().kvq_encode_e4m3(_addr(x), _addr(out), n, _stream(stream))


def kvq_encode_e2m1(x, out, n: int, stream=None) -> int:
    return lib().kvq_encode_e2m1(_addr(x), _addr(out), n, _stream(stream))


def kvq_encode_prob_e4m3(p, out, n: int, prob_scale: float, stream=None) -> tuple[int, int]:
    """E4M3 codes of fl32(p / prob_scale) as the decode kernels compute them;
    returns (status, 1 if the reciprocal path was used else 0)."""
    used = _int(0)
    st = lib().kvq_encode_prob_e4m3(_addr(p), _addr(out), n, prob_scale, ctypes.byref(used),
                                    _stream(stream))
    return st, int(used.value)


def kvq_quantize_fp8(x, n: int, scale: float, head_scale, head_len: int, num_heads: int, out,
                     stream=None) -> int:
    """E4M3 codes of bf16 x with a per-tensor scale or per-head scales."""
    return lib().kvq_quantize_fp8(_addr(x), n, scale, _addr(head_scale), head_len, num_heads,
                                  _addr(out), _stream(stream))


def kvq_prefill(cache: kvq_cache, params: kvq_decode_params, q_len: int, q, out,
                stream=None) -> int:
    """Causal prefill attention of q_len new tokens per request (no KV split)."""
    return lib().kvq_prefill(_ref(cache), _ref(params), q_len, _addr(q), _addr(out),
                             _stream(stream))
