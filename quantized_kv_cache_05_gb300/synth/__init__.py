"""Seeded synthetic inputs for the quantized-KV decode workloads.

This package draws random numbers and describes workload shapes; it holds
none of the method's arithmetic.  Both the CUDA library's tests and benchmark
and the CPU oracle take their inputs from here -- it is the only code the two
sides share.

The generator itself is ``gen.c`` (counter-based SplitMix64 streams,
Box-Muller normals rounded to bf16); see its header for the exact definition.
Tensor ids: Q = 0, K = 1 (MLA: the latent kv_c), V = 2, K_PE = 3.
Purposes: 0 values, 1 element outliers, 2 outlier channels, 3 sequence
lengths, 4 page permutation.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libkvqsynth.so")
_lock = threading.Lock()
_lib = None

T_Q, T_K, T_V, T_KPE = 0, 1, 2, 3
P_VALUES, P_OUTLIERS, P_CHANNELS, P_LENGTHS, P_PAGES = 0, 1, 2, 3, 4


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
               _SRC, "-o", _LIB + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            L.syn_key.restype = ctypes.c_uint64
            L.syn_key.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32]
            L.syn_draw.restype = ctypes.c_uint64
            L.syn_draw.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            L.syn_fill_bf16.restype = None
            L.syn_fill_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64,
                                        ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p,
                                        ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                        ctypes.c_void_p, ctypes.c_int]
            _lib = L
    return _lib


def threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def fill_bf16(seed: int, tensor: int, n: int, offset: int = 0, D: int = 0,
              chan_mask: Optional[np.ndarray] = None, chan_mult: float = 1.0,
              elem_p: float = 0.0, elem_mult: float = 1.0,
              out: Optional[np.ndarray] = None) -> np.ndarray:
    """Elements offset..offset+n of a tensor, as bf16 bit patterns (uint16)."""
    if out is None:
        out = np.empty(n, np.uint16)
    assert out.dtype == np.uint16 and out.flags["C_CONTIGUOUS"] and out.size == n
    cm = None
    if chan_mask is not None:
        cm = np.ascontiguousarray(chan_mask, np.uint8)
        assert cm.size == D
    lib().syn_fill_bf16(seed, tensor, offset, n, D,
                        None if cm is None else cm.ctypes.data, chan_mult, elem_p, elem_mult,
                        out.ctypes.data, threads())
    return out


def draws(seed: int, tensor: int, purpose: int, n: int) -> np.ndarray:
    L = lib()
    key = L.syn_key(seed, tensor, purpose)
    return np.array([L.syn_draw(key, i) for i in range(n)], np.uint64)


def bf16_to_f32(u16: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact)."""
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def pick_channels(seed: int, D: int, k: int) -> list[int]:
    """k distinct channels in [0, D), drawn once from the channel stream."""
    out: list[int] = []
    d = draws(seed, 0, P_CHANNELS, 64 * k)
    for r in d:
        c = int(r % np.uint64(D))
        if c not in out:
            out.append(c)
        if len(out) == k:
            return out
    raise RuntimeError("pick_channels: ran out of draws")


def uniform_lengths(seed: int, B: int, lo: int, hi: int) -> np.ndarray:
    """B integers uniform on {lo..hi} (inclusive)."""
    d = draws(seed, 0, P_LENGTHS, B)
    return (lo + (d % np.uint64(hi - lo + 1))).astype(np.int32)


def permutation(seed: int, n: int) -> np.ndarray:
    """Fisher-Yates permutation of 0..n-1 from the page stream."""
    L = lib()
    key = L.syn_key(seed, 0, P_PAGES)
    p = np.arange(n, dtype=np.int32)
    for i in range(n - 1, 0, -1):
        j = int(L.syn_draw(key, i) % (i + 1))
        p[i], p[j] = p[j], p[i]
    return p


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    """Shapes and value recipe of one decode workload.

    Logical input layouts (the quantize-on-append input layout):
      q  [B][Hq][Dqk]          (MLA: 512 latent + 64 rope, concatenated)
      k  [B][Lmax][Hkv][D]     (MLA: kv_c [B][Lmax][1][512])
      v  [B][Lmax][Hkv][Dv]    (absent for MLA: V is the latent kv_c)
      kpe [B][Lmax][rope]      (MLA only)
    Request b uses the first seq_lens[b] positions.
    """
    name: str
    fmt: str                 # "fp8" or "nvfp4"
    B: int
    Hq: int
    Hkv: int
    D: int                   # K head dim (MLA: latent dim 512)
    seq_lens: np.ndarray
    page_size: int = 0       # 0 = contiguous cache (one page per request)
    rope: int = 0            # MLA rope dim (0 = not MLA)
    seed: int = 0
    chan_outliers: int = 0   # number of outlier channels (same for Q, K, V)
    chan_mult: float = 1.0
    elem_p: float = 0.0      # per-element outlier probability
    elem_mult: float = 1.0
    prob_fp8: bool = False   # FP8-quantized softmax probabilities
    out: str = "f32"         # "f32", "bf16" or "e4m3"
    splits: tuple = (1,)
    permute_pages: bool = False
    head_scales: bool = False     # per-kv-head static scales ("attn_head" strategy)
    head_exp: tuple = ()          # K/V of kv head h times 2^head_exp[h % len] (exact)
    q_fp8: bool = False           # FP8 query (E4M3 codes with a per-tensor scale)

    @property
    def mla(self) -> bool:
        return self.rope > 0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def Dqk(self) -> int:
        return self.D + self.rope

    @property
    def Dv(self) -> int:
        return self.D

    @property
    def Lmax(self) -> int:
        return int(np.max(self.seq_lens)) if len(self.seq_lens) else 0

    @property
    def sm_scale(self) -> float:
        """fl32(1/sqrt(d)) with d the head dim (MLA: 192 = 128 nope + 64 rope
        of the un-absorbed head)."""
        d = 192 if self.mla else self.D
        return float(np.float32(1.0 / np.sqrt(np.float64(d))))

    @property
    def prob_scale(self) -> float:
        return float(np.float32(1.0 / 448.0)) if self.prob_fp8 else 0.0

    def chan_mask(self) -> Optional[np.ndarray]:
        if self.chan_outliers == 0:
            return None
        m = np.zeros(self.D, np.uint8)
        for c in pick_channels(self.seed, self.D, self.chan_outliers):
            m[c] = 1
        return m

    def _fill(self, tensor: int, n: int, offset: int, D: int, out=None) -> np.ndarray:
        cm = self.chan_mask() if D == self.D else None
        return fill_bf16(self.seed, tensor, n, offset, D, cm, self.chan_mult, self.elem_p,
                         self.elem_mult, out)

    def q(self) -> np.ndarray:
        n = self.B * self.Hq * self.Dqk
        if self.mla:
            # the latent part and the rope part of the query are one tensor
            return fill_bf16(self.seed, T_Q, n).reshape(self.B, self.Hq, self.Dqk)
        return self._fill(T_Q, n, 0, self.D).reshape(self.B, self.Hq, self.Dqk)

    def kv_rows(self, tensor: int, b: int, t0: int = 0, t1: Optional[int] = None) -> np.ndarray:
        """Rows [t0, t1) of request b of K (tensor 1) or V (tensor 2):
        [t1-t0][Hkv][D] bf16."""
        if t1 is None:
            t1 = int(self.seq_lens[b])
        row = self.Hkv * self.D
        off = (b * self.Lmax + t0) * row
        r = self._fill(tensor, (t1 - t0) * row, off, self.D).reshape(t1 - t0, self.Hkv, self.D)
        return self._head_skew(r)

    def _head_skew(self, r: np.ndarray) -> np.ndarray:
        """Multiply kv head h of rows [T][Hkv][D] (bf16 bits) by 2^head_exp[h]:
        an exponent shift, exact while the result stays a normal bf16."""
        if not self.head_exp:
            return r
        e = np.array([self.head_exp[h % len(self.head_exp)] for h in range(self.Hkv)], np.int32)
        x = bf16_to_f32(r) * np.exp2(e.astype(np.float32))[None, :, None]
        return f32_to_bf16(x)

    def kpe_rows(self, b: int, t0: int = 0, t1: Optional[int] = None) -> np.ndarray:
        if t1 is None:
            t1 = int(self.seq_lens[b])
        off = (b * self.Lmax + t0) * self.rope
        return fill_bf16(self.seed, T_KPE, (t1 - t0) * self.rope, off).reshape(t1 - t0,
                                                                                 self.rope)

    def full(self, tensor: int) -> np.ndarray:
        """The whole [B][Lmax][Hkv][D] tensor (rows past seq_lens[b] drawn too)."""
        if tensor == T_KPE:
            n = self.B * self.Lmax * self.rope
            return fill_bf16(self.seed, T_KPE, n).reshape(self.B, self.Lmax, self.rope)
        n = self.B * self.Lmax * self.Hkv * self.D
        r = self._fill(tensor, n, 0, self.D).reshape(self.B * self.Lmax, self.Hkv, self.D)
        return self._head_skew(r).reshape(self.B, self.Lmax, self.Hkv, self.D)

    def pages_per_seq(self) -> int:
        ps = self.page_size or max(16, -(-self.Lmax // 16) * 16)
        return -(-self.Lmax // ps)

    def page_size_eff(self) -> int:
        return self.page_size or max(16, -(-self.Lmax // 16) * 16)

    def block_table(self) -> tuple[np.ndarray, int]:
        """(block_table [B][pages_per_seq] int32, num_pages).  Physical page
        ids are a random permutation of all needed pages when permute_pages."""
        ps = self.page_size_eff()
        pps = self.pages_per_seq()
        need = [-(-int(L) // ps) for L in self.seq_lens]
        total = int(sum(need))
        ids = permutation(self.seed, total) if self.permute_pages else np.arange(total,
                                                                                 dtype=np.int32)
        bt = np.zeros((self.B, pps), np.int32)
        k = 0
        for b in range(self.B):
            for p in range(need[b]):
                bt[b, p] = ids[k]
                k += 1
        return bt, max(total, 1)


def tiny_fp8(L: int = 256) -> Workload:
    """FP8 KV, batch 1, 4 query heads on 1 kv head, head_dim 64, 256 tokens,
    two outlier channels x20 shared by Q, K, V; seed 0."""
    return Workload("tiny_fp8", "fp8", 1, 4, 1, 64, np.array([L], np.int32),
                    chan_outliers=2, chan_mult=20.0, splits=(1, 2), out="f32")


def gqa_fp8(L: int = 8192) -> Workload:
    """FP8 KV, GQA 4:1: batch 2, 32 query / 8 kv heads, head_dim 128;
    1% of elements x10; bf16 output."""
    return Workload(f"gqa_fp8_L{L}", "fp8", 2, 32, 8, 128, np.array([L, L], np.int32),
                    elem_p=0.01, elem_mult=10.0, splits=(1, 2, 4, 8, 0), out="bf16")


def nvfp4(L: int = 8192) -> Workload:
    """NVFP4 KV: batch 1, 32 query / 8 kv heads, head_dim 128, N(0,1)."""
    return Workload(f"nvfp4_L{L}", "nvfp4", 1, 32, 8, 128, np.array([L], np.int32),
                    splits=(1, 2, 4, 8, 0), out="f32")


def paged_fp8_probs(B: int = 64, lo: int = 512, hi: int = 8192, seed: int = 0) -> Workload:
    """Paged FP8 KV, MHA 16 heads, head_dim 128, lengths uniform on
    {lo..hi}, 16-token pages in random physical order, FP8 probabilities and
    FP8 output."""
    lens = uniform_lengths(seed, B, lo, hi)
    return Workload("paged_fp8_probs", "fp8", B, 16, 16, 128, lens, page_size=16,
                    permute_pages=True, prob_fp8=True, out="e4m3", splits=(1, 0), seed=seed)


def gqa_fp8_batch(B: int, L: int) -> Workload:
    """The GQA FP8 shapes and values with a larger batch (B requests of L
    tokens): a decode step with enough bytes that the launch's fixed latency
    is a small part of it."""
    w = gqa_fp8(L)
    w.name = f"gqa_fp8_B{B}_L{L}"
    w.B = B
    w.seq_lens = np.full(B, L, np.int32)
    return w


def gqa_fp8_head_scales(L: int = 8192) -> Workload:
    """The GQA FP8 workload with per-kv-head static scales (compressed-tensors
    PR 436 "attn_head" strategy): same shapes and values, one scale per kv
    head from that head's amax."""
    w = gqa_fp8(L)
    w.name = f"gqa_fp8_head_L{L}"
    w.head_scales = True
    return w


def gqa_fp8_query(L: int = 8192) -> Workload:
    """The GQA FP8 workload with an FP8 query (compressed-tensors PR 436
    "QKV-FP8-Tensor": a static per-tensor query scale from its amax)."""
    w = gqa_fp8(L)
    w.name = f"gqa_fp8_q8_L{L}"
    w.q_fp8 = True
    return w


def mla_nvfp4(B: int = 32, L: int = 4096) -> Workload:
    """MLA absorbed decode: 16 heads on one NVFP4 latent cache (512) plus a
    bf16 rope key (64); scale 1/sqrt(192)."""
    return Workload("mla_nvfp4", "nvfp4", B, 16, 1, 512, np.full(B, L, np.int32), rope=64,
                    splits=(1, 0), out="f32")
