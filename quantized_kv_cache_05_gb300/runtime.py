"""Device-memory plumbing around the C ABI: a paged quantized KV cache held in
torch tensors, and one decode step (partial + combine).

Marshalling only -- torch allocates memory and supplies streams; every
computation is a libkvq.so kernel.  Nothing here falls back to torch math.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

from . import kvq

FMT = {"fp8": kvq.KVQ_FP8_E4M3, "nvfp4": kvq.KVQ_NVFP4}
OUT = {"f32": kvq.KVQ_OUT_F32, "bf16": kvq.KVQ_OUT_BF16, "e4m3": kvq.KVQ_OUT_E4M3}
OUT_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.uint8}


class QuantizedKVCache:
    """Paged FP8 / NVFP4 KV cache (layout of ``kvq_cache`` in include/kvq.h).

    codes  uint8 [num_pages][Hkv][page_size][row]   row = D (FP8) or D/2 (NVFP4)
    bscale uint8 [num_pages][Hkv][page_size][D/16]  (NVFP4)
    k_pe   bf16  [num_pages][page_size][rope]       (MLA; V is the latent)
    """

    def __init__(self, fmt: str, num_pages: int, page_size: int, num_kv_heads: int,
                 head_dim: int, block_table: torch.Tensor, k_scale: float, v_scale: float,
                 rope_dim: int = 0, device: str | torch.device = "cuda",
                 k_head_scale: Optional[torch.Tensor] = None,
                 v_head_scale: Optional[torch.Tensor] = None):
        self.fmt = fmt
        self.num_pages, self.page_size = num_pages, page_size
        self.Hkv, self.D, self.rope = num_kv_heads, head_dim, rope_dim
        self.k_scale, self.v_scale = float(k_scale), float(v_scale)
        row = head_dim if fmt == "fp8" else head_dim // 2
        shape = (num_pages, num_kv_heads, page_size, row)
        self.k_codes = torch.zeros(shape, dtype=torch.uint8, device=device)
        self.v_codes = None if rope_dim else torch.zeros(shape, dtype=torch.uint8, device=device)
        self.k_bscale = self.v_bscale = None
        if fmt == "nvfp4":
            sshape = (num_pages, num_kv_heads, page_size, head_dim // 16)
            self.k_bscale = torch.zeros(sshape, dtype=torch.uint8, device=device)
            if not rope_dim:
                self.v_bscale = torch.zeros(sshape, dtype=torch.uint8, device=device)
        self.k_pe = (torch.zeros((num_pages, page_size, rope_dim), dtype=torch.bfloat16,
                                 device=device) if rope_dim else None)
        self.block_table = block_table.to(device=device, dtype=torch.int32).contiguous()
        self.max_pages_per_seq = self.block_table.shape[1]
        # per-kv-head scales (float32 [Hkv] on the device), replacing k_scale / v_scale
        def _hs(t):
            if t is None:
                return None
            t = t.to(device=device, dtype=torch.float32).contiguous()
            assert t.numel() == num_kv_heads, "one scale per kv head"
            return t
        self.k_head_scale, self.v_head_scale = _hs(k_head_scale), _hs(v_head_scale)

    @property
    def mla(self) -> bool:
        return self.rope > 0

    def struct(self) -> kvq.kvq_cache:
        c = kvq.kvq_cache()
        c.fmt = FMT[self.fmt]
        c.num_pages, c.page_size = self.num_pages, self.page_size
        c.num_kv_heads, c.head_dim = self.Hkv, self.D
        c.k_codes = self.k_codes.data_ptr()
        c.v_codes = self.v_codes.data_ptr() if self.v_codes is not None else None
        c.k_bscale = self.k_bscale.data_ptr() if self.k_bscale is not None else None
        c.v_bscale = self.v_bscale.data_ptr() if self.v_bscale is not None else None
        c.k_scale, c.v_scale = self.k_scale, self.v_scale
        c.block_table = self.block_table.data_ptr()
        c.max_pages_per_seq = self.max_pages_per_seq
        c.rope_dim = self.rope
        c.k_pe = self.k_pe.data_ptr() if self.k_pe is not None else None
        c.v_is_k_latent = 1 if self.mla else 0
        c.k_head_scale = self.k_head_scale.data_ptr() if self.k_head_scale is not None else None
        c.v_head_scale = self.v_head_scale.data_ptr() if self.v_head_scale is not None else None
        return c

    def append(self, k_new: torch.Tensor, v_new: Optional[torch.Tensor],
               start_pos: torch.Tensor, kpe_new: Optional[torch.Tensor] = None,
               stream=None) -> None:
        """k_new/v_new bf16 [B][T][Hkv][D]; start_pos int32 [B] (device)."""
        B, T = k_new.shape[0], k_new.shape[1]
        kvq.check(kvq.kvq_quantize_append(self.struct(), k_new, v_new, kpe_new, start_pos, B, T,
                                          stream), "kvq_quantize_append")


@dataclasses.dataclass
class DecodeConfig:
    batch: int
    num_q_heads: int
    qk_dim: int
    v_dim: int
    num_splits: int
    max_kv_len: int
    sm_scale: float
    prob_scale: float = 0.0
    out: str = "f32"
    out_scale: float = 1.0
    # > 0: the call right before on the stream is the append of the last
    # fresh_tokens positions, and the decode overlaps with it (kvq_decode_params)
    fresh_tokens: int = 0
    # FP8 query: q holds E4M3 codes, dequantized with q_scale or the per-head
    # q_head_scale tensor (float32 [num_q_heads] on the device)
    q_fp8: bool = False
    q_scale: float = 1.0
    q_head_scale: Optional[torch.Tensor] = None

    def params(self, seq_lens: torch.Tensor, error_flag: Optional[torch.Tensor] = None
               ) -> kvq.kvq_decode_params:
        p = kvq.kvq_decode_params()
        p.batch, p.num_q_heads = self.batch, self.num_q_heads
        p.qk_dim, p.v_dim, p.num_splits = self.qk_dim, self.v_dim, self.num_splits
        p.seq_lens = seq_lens.data_ptr()
        p.max_kv_len = self.max_kv_len
        p.sm_scale, p.prob_scale = self.sm_scale, self.prob_scale
        p.out_dtype, p.out_scale = OUT[self.out], self.out_scale
        p.error_flag = error_flag.data_ptr() if error_flag is not None else None
        p.fresh_tokens = self.fresh_tokens
        p.q_fp8 = 1 if self.q_fp8 else 0
        p.q_scale = self.q_scale
        p.q_head_scale = self.q_head_scale.data_ptr() if self.q_head_scale is not None else None
        return p


class DecodeWorkspace:
    """Split partials for one decode configuration (caller-owned scratch)."""

    def __init__(self, cfg: DecodeConfig, device="cuda"):
        rows = cfg.batch * cfg.num_q_heads * cfg.num_splits
        self.part_o = torch.empty(rows * cfg.v_dim, dtype=torch.float32, device=device)
        self.part_lse = torch.empty(rows, dtype=torch.float32, device=device)
        self.out = torch.empty((cfg.batch, cfg.num_q_heads, cfg.v_dim), dtype=OUT_TORCH[cfg.out],
                               device=device)


class FusedWorkspace(DecodeWorkspace):
    """Scratch of kvq_decode: split partials plus arrival counters, which are
    zeroed once here; every call leaves them at zero again."""

    def __init__(self, cfg: DecodeConfig, num_kv_heads: int, device="cuda"):
        super().__init__(cfg, device)
        self.counters = torch.zeros(cfg.batch * num_kv_heads, dtype=torch.int32, device=device)


def decode_fused(cache: QuantizedKVCache, q: torch.Tensor, seq_lens: torch.Tensor,
                 cfg: DecodeConfig, ws: Optional[FusedWorkspace] = None,
                 error_flag: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One decode step in one launch (kvq_decode)."""
    ws = ws or FusedWorkspace(cfg, cache.Hkv, q.device)
    p = cfg.params(seq_lens, error_flag)
    kvq.check(kvq.kvq_decode(cache.struct(), p, q, ws.part_o, ws.part_lse, ws.counters, ws.out,
                             stream), "kvq_decode")
    return ws.out


def auto_splits(batch: int, num_kv_heads: int, q_per_kv: int, max_kv_len: int, fmt: str,
                device: int | None = None) -> int:
    if device is None:
        device = torch.cuda.current_device()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    st, s = kvq.kvq_auto_splits(sms, batch, num_kv_heads, q_per_kv, max_kv_len, FMT[fmt])
    kvq.check(st, "kvq_auto_splits")
    return s


def decode(cache: QuantizedKVCache, q: torch.Tensor, seq_lens: torch.Tensor, cfg: DecodeConfig,
           ws: Optional[DecodeWorkspace] = None, error_flag: Optional[torch.Tensor] = None,
           stream=None) -> torch.Tensor:
    """One decode step: kvq_decode_partial then kvq_decode_combine."""
    ws = ws or DecodeWorkspace(cfg, q.device)
    p = cfg.params(seq_lens, error_flag)
    c = cache.struct()
    kvq.check(kvq.kvq_decode_partial(c, p, q, ws.part_o, ws.part_lse, stream),
              "kvq_decode_partial")
    kvq.check(kvq.kvq_decode_combine(p, ws.part_o, ws.part_lse, ws.out, stream),
              "kvq_decode_combine")
    return ws.out


def prefill(cache: QuantizedKVCache, q: torch.Tensor, seq_lens: torch.Tensor, cfg: DecodeConfig,
            q_len: int, out: Optional[torch.Tensor] = None,
            error_flag: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Causal prefill attention of q_len new tokens per request (kvq_prefill):
    q bf16 [batch][q_len][Hq][D] -> out [batch][q_len][Hq][D]."""
    if out is None:
        out = torch.empty((cfg.batch, q_len, cfg.num_q_heads, cfg.v_dim), dtype=OUT_TORCH[cfg.out],
                          device=q.device)
    p = cfg.params(seq_lens, error_flag)
    kvq.check(kvq.kvq_prefill(cache.struct(), p, q_len, q, out, stream), "kvq_prefill")
    return out
