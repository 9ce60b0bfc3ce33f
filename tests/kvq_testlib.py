"""Test plumbing: the same seeded workload set up on the GPU (through the C
ABI) and in the oracle, plus the comparison rules.

Comparison rules (floating point):
  * fp32 output: max |gpu - oracle| <= 2e-3 and cosine >= 0.9999 over the
    whole output;
  * bf16 output: within one bf16 step of bf16_rne(oracle), or within 2e-3;
  * E4M3 output: codes equal, or one code step apart where the oracle's
    pre-rounding value lies within 1e-3 (relative) of the rounding midpoint.
Integer / byte work (codes, block scales) must be bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from quantized_kv_cache_05_gb300 import kvq, runtime, synth

F32_ATOL = 2e-3
COS_MIN = 0.9999


def to_dev_bf16(a: np.ndarray, device="cuda") -> torch.Tensor:
    a = np.ascontiguousarray(a, np.uint16)
    return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


class Setup:
    """Workload `w` quantized into a device cache, with the oracle's view."""

    def __init__(self, w: synth.Workload, device="cuda", oracle_heads=None):
        self.w = w
        self.device = device
        B, Hkv, D = w.B, w.Hkv, w.D
        bt, npages = w.block_table()
        self.bt = bt
        self.ps = w.page_size_eff()
        self.q = w.q()
        self.k = [w.kv_rows(synth.T_K, b) for b in range(B)]
        self.v = None if w.mla else [w.kv_rows(synth.T_V, b) for b in range(B)]
        self.kpe = [w.kpe_rows(b) for b in range(B)] if w.mla else None

        # --- static scales: oracle (reference) and GPU amax kernel (product)
        amax_k = max(oracle.amax_bf16(x) for x in self.k)
        amax_v = max(oracle.amax_bf16(x) for x in self.v) if self.v else amax_k
        sc = oracle.fp8_tensor_scale if w.fmt == "fp8" else oracle.nvfp4_global_scale
        self.k_scale, self.v_scale = sc(amax_k), sc(amax_v)
        fmt = runtime.FMT[w.fmt]
        self.gpu_amax_k = self._gpu_amax(self.k)
        self.gpu_amax_v = self._gpu_amax(self.v) if self.v else self.gpu_amax_k
        st1, gk = kvq.kvq_tensor_scale(fmt, self.gpu_amax_k)
        st2, gv = kvq.kvq_tensor_scale(fmt, self.gpu_amax_v)
        kvq.check(st1)
        kvq.check(st2)
        self.gpu_k_scale, self.gpu_v_scale = gk, gv
        # per-kv-head scales ("attn_head"): oracle over all requests' rows of a
        # head; product: the amax kernel on each head's rows, then the scale call
        self.k_head = self.v_head = None
        khs = vhs = None
        if getattr(w, "head_scales", False):
            hsc = oracle.fp8_head_scales if w.fmt == "fp8" else oracle.nvfp4_head_scales
            kall = np.concatenate(self.k, axis=0)
            vall = np.concatenate(self.v, axis=0)
            self.k_head, self.v_head = hsc(kall), hsc(vall)
            khs = self._gpu_head_scales(kall, fmt)
            vhs = self._gpu_head_scales(vall, fmt)
            assert np.array_equal(khs, self.k_head) and np.array_equal(vhs, self.v_head)
            khs, vhs = torch.from_numpy(khs), torch.from_numpy(vhs)

        # --- device cache, filled request by request through the append call
        self.cache = runtime.QuantizedKVCache(w.fmt, npages, self.ps, Hkv, D, torch.from_numpy(bt),
                                              gk, gv, rope_dim=w.rope, device=device,
                                              k_head_scale=khs, v_head_scale=vhs)
        zero = torch.zeros(1, dtype=torch.int32, device=device)
        for b in range(B):
            if int(w.seq_lens[b]) == 0:
                continue
            c = self.cache.struct()
            c.block_table = self.cache.block_table[b].data_ptr()
            k_t = to_dev_bf16(self.k[b][None], device)
            v_t = to_dev_bf16(self.v[b][None], device) if self.v else None
            kpe_t = to_dev_bf16(self.kpe[b][None], device) if self.kpe else None
            kvq.check(kvq.kvq_quantize_append(c, k_t, v_t, kpe_t, zero, 1, k_t.shape[1]),
                      "append")
        self.q_t = to_dev_bf16(self.q, device)
        self.seq_lens_t = torch.from_numpy(np.ascontiguousarray(w.seq_lens, np.int32)).to(device)
        torch.cuda.synchronize()
        self._host_cache = None

    def _gpu_head_scales(self, rows: np.ndarray, fmt: int) -> np.ndarray:
        out = []
        for h in range(rows.shape[1]):
            a = self._gpu_amax([np.ascontiguousarray(rows[:, h])])
            st, s = kvq.kvq_tensor_scale(fmt, a)
            kvq.check(st)
            out.append(s)
        return np.array(out, np.float32)

    def _gpu_amax(self, rows) -> float:
        flat = np.concatenate([r.reshape(-1) for r in rows]) if rows else np.zeros(0, np.uint16)
        x = to_dev_bf16(flat, self.device)
        out = torch.empty(1, dtype=torch.float32, device=self.device)
        kvq.check(kvq.kvq_amax_bf16(x, x.numel(), out), "amax")
        return float(out.item())

    # ----------------------------------------------------------- GPU views
    def host_cache(self):
        if self._host_cache is None:
            c = self.cache
            self._host_cache = {
                "k": c.k_codes.cpu().numpy(),
                "v": c.v_codes.cpu().numpy() if c.v_codes is not None else None,
                "ks": c.k_bscale.cpu().numpy() if c.k_bscale is not None else None,
                "vs": c.v_bscale.cpu().numpy() if c.v_bscale is not None else None,
                "kpe": bf16_bits(c.k_pe) if c.k_pe is not None else None,
            }
        return self._host_cache

    def gpu_rows(self, name: str, b: int, kvh: int = 0) -> np.ndarray:
        """Rows [0, L_b) of request b, kv head kvh, gathered via the block table."""
        L = int(self.w.seq_lens[b])
        pos = np.arange(L)
        pages = self.bt[b, pos // self.ps]
        hc = self.host_cache()[name]
        if name == "kpe":
            return hc[pages, pos % self.ps]
        return hc[pages, kvh, pos % self.ps]

    # --------------------------------------------------------- oracle view
    def oracle_scale(self, which: str, kvh: int) -> float:
        heads = self.k_head if which == "k" else self.v_head
        if heads is not None:
            return float(heads[kvh])
        return self.k_scale if which == "k" else self.v_scale

    def oracle_codes(self, which: str, b: int, kvh: int = 0):
        rows = (self.k if which == "k" else self.v)[b]
        heads = self.k_head if which == "k" else self.v_head
        if heads is not None:   # per-kv-head quantizers on all heads, this head's slice
            if self.w.fmt == "fp8":
                return oracle.fp8_quantize_heads(rows, heads)[:, kvh], None
            c, bs = oracle.nvfp4_quantize_heads(rows, heads)
            return c[:, kvh], bs[:, kvh]
        x = rows[:, kvh, :]
        s = self.k_scale if which == "k" else self.v_scale
        if self.w.fmt == "fp8":
            return oracle.fp8_quantize(x, s), None
        return oracle.nvfp4_quantize(x, s)

    def oracle_dequant(self, which: str, b: int, kvh: int = 0) -> np.ndarray:
        codes, bs = self.oracle_codes(which, b, kvh)
        s = self.oracle_scale(which, kvh)
        if self.w.fmt == "fp8":
            return oracle.fp8_dequant(codes, s)
        return oracle.nvfp4_dequant(codes, bs, s)

    def oracle_kv(self, b: int, kvh: int):
        """(K^ [L][Dqk], V^ [L][Dv]) in float64 for one (request, kv head)."""
        kh = self.oracle_dequant("k", b, kvh)
        if self.w.mla:
            kpe = synth.bf16_to_f32(self.kpe[b]).astype(np.float64)
            return np.concatenate([kh, kpe], axis=1), kh
        return kh, self.oracle_dequant("v", b, kvh)

    def q64(self) -> np.ndarray:
        return synth.bf16_to_f32(self.q).astype(np.float64)

    def oracle_decode(self, mode: int = 0, s: int = 1, heads=None):
        """Oracle outputs [B][Hq][Dv] (NaN where not computed) and lse."""
        w = self.w
        q = self.q64()
        out = np.full((w.B, w.Hq, w.Dv), np.nan)
        lse = np.full((w.B, w.Hq), np.nan)
        pairs = heads if heads is not None else [(b, h) for b in range(w.B) for h in range(w.Hkv)]
        for b, kvh in pairs:
            kh, vh = self.oracle_kv(b, kvh)
            L = int(w.seq_lens[b])
            qs = q[b, kvh * w.G:(kvh + 1) * w.G][None]
            o, l = oracle.decode_batch(qs, kh[None, None], vh[None, None], np.array([L]),
                                       w.sm_scale, mode=mode, s=s, prob_scale=w.prob_scale)
            out[b, kvh * w.G:(kvh + 1) * w.G] = o[0]
            lse[b, kvh * w.G:(kvh + 1) * w.G] = l[0]
        return out, lse

    # --------------------------------------------------------- GPU decode
    def config(self, s: int, out: str = "f32", out_scale: float = 1.0) -> runtime.DecodeConfig:
        w = self.w
        return runtime.DecodeConfig(w.B, w.Hq, w.Dqk, w.Dv, s, w.Lmax, w.sm_scale,
                                    w.prob_scale, out, out_scale)

    def gpu_decode(self, s: int, out: str = "f32", out_scale: float = 1.0):
        cfg = self.config(s, out, out_scale)
        ws = runtime.DecodeWorkspace(cfg, self.device)
        flag = torch.zeros(1, dtype=torch.int32, device=self.device)
        res = runtime.decode(self.cache, self.q_t, self.seq_lens_t, cfg, ws, flag)
        torch.cuda.synchronize()
        assert int(flag.item()) == 0, f"device error flag {int(flag.item())}"
        return res, ws


# ------------------------------------------------------------- comparisons

def assert_f32_close(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    m = ~np.isnan(ref)
    g, r = gpu[m].astype(np.float64), ref[m]
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = np.max(np.abs(g - r)) if g.size else 0.0
    cos = float(g @ r / (np.linalg.norm(g) * np.linalg.norm(r))) if np.any(r) else 1.0
    assert err <= F32_ATOL and cos >= COS_MIN, f"{what}: max-abs {err:.3g}, cosine {cos:.8f}"
    return err, cos


def _bf16_ordered(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)


def assert_bf16_close(gpu_bits: np.ndarray, ref: np.ndarray, what: str = ""):
    """Within one bf16 step of bf16_rne(oracle), or within the fp32 absolute
    tolerance (near zero a sign flip of a tiny value is many steps)."""
    m = ~np.isnan(ref)
    rb = synth.f32_to_bf16(ref[m].astype(np.float32))
    d = np.abs(_bf16_ordered(gpu_bits[m]) - _bf16_ordered(rb))
    gv = synth.bf16_to_f32(gpu_bits[m]).astype(np.float64)
    ok = (d <= 1) | (np.abs(gv - ref[m]) <= F32_ATOL)
    assert ok.all(), f"{what}: {int((~ok).sum())} bf16 outputs off (max {d[~ok].max()} steps)"
    return int((d >= 1).sum())


def assert_e4m3_close(gpu_codes: np.ndarray, ref: np.ndarray, out_scale: float, what=""):
    m = ~np.isnan(ref)
    rc = oracle.fp8_output(ref[m], out_scale)
    gc = gpu_codes[m]
    bad = np.nonzero(gc != rc)[0]
    pre = (ref[m].astype(np.float32) / np.float32(out_scale)).astype(np.float64)
    for i in bad:
        a = oracle.e4m3_decode(np.array([rc[i]], np.uint8))[0]
        bval = oracle.e4m3_decode(np.array([gc[i]], np.uint8))[0]
        vals = np.sort(oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)))
        # adjacent on the grid (same sign side)
        ia, ib = np.searchsorted(vals, abs(a)), np.searchsorted(vals, abs(bval))
        assert abs(ia - ib) <= 1 and (np.sign(a) == np.sign(bval) or a == 0 or bval == 0), \
            f"{what}: code {gc[i]:#x} vs {rc[i]:#x}"
        mid = (a + bval) / 2
        assert abs(pre[i] - mid) <= 1e-3 * max(abs(mid), 2.0 ** -9), \
            f"{what}: code flip away from a midpoint ({pre[i]} vs mid {mid})"
    return len(bad)
