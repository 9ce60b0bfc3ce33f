"""Benchmark: split-KV decode over a quantized KV cache on one GB300.

One step = the whole decode hot path for one new token per request:
quantize-on-append of the new K/V rows, then the split-KV decode with its
combine in one launch (kvq_decode; split count from kvq_auto_splits), over a
cache of kv_len tokens per request that is resident in HBM.  The headline workload is GQA
4:1 FP8: batch 2, 32 query / 8 kv heads, head_dim 128, kv_len 32768, 1% of
elements x10, bf16 output.

Timing: W warm-up steps, then K timed steps; before every timed step the L2
is flushed by writing one 256 MiB buffer and then reading another (the read
evicts the written lines, so the timed step neither finds its data in L2 nor
pays for write-backs of the flush), and each step is bracketed by CUDA events
on the launch stream (the two launches are replayed as one CUDA graph).
`value` is the mean device time per step in microseconds (lower is better); KV GB/s = attended cache bytes / step time.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ours|reference]
                    [--no-sweep] [--workload gqa_fp8|nvfp4|paged_fp8_probs|mla_nvfp4]

--workload picks the workload of the main line (default: the headline GQA
FP8 workload above); the others are the sweep's workloads at their own sizes.

With --impl reference the CPU oracle is timed on the same workload on the
host cores (the reference arm); under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("decode-attention µs/step and KV-cache GB/s (% of GB300 HBM peak) vs kv_len")
HEADLINE_L = 32768
FLUSH_BYTES = 256 << 20


def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


# ---------------------------------------------------------------------------
# peaks, clocks, ncu traffic
# ---------------------------------------------------------------------------

def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


KERNEL_SOURCES = {
    "decode": ["kvq_decode.cuh", "kvq_decode.cu", "kvq_decode_nvfp4.cu", "kvq_attn.cuh",
               "kvq_device.cuh", "kvq_internal.h"],
    "mla": ["kvq_mla.cu", "kvq_attn.cuh", "kvq_device.cuh", "kvq_internal.h"],
}


def kernel_source_hash(kind: str = "decode"):
    """Hash of the kernel sources with comments and whitespace removed (the
    counters of a capture depend on the code only)."""
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "quantized_kv_cache_05_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, kind: str = "decode"):
    """DRAM bytes per launch of the decode kernel from the committed ncu
    summary, when it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("source_hash") == kernel_source_hash(kind):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        time.sleep(0.25)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(value: float, device=None) -> float:
    """Largest per-rank value (the job's time is its slowest replica).  Works
    with NCCL (device tensor) and gloo (CPU tensor)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

class Bench:
    def __init__(self, w, device, splits=0):
        import torch
        from quantized_kv_cache_05_gb300 import kvq, runtime, synth
        self.torch, self.kvq, self.runtime, self.synth = torch, kvq, runtime, synth
        self.w, self.device = w, device
        torch.cuda.set_device(device)
        self.stream = torch.cuda.Stream(device)
        B, Hkv, D, L = w.B, w.Hkv, w.D, w.Lmax
        bt, npages = w.block_table()
        ps = w.page_size_eff()
        fmt = runtime.FMT[w.fmt]
        with torch.cuda.stream(self.stream):
            # calibrate the static scales on the device (amax kernel)
            amax = {}
            self.q = self._bf16(w.q())
            tensors = [synth.T_K] if w.mla else [synth.T_K, synth.T_V]
            dev_rows = {}
            for t in tensors:
                a = torch.zeros(1, dtype=torch.float32, device=device)
                m = 0.0
                rows = []
                for b in range(B):
                    x = self._bf16(w.kv_rows(t, b))
                    kvq.check(kvq.kvq_amax_bf16(x, x.numel(), a, self.stream))
                    m = max(m, float(a.item()))
                    rows.append(x)
                amax[t] = m
                dev_rows[t] = rows
            ks = kvq.kvq_tensor_scale(fmt, amax[synth.T_K])[1]
            vs = kvq.kvq_tensor_scale(fmt, amax.get(synth.T_V, amax[synth.T_K]))[1]
            head_sc = {}
            if getattr(w, "head_scales", False):
                # per-kv-head scales: the amax kernel on each head's rows
                for t in tensors:
                    hs = []
                    for h in range(Hkv):
                        m = 0.0
                        for x in dev_rows[t]:
                            xh = x[:, h].contiguous()
                            a = torch.zeros(1, dtype=torch.float32, device=device)
                            kvq.check(kvq.kvq_amax_bf16(xh, xh.numel(), a, self.stream))
                            m = max(m, float(a.item()))
                        hs.append(kvq.kvq_tensor_scale(fmt, m)[1])
                    head_sc[t] = torch.tensor(hs, dtype=torch.float32)
            self.cache = runtime.QuantizedKVCache(w.fmt, npages, ps, Hkv, D, torch.from_numpy(bt),
                                                  ks, vs, rope_dim=w.rope, device=device,
                                                  k_head_scale=head_sc.get(synth.T_K),
                                                  v_head_scale=head_sc.get(synth.T_V))
            zero = torch.zeros(1, dtype=torch.int32, device=device)
            kpe_rows = [self._bf16(w.kpe_rows(b)) for b in range(B)] if w.mla else None
            for b in range(B):
                c = self.cache.struct()
                c.block_table = self.cache.block_table[b].data_ptr()
                k = dev_rows[synth.T_K][b][None]
                v = None if w.mla else dev_rows[synth.T_V][b][None]
                kpe = kpe_rows[b][None] if w.mla else None
                kvq.check(kvq.kvq_quantize_append(c, k, v, kpe, zero, 1, k.shape[1], self.stream))
            # the new token of each step: the last row of each request,
            # re-appended at position L_b - 1 (same work every step)
            last = [int(x) - 1 for x in w.seq_lens]
            self.k_new = torch.stack([dev_rows[synth.T_K][b][last[b]:last[b] + 1]
                                      for b in range(B)]).contiguous()
            self.v_new = None if w.mla else torch.stack(
                [dev_rows[synth.T_V][b][last[b]:last[b] + 1] for b in range(B)]).contiguous()
            self.kpe_new = torch.stack([kpe_rows[b][last[b]:last[b] + 1]
                                        for b in range(B)]).contiguous() if w.mla else None
            self.start_pos = torch.tensor(last, dtype=torch.int32, device=device)
            self.seq_lens = torch.from_numpy(np.ascontiguousarray(w.seq_lens, np.int32)).to(device)
            del dev_rows, kpe_rows
            # the step's inputs (q and the new K/V rows) as views of one device
            # buffer, so that the end-to-end step moves them with one copy
            self._pack_inputs()
        self.stream.synchronize()
        self.q_scale = 1.0
        self.q_codes = None
        if getattr(w, "q_fp8", False):
            # FP8 query: per-tensor scale from the amax kernel, codes from
            # kvq_quantize_fp8 (the step then reads the codes)
            with torch.cuda.stream(self.stream):
                a = torch.zeros(1, dtype=torch.float32, device=device)
                kvq.check(kvq.kvq_amax_bf16(self.q, self.q.numel(), a, self.stream))
                self.q_scale = kvq.kvq_tensor_scale(kvq.KVQ_FP8_E4M3, float(a.item()))[1]
                self.q_codes = torch.empty(self.q.shape, dtype=torch.uint8, device=device)
                kvq.check(kvq.kvq_quantize_fp8(self.q, self.q.numel(), self.q_scale, None, 0, 0,
                                               self.q_codes, self.stream))
            self.stream.synchronize()
        self.splits = splits or runtime.auto_splits(B, Hkv, w.G, w.Lmax, w.fmt, device)
        self.out_scale = 1.0
        if w.out == "e4m3":
            # calibrate the output scale from an fp32-output pass (amax / 448)
            cfg32 = self._cfg("f32", 1.0)
            o = runtime.decode(self.cache, self.q, self.seq_lens, cfg32, None, None, self.stream)
            a = torch.zeros(1, dtype=torch.float32, device=device)
            ob = o.to(torch.bfloat16)   # amax over bf16-rounded outputs (calibration only)
            kvq.check(kvq.kvq_amax_bf16(ob, ob.numel(), a, self.stream))
            self.out_scale = kvq.kvq_tensor_scale(kvq.KVQ_FP8_E4M3, float(a.item()) * 1.01)[1]
        self.cfg = self._cfg(w.out, self.out_scale)
        self.ws = runtime.FusedWorkspace(self.cfg, w.Hkv, device)
        self.flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.flush_rd = torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.flush_sink = torch.zeros(1, dtype=torch.float32, device=device)
        self.graph_step = self._capture(full=True)
        self.graph_partial = self._capture(full=False)

    def _pack_inputs(self):
        t = self.torch
        parts = [x for x in (self.q, self.k_new, self.v_new, self.kpe_new) if x is not None]
        offs, n = [], 0
        for x in parts:
            offs.append(n)
            n += (x.numel() * x.element_size() + 255) // 256 * 256
        self.inputs = t.empty(n, dtype=t.uint8, device=self.device)
        views = []
        for x, o in zip(parts, offs):
            v = self.inputs[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape)
            v.copy_(x)
            views.append(v)
        it = iter(views)
        self.q = next(it)
        self.k_new = next(it)
        self.v_new = next(it) if self.v_new is not None else None
        self.kpe_new = next(it) if self.kpe_new is not None else None

    def _bf16(self, a):
        t = self.torch
        a = np.ascontiguousarray(a, np.uint16)
        return t.from_numpy(a.view(np.int16)).to(self.device, non_blocking=False).view(t.bfloat16)

    def _cfg(self, out, out_scale):
        w = self.w
        cfg = self.runtime.DecodeConfig(w.B, w.Hq, w.Dqk, w.Dv, getattr(self, "splits", 1),
                                        w.Lmax, w.sm_scale, w.prob_scale, out, out_scale)
        if getattr(self, "q_codes", None) is not None:
            cfg.q_fp8, cfg.q_scale = True, self.q_scale
        return cfg

    def _launch(self, full: bool, stream, io=None):
        """full: append + kvq_decode (one step); else kvq_decode alone.  io:
        (q, k_new, v_new, kpe_new, out) to use instead of the device tensors
        (e.g. pinned host memory)."""
        kvq = self.kvq
        c = self.cache.struct()
        p = self.cfg.params(self.seq_lens)
        q, k, v, kpe, out = io or (self.q, self.k_new, self.v_new, self.kpe_new, self.ws.out)
        if self.q_codes is not None and io is None:
            q = self.q_codes
        if full:
            kvq.check(kvq.kvq_quantize_append(c, k, v, kpe, self.start_pos, self.w.B, 1, stream))
            p.fresh_tokens = 1   # the decode overlaps with the append of the last position
        kvq.check(kvq.kvq_decode(c, p, q, self.ws.part_o, self.ws.part_lse, self.ws.counters,
                                 out, stream))

    def _launch_prefill(self, full: bool, stream):
        """The same step with the non-split prefill kernel (kvq_prefill, one
        query token per request) in place of the split decode."""
        kvq = self.kvq
        c = self.cache.struct()
        p = self.cfg.params(self.seq_lens)
        if full:
            kvq.check(kvq.kvq_quantize_append(c, self.k_new, self.v_new, self.kpe_new,
                                              self.start_pos, self.w.B, 1, stream))
        kvq.check(kvq.kvq_prefill(c, p, 1, self.q, self.ws.out, stream))

    def time_prefill(self, steps: int, warmup: int):
        """(step us: append + prefill as one graph, kernel us: one direct call)."""
        t = self.torch
        with t.cuda.stream(self.stream):
            self._launch_prefill(True, self.stream)
        self.stream.synchronize()
        g = t.cuda.CUDAGraph()
        with t.cuda.graph(g, stream=self.stream):
            self._launch_prefill(True, t.cuda.current_stream())
        step = statistics.mean(self.time_graph(g, steps, warmup))
        times = []
        with t.cuda.stream(self.stream):
            for i in range(warmup + steps):
                self.flush_l2(i)
                e0 = t.cuda.Event(enable_timing=True)
                e1 = t.cuda.Event(enable_timing=True)
                e0.record(self.stream)
                self._launch_prefill(False, self.stream)
                e1.record(self.stream)
                if i >= warmup:
                    times.append((e0, e1))
        self.stream.synchronize()
        return step, statistics.mean([a.elapsed_time(b) * 1e3 for a, b in times])

    def _capture(self, full: bool):
        t = self.torch
        with t.cuda.stream(self.stream):
            self._launch(full, self.stream)     # warm (sets kernel attributes)
        self.stream.synchronize()
        g = t.cuda.CUDAGraph()
        with t.cuda.graph(g, stream=self.stream):
            self._launch(full, t.cuda.current_stream())
        return g

    def flush_l2(self, i: int):
        """Evict L2: write a 256 MiB buffer, then read a second one so the
        dirty lines are written back before the timed step."""
        self.flush.fill_(float(i))
        torch = self.torch
        torch.sum(self.flush_rd, dim=0, keepdim=True, out=self.flush_sink)

    def time_graph(self, g, steps: int, warmup: int):
        t = self.torch
        times = []
        with t.cuda.stream(self.stream):
            for i in range(warmup + steps):
                self.flush_l2(i)
                e0 = t.cuda.Event(enable_timing=True)
                e1 = t.cuda.Event(enable_timing=True)
                e0.record(self.stream)
                g.replay()
                e1.record(self.stream)
                if i >= warmup:
                    times.append((e0, e1))
        self.stream.synchronize()
        return [a.elapsed_time(b) * 1e3 for a, b in times]   # microseconds

    def time_plain(self, full: bool, steps: int, warmup: int):
        """The same step launched directly through the API (no CUDA graph)."""
        t = self.torch
        times = []
        with t.cuda.stream(self.stream):
            for i in range(warmup + steps):
                self.flush_l2(i)
                e0 = t.cuda.Event(enable_timing=True)
                e1 = t.cuda.Event(enable_timing=True)
                e0.record(self.stream)
                self._launch(full, self.stream)
                e1.record(self.stream)
                if i >= warmup:
                    times.append((e0, e1))
        self.stream.synchronize()
        return [a.elapsed_time(b) * 1e3 for a, b in times]

    def e2e(self, steps: int, warmup: int):
        """Through the public API with host buffers: one pinned H2D copy of the
        step's q and new K/V rows (packed), append + kvq_decode, D2H of the
        output."""
        t = self.torch
        hin = self.inputs.cpu().pin_memory()   # q and the new K/V rows, packed
        hout = t.empty(self.ws.out.shape, dtype=self.ws.out.dtype).pin_memory()
        bi = hin.numel()
        bo = hout.numel() * hout.element_size()
        times = []
        with t.cuda.stream(self.stream):
            for i in range(warmup + steps):
                self.flush_l2(i)
                e0 = t.cuda.Event(enable_timing=True)
                e1 = t.cuda.Event(enable_timing=True)
                e0.record(self.stream)
                self.inputs.copy_(hin, non_blocking=True)
                self._launch(True, self.stream)
                hout.copy_(self.ws.out, non_blocking=True)
                e1.record(self.stream)
                e1.synchronize()
                if i >= warmup:
                    times.append(e0.elapsed_time(e1) * 1e3)
        return statistics.mean(times), bi, bo

    def e2e_zero_copy(self, steps: int, warmup: int):
        """Through the public API with host buffers read and written in place:
        q and the new K/V rows in pinned host memory (packed), the output too;
        the kernels reach them over the CPU-GPU link (no separate copies)."""
        t = self.torch
        hin = self.inputs.cpu().pin_memory()
        hout = t.empty(self.ws.out.shape, dtype=self.ws.out.dtype).pin_memory()
        views, off = [], 0
        for x in (self.q, self.k_new, self.v_new, self.kpe_new):
            if x is None:
                views.append(None)
                continue
            o = x.data_ptr() - self.inputs.data_ptr()
            views.append(hin[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape))
        io = (views[0], views[1], views[2], views[3], hout)
        times = []
        with t.cuda.stream(self.stream):
            for i in range(warmup + steps):
                self.flush_l2(i)
                e0 = t.cuda.Event(enable_timing=True)
                e1 = t.cuda.Event(enable_timing=True)
                e0.record(self.stream)
                self._launch(True, self.stream, io)
                e1.record(self.stream)
                e1.synchronize()
                if i >= warmup:
                    times.append(e0.elapsed_time(e1) * 1e3)
        same = bool(t.equal(hout, self.ws.out.cpu()))
        return statistics.mean(times), hin.numel(), hout.numel() * hout.element_size(), same

    def kv_bytes(self) -> int:
        """Attended cache bytes per step: codes (+ block scales, + rope keys)."""
        w = self.w
        tok = int(np.sum(w.seq_lens))
        if w.mla:
            per = w.D // 2 + w.D // 16 + 2 * w.rope
        else:
            row = w.D if w.fmt == "fp8" else w.D // 2 + w.D // 16
            per = 2 * w.Hkv * row
        return tok * per

    def table_bytes(self) -> int:
        """Block-table entries the decode reads: one 4-byte entry per page of
        each request, once per kv head (each (request, kv head) CTA group
        reads its own chunks' entries)."""
        w = self.w
        ps = w.page_size_eff()
        pages = int(sum(-(-int(L) // ps) for L in w.seq_lens))
        return pages * 4 * (1 if w.mla else w.Hkv)

    def algorithmic_bytes(self) -> int:
        """Algorithmic HBM bytes of one decode launch: the attended cache
        bytes (codes, block scales, rope keys) and the block-table entries.
        The split partials, q and the output are reported separately."""
        return self.kv_bytes() + self.table_bytes()

    def side_bytes(self) -> dict:
        """Bytes one kvq_decode launch moves besides the algorithmic ones."""
        w = self.w
        return {"split_partials": 2 * w.B * w.Hq * self.splits * (w.Dv + 1) * 4,
                "q": w.B * w.Hq * w.Dqk * 2,
                "out": w.B * w.Hq * w.Dv * self.ws.out.element_size()}


def _workloads():
    from quantized_kv_cache_05_gb300 import synth
    return {
        "gqa_fp8": {
            "make": lambda L: synth.gqa_fp8(L), "kind": "decode",
            "kernel": "partial_kernel<FP8,128> (kvq_decode, fused combine)",
            "dtype": "fp8_e4m3 KV codes -> f16 mma.sync, f32 accumulate",
            "data": "synthetic (seeded bf16 N(0,1), 1% x10 outliers)",
            "desc": lambda w: (f"gqa_fp8: batch {w.B}, Hq {w.Hq}, Hkv {w.Hkv}, head_dim {w.D}, "
                               f"kv_len {int(w.Lmax)}, FP8 E4M3 per-tensor KV, bf16 out, s=auto")},
        "nvfp4": {
            "make": lambda L: synth.nvfp4(L), "kind": "decode",
            "kernel": "partial_kernel<NVFP4,128> (kvq_decode, fused combine)",
            "dtype": "nvfp4 (e2m1 + e4m3 block scales) KV -> f16 mma.sync, f32 accumulate",
            "data": "synthetic (seeded bf16 N(0,1))",
            "desc": lambda w: (f"nvfp4: batch {w.B}, Hq {w.Hq}, Hkv {w.Hkv}, head_dim {w.D}, "
                               f"kv_len {int(w.Lmax)}, NVFP4 KV, f32 out, s=auto")},
        "paged_fp8_probs": {
            "make": lambda L: synth.paged_fp8_probs(), "kind": "decode",
            "kernel": "partial_kernel<FP8,128,probq> (kvq_decode, fused combine)",
            "dtype": "fp8_e4m3 KV and probabilities -> f16 mma.sync, f32 accumulate",
            "data": "synthetic (seeded bf16 N(0,1); lengths uniform 512..8192)",
            "desc": lambda w: (f"paged_fp8_probs: batch {w.B}, MHA {w.Hq} heads, head_dim {w.D}, "
                               f"16-token pages in random order, FP8 probabilities, E4M3 out, s=auto")},
        "mla_nvfp4": {
            "make": lambda L: synth.mla_nvfp4(), "kind": "mla",
            "kernel": "mla_tc_kernel (tcgen05, kvq_decode with fused combine)",
            "dtype": "nvfp4 latent -> f16 tcgen05.mma, bf16 rope, f32 accumulate in TMEM",
            "data": "synthetic (seeded bf16 N(0,1))",
            "desc": lambda w: (f"mla_nvfp4: batch {w.B}, 16 heads, NVFP4 latent 512 + bf16 rope 64, "
                               f"kv_len {int(w.Lmax)}, f32 out, s=auto")},
    }


WORKLOADS = None


def run_ours(args):
    import torch
    import torch.distributed as dist
    from quantized_kv_cache_05_gb300 import synth

    rank, world = env_int("RANK", 0), env_int("WORLD_SIZE", 1)
    local = env_int("LOCAL_RANK", 0)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    spec = WORKLOADS[args.workload]
    w = spec["make"](args.kv_len)
    bench = Bench(w, device)
    peak, peak_kind = hbm_peak()

    # --- timed region: K graph replays of the whole step
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        step_us = bench.time_graph(bench.graph_step, args.steps, args.warmup)
        part_us = bench.time_graph(bench.graph_partial, args.steps, args.warmup)
        plain_us = bench.time_plain(True, args.steps, args.warmup)
        part_plain_us = bench.time_plain(False, args.steps, args.warmup)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    us = max_over_ranks(statistics.mean(step_us), device)
    e2e_us, bi, bo = bench.e2e(max(10, args.steps // 2), args.warmup)
    zc_us, zbi, zbo, zc_same = bench.e2e_zero_copy(max(10, args.steps // 2), args.warmup)
    # the roofline kernel timed as a user launches it: one direct kvq_decode
    # call between two events on its stream (the graph-replayed figure is
    # reported beside it and carries the graph launch on top)
    part = statistics.mean(part_plain_us)
    achieved = bench.algorithmic_bytes() / (part * 1e-6) / 1e9
    traffic = ncu_traffic(w.name, spec["kind"])
    kvb = bench.kv_bytes()
    line = {
        "metric": METRIC,
        "value": round(us, 3),
        "unit": "us/step",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(us / 1e3, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": spec["dtype"],
        "data": spec["data"],
        "config": {
            "workload": spec["desc"](w),
            "batch": w.B, "kv_len": int(w.Lmax), "splits": bench.splits,
            "step": "append 1 token + kvq_decode (partial with fused combine, overlapping the append: fresh_tokens=1), one CUDA graph",
            "l2": "flushed before every timed step (256 MiB write, then 256 MiB read)",
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "kv_bytes_per_step": kvb,
        "kv_gbs": round(kvb / (us * 1e-6) / 1e9, 1),
        "kv_hbm_frac": round(kvb / (us * 1e-6) / 1e9 / peak, 4),
        "step_stats_us": pct(step_us),
        "plain_launch_us": pct(plain_us),
        "partial_us": round(part, 3),
        "partial_graph_us": round(statistics.mean(part_us), 3),
        "roofline": {
            "kernel": spec["kernel"],
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "algorithmic_bytes_per_launch": bench.algorithmic_bytes(),
            "algorithmic_bytes": "attended KV codes + block scales + rope keys + block-table entries",
            "other_bytes_per_launch": bench.side_bytes(),
            "traffic": traffic,
        },
        "e2e": {"value": round(e2e_us, 3), "unit": "us/step", "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo,
                "method": "one pinned H2D copy of q + new K/V rows, append + kvq_decode, one D2H copy"},
        "e2e_zero_copy": {"value": round(zc_us, 3), "unit": "us/step", "h2d_bytes_per_step": zbi,
                          "d2h_bytes_per_step": zbo, "output_matches_device_run": zc_same,
                          "method": "kernels read q + new K/V rows from pinned host memory and "
                                    "write the output there (NVLink-C2C), no separate copies"},
        # graph step (append + decode), graph partial (decode), plain step, plain partial
        "gpu_launches": 2 * args.steps + args.steps + 2 * args.steps + args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_sweep:
        line["sweep"] = sweep(device, args)
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(w, bench, seconds=args.cpu_seconds)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def pct(xs):
    """mean, median, p10 and p90 of per-step times (microseconds)."""
    a = np.asarray(xs, dtype=np.float64)
    return {"mean": round(float(a.mean()), 3), "median": round(float(np.median(a)), 3),
            "p10": round(float(np.percentile(a, 10)), 3),
            "p90": round(float(np.percentile(a, 90)), 3), "n": int(a.size)}


def sweep(device, args):
    """Partial + combine (+ append) per workload, kv_len and split count."""
    from quantized_kv_cache_05_gb300 import synth
    peak, _ = hbm_peak()
    res = []
    plans = [("gqa_fp8", synth.gqa_fp8, [1024, 8192, 32768], [1, 2, 4, 8, 0]),
             ("nvfp4", synth.nvfp4, [2048, 8192, 32768], [1, 2, 4, 8, 0]),
             ("paged_fp8_probs", lambda L: synth.paged_fp8_probs(), [0], [1, 2, 0]),
             ("mla_nvfp4", lambda L: synth.mla_nvfp4(), [0], [1, 2, 4, 8, 0]),
             ("gqa_fp8_head_scales", synth.gqa_fp8_head_scales, [8192, 32768], [0]),
             ("gqa_fp8_query", synth.gqa_fp8_query, [8192, 32768], [0]),
             # larger batches of the GQA FP8 shape: bandwidth sustained once the
             # step's bytes dwarf its fixed latency (not one of the five configs)
             ("gqa_fp8_B16", lambda L: synth.gqa_fp8_batch(16, L), [8192], [0]),
             ("gqa_fp8_B8", lambda L: synth.gqa_fp8_batch(8, L), [32768], [0])]
    for name, mk, lens, splits in plans:
        for L in lens:
            w = mk(L) if L else mk(None)
            base = None
            for s in splits:
                try:
                    b = Bench(w, device, splits=s) if base is None else base.with_splits(s)
                except Exception as e:   # unsupported split for this workload
                    res.append({"workload": name, "kv_len": L, "s": s, "error": str(e)[:120]})
                    continue
                base = base or b
                st = b.time_graph(b.graph_step, args.sweep_steps, 3)
                us = statistics.mean(st)
                ku = statistics.mean(b.time_plain(False, args.sweep_steps, 3))
                kvb = b.kv_bytes()
                ab = b.algorithmic_bytes()
                res.append({"workload": name, "kv_len": L or int(w.Lmax), "s": s or "auto",
                            "splits": b.splits, "us_per_step": round(us, 2),
                            "kv_gbs": round(kvb / (us * 1e-6) / 1e9, 1),
                            "kv_hbm_frac": round(kvb / (us * 1e-6) / 1e9 / peak, 3),
                            "kernel_us": round(ku, 2),
                            "kernel_hbm_frac": round(ab / (ku * 1e-6) / 1e9 / peak, 3)})
            if base is not None and name in ("gqa_fp8", "nvfp4"):
                # the pages' comparison: the non-split prefill kernel on the
                # same decode step (one query token per request)
                us, ku = base.time_prefill(args.sweep_steps, 3)
                kvb = base.kv_bytes()
                res.append({"workload": name, "kv_len": L, "s": "prefill",
                            "us_per_step": round(us, 2),
                            "kv_gbs": round(kvb / (us * 1e-6) / 1e9, 1),
                            "kv_hbm_frac": round(kvb / (us * 1e-6) / 1e9 / peak, 3),
                            "kernel_us": round(ku, 2),
                            "kernel_hbm_frac": round(base.algorithmic_bytes() / (ku * 1e-6) / 1e9
                                                     / peak, 3)})
            del base
    return res


def _with_splits(self, s):
    import copy
    nb = copy.copy(self)
    nb.splits = s or self.runtime.auto_splits(self.w.B, self.w.Hkv, self.w.G, self.w.Lmax,
                                              self.w.fmt, self.device)
    nb.cfg = nb._cfg(self.w.out, self.out_scale)
    nb.ws = self.runtime.FusedWorkspace(nb.cfg, self.w.Hkv, self.device)
    nb.graph_step = nb._capture(full=True)
    nb.graph_partial = None
    return nb


Bench.with_splits = _with_splits


# ---------------------------------------------------------------------------
# the CPU oracle (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_step_time(w, groups, nthreads, s=1):
    """Seconds for the oracle's decode step on the given (request, kv head)
    groups: quantize the step's new K/V row (the one-token append), dequantize
    the group's cached codes (FP8, or NVFP4; MLA: the latent plus the bf16 rope
    keys) and run exact attention for its query heads, or the FP8-probability
    reading with s splits.  Quantizing the rest of the cache is setup and not
    timed; the per-tensor scales come from the sampled requests."""
    import concurrent.futures
    import oracle
    from quantized_kv_cache_05_gb300 import synth

    q = synth.bf16_to_f32(w.q()).astype(np.float64)
    reqs = sorted({b for b, _ in groups})
    k_rows = {b: w.kv_rows(synth.T_K, b) for b in reqs}
    v_rows = None if w.mla else {b: w.kv_rows(synth.T_V, b) for b in reqs}
    tensor_scale = oracle.fp8_tensor_scale if w.fmt == "fp8" else oracle.nvfp4_global_scale
    ks = tensor_scale(max(oracle.amax_bf16(k_rows[b]) for b in reqs))
    vs = ks if w.mla else tensor_scale(max(oracle.amax_bf16(v_rows[b]) for b in reqs))

    def quant(x, scale):
        return (oracle.fp8_quantize(x, scale), None) if w.fmt == "fp8" else \
            oracle.nvfp4_quantize(x, scale)

    def dequant(cb, scale):
        codes, bs = cb
        return oracle.fp8_dequant(codes, scale) if w.fmt == "fp8" else \
            oracle.nvfp4_dequant(codes, bs, scale)

    codes = {}
    for b, h in groups:
        kc = quant(k_rows[b][:, h], ks)
        vc = None if w.mla else quant(v_rows[b][:, h], vs)
        kpe = w.kpe_rows(b) if w.mla else None
        codes[(b, h)] = (kc, vc, kpe)
    mode = 1 if w.prob_fp8 else 0

    # the step's append: the new token's K/V row of each group (its last row)
    new_rows = {(b, h): (k_rows[b][-1:, h], None if w.mla else v_rows[b][-1:, h])
                for b, h in groups}

    def one(bh):
        b, h = bh
        kn, vn = new_rows[bh]
        quant(kn, ks)
        if vn is not None:
            quant(vn, vs)
        kc, vc, kpe = codes[bh]
        kh = dequant(kc, ks)
        if w.mla:
            vh = kh
            kh = np.concatenate([kh, synth.bf16_to_f32(kpe).astype(np.float64)], axis=1)
        else:
            vh = dequant(vc, vs)
        qs = q[b, h * w.G:(h + 1) * w.G][None]
        oracle.decode_batch(qs, kh[None, None], vh[None, None], np.array([kh.shape[0]]),
                            w.sm_scale, mode=mode, s=s, prob_scale=w.prob_scale, nthreads=1)

    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(nthreads) as ex:
        list(ex.map(one, groups))
    return time.perf_counter() - t0


def cpu_baseline(w, bench=None, seconds=10.0):
    nthreads = os.cpu_count() or 1
    s = bench.splits if (bench is not None and w.prob_fp8) else 1
    all_groups = [(b, h) for b in range(w.B) for h in range(w.Hkv)]
    # size the sample: time one group, then take as many as fit the budget
    t1 = oracle_step_time(w, all_groups[:1], 1, s)
    n = int(max(1, min(len(all_groups), seconds / max(t1, 1e-6) * nthreads / 2)))
    sample = all_groups[:n]
    reps, tot = 0, 0.0
    while tot < seconds / 2 and reps < 50:
        tot += oracle_step_time(w, sample, nthreads, s)
        reps += 1
    per_step = tot / reps * len(all_groups) / len(sample)
    return {"value": round(per_step * 1e6, 1), "unit": "us/step", "cores": nthreads,
            "kind": "oracle",
            "sample": f"{len(sample)} of {len(all_groups)} (request, kv head) groups, "
                      f"{reps} repetitions, scaled to the whole step; each group: quantize "
                      f"its new K/V row, dequantize its cache, exact attention"}


def run_reference(args):
    """The oracle, as it stands, on this arm's workload (host cores; rank 0
    only).  FP8-probability mode is timed with one chunk per request: the
    oracle's work per token does not depend on the split count."""
    rank = env_int("RANK", 0)
    if rank != 0:
        return
    spec = WORKLOADS[args.workload]
    w = spec["make"](args.kv_len)
    nthreads = os.cpu_count() or 1
    groups = [(b, h) for b in range(w.B) for h in range(w.Hkv)]
    t1 = oracle_step_time(w, groups[:1], 1)
    n = int(max(1, min(len(groups), 2.0 / max(t1, 1e-6) * nthreads / 2)))
    sample = groups[:n]
    for _ in range(args.warmup if args.warmup < 3 else 1):
        oracle_step_time(w, sample, nthreads)
    times = [oracle_step_time(w, sample, nthreads) * len(groups) / len(sample)
             for _ in range(args.steps)]
    us = statistics.mean(times) * 1e6
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(us, 1), "unit": "us/step", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": spec["data"],
        "config": {"workload": spec["desc"](w), "batch": w.B, "kv_len": int(w.Lmax),
                   "step": "fp64 oracle: dequantize the cache, attention per (request, kv head)",
                   "parallelism": f"{nthreads} host threads"},
        "cpu_baseline": {"value": round(us, 1), "unit": "us/step", "cores": nthreads,
                         "kind": "oracle",
                         "sample": f"{len(sample)} of {len(groups)} (request, kv head) groups "
                                   f"per step, scaled to the whole step"},
        "e2e": {"value": round(us, 1), "unit": "us/step", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--kv-len", type=int, default=HEADLINE_L)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--sweep-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--workload", default="gqa_fp8",
                    choices=["gqa_fp8", "nvfp4", "paged_fp8_probs", "mla_nvfp4"])
    args = ap.parse_args()
    global WORKLOADS
    WORKLOADS = _workloads()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
