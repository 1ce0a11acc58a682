#!/usr/bin/env python
"""Benchmark of the quantized-KV hot path on GB300: one JSON line on stdout.

A step is one pass of the whole path over one batch: for the decode workloads
(default c3, Llama-3.1-8B-shaped, 16 x 32768 tokens, 3.5-bit K + QJL / 3.5-bit
V) it appends one new token per sequence and runs decode attention over the
L+1 cached tokens (tq_append_decode: quantize-append, query prep, split-K
partials, merge); c1 (one head, 1024 fp32 tokens) decodes without an append.
Headline value: packed cache bytes read per decode step / step time (GB/s) on
c3; the c4, c5 and c1 decode workloads ride along under their own keys, and
the c2 quantize rate (vectors/s) under "quantize".  Inputs are synthetic
(seeded) and resident in HBM; caches under twice the L2 size get an L2 flush
before every timed step.  cpu_baseline: the fp64 oracle on the host cores
(every core, and one core alone).  --impl reference times the oracle alone on
the same workload.
"""

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from online_kv_cache_02_gb300 import workloads as wl  # noqa: E402

L2_BYTES = 129 * 2 ** 20


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="c3", choices=["c1", "c3", "c4", "c5"])
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling runs)")
    ap.add_argument("--no-quantize", action="store_true", help="skip the c2 quantize measurement")
    ap.add_argument("--only", default="", choices=["", "quantize", "search", "causal"],
                    help="quantize: run the c2 quantize measurement alone (profiling; --batch scales it)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-others", action="store_true", help="time the headline decode workload only")
    ap.add_argument("--cpu-workers", type=int, default=0, help="oracle worker processes (0: every host core)")
    return ap.parse_args(argv)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def tensor_peak():
    """Dense fp16 tensor peak in TFLOP/s: the measured bf16 burst figure (fp16 and bf16 share one rate), else the
    fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16 burst; fp16 runs at the same rate)"
    return 1900.0, "fallback"


# ---------------------------------------------------------------------------
# clocks (NVML through ctypes; read-only queries)
# ---------------------------------------------------------------------------

REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
           0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting", 0x1: "gpu_idle"}


class ClockSampler:
    def __init__(self, torch):
        self.ok = False
        self.samples = []
        self.reasons = 0
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(torch.cuda.current_device())
            bus = getattr(props, "pci_bus_id", None)
            got = 1
            if bus is not None:
                busid = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), bus, getattr(props, "pci_device_id", 0))
                got = self.nv.nvmlDeviceGetHandleByPciBusId_v2(busid.encode(), ctypes.byref(self.h))
            if got != 0:
                got = self.nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h))
            if got != 0:
                return
            mx = ctypes.c_uint()
            self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
            self.max_mhz = mx.value
            self.reason_fn = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(self.nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
        except OSError:
            pass

    def _run(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        while not self.stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) == 0:
                self.samples.append(c.value)
            if self.reason_fn(self.h, ctypes.byref(r)) == 0:
                self.reasons |= r.value
            time.sleep(0.001)

    def __enter__(self):
        if self.ok:
            self.stop = threading.Event()
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self.stop.set()
            self.t.join()

    def result(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "samples": len(self.samples),
                "reasons": [n for b, n in REASONS.items() if self.reasons & b and n != "gpu_idle"]}


def traffic_for(kernel_file, kernel, workload):
    """dram bytes per launch of `kernel` on `workload` from a committed ncu capture (profiles/ncu_traffic.json),
    or None when there is none or the kernel source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    with open(os.path.join(ROOT, "online_kv_cache_02_gb300", "csrc", kernel_file), "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    if rec.get("source_sha") != sha:
        return None
    return rec.get("bytes_per_launch", {}).get(workload)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class DecodeBench:
    """One decode workload resident on the GPU.  A step with append (c3-c5) is one tq_append_decode_ex call:
    quantize-append the new token at position L, decode over L+1; without append (c1) it is one
    tq_decode_attention_ex call over the cached tokens (its three stages one by one in the pass that times the
    partials kernel by events)."""

    def __init__(self, w, torch, tq):
        self.w, self.torch, self.tq = w, torch, tq
        dev = torch.device("cuda", torch.cuda.current_device())
        self.dev = dev
        cfg = tq.make_config(k_bits=w.k_bits, v_bits=w.v_bits, m=w.m, seed=w.seed, k_qjl=w.qjl)
        self.ctx = tq.tq_create_ex(cfg)
        B, H, Hq = w.batch, w.kv_heads, w.q_heads
        self.f32 = w.dtype == "f32"
        self.tdt = torch.float32 if self.f32 else torch.bfloat16
        self.dt = tq.TQ_F32 if self.f32 else tq.TQ_BF16
        self.lens = wl.seq_lens(w)
        self.bt = wl.block_table(w)
        self.pps = self.bt.shape[1]
        self.num_pages = B * self.pps
        kpb, vpb = tq.tq_cache_layout(self.ctx, H)
        self.kc = torch.empty(self.num_pages * kpb, dtype=torch.uint8, device=dev)
        self.vc = torch.empty(self.num_pages * vpb, dtype=torch.uint8, device=dev)
        self.bt_d = torch.from_numpy(self.bt).to(dev)
        zero = torch.zeros(1, dtype=torch.int32, device=dev)
        # history: quantize every cached token once (untimed)
        for b in range(B):
            L = int(self.lens[b])
            for s0 in range(0, L, 8192):
                n = min(8192, L - s0)
                K = torch.from_numpy(wl.kv_tokens(w, "k", b, s0, n)).to(dev).to(self.tdt)
                V = torch.from_numpy(wl.kv_tokens(w, "v", b, s0, n)).to(dev).to(self.tdt)
                zero.fill_(s0)
                tq.tq_quantize(self.ctx, K, V, self.dt, 1, n, H, zero, self.bt_d[b], self.pps, self.num_pages,
                               self.kc, self.vc)
        torch.cuda.synchronize()
        assert tq.tq_check_device_status(self.ctx) == 0
        self.append = w.append
        extra = 1 if w.append else 0
        # a step's inputs (query, and the new token's K and V) side by side in one pinned host buffer and one
        # device buffer, so the end-to-end step copies them in one transfer; each part starts 256-byte aligned
        parts = [torch.from_numpy(wl.queries(w)).to(self.tdt)]
        if w.append:
            parts += [torch.from_numpy(wl.new_tokens(w, "k")).to(self.tdt),
                      torch.from_numpy(wl.new_tokens(w, "v")).to(self.tdt)]
        esz = parts[0].element_size()
        offs, n = [], 0
        for t in parts:
            offs.append(n)
            n += -(-t.numel() * esz // 256) * 256 // esz
        self.in_h = torch.empty(n, dtype=self.tdt).pin_memory()
        for t, o in zip(parts, offs):
            self.in_h[o:o + t.numel()].copy_(t.reshape(-1))
        self.in_d = self.in_h.to(dev)
        views = [self.in_d[o:o + t.numel()].view(t.shape) for t, o in zip(parts, offs)]
        self.q = views[0]
        if w.append:
            self.knew, self.vnew = views[1], views[2]
        self.start = torch.from_numpy(self.lens.astype(np.int32)).to(dev)
        self.max_len = int(self.lens.max()) + extra
        # split-K chunk: the workload's own, else the library's choice for the actual total length
        self.chunk = w.chunk or tq.tq_decode_chunk(self.ctx, B, Hq, H, int((self.lens + extra).sum()), self.max_len,
                                                   fused_append=w.append)
        self.ws_n = tq.tq_workspace_size(self.ctx, B, Hq, self.max_len, self.chunk)
        self.ws = torch.empty(self.ws_n, dtype=torch.uint8, device=dev)
        self.out = torch.empty(B, Hq, 128, dtype=torch.float32, device=dev)
        self.out_h = torch.empty(B, Hq, 128, dtype=torch.float32).pin_memory()
        self.tokens = int((self.lens + extra).sum())
        self.bytes_step = self.tokens * H * wl.packed_bytes_per_token_head(w)
        # append (one quantize launch for K and V) + qprep + partials + merge
        self.launches_per_step = 4 if w.append else 3

    def _marshal(self, stream):
        """ctypes arguments of the per-step call, built once per stream (pointers are fixed)."""
        import ctypes
        w, tq = self.w, self.tq
        sp = stream.cuda_stream
        scale = ctypes.c_float(1.0 / math.sqrt(128))
        if self.append:
            args = [self.ctx, self.knew.data_ptr(), self.vnew.data_ptr(), self.q.data_ptr(), self.dt,
                    w.batch, w.q_heads, w.kv_heads, self.start.data_ptr(), self.max_len,
                    self.bt_d.data_ptr(), self.pps, self.num_pages, self.kc.data_ptr(), self.vc.data_ptr(),
                    self.chunk, scale, self.out.data_ptr(), self.ws.data_ptr(), self.ws_n, sp]
        else:
            args = [self.ctx, self.q.data_ptr(), self.dt, w.batch, w.q_heads, w.kv_heads, self.start.data_ptr(),
                    self.max_len, self.bt_d.data_ptr(), self.pps, self.num_pages, self.kc.data_ptr(),
                    self.vc.data_ptr(), self.chunk, scale, self.out.data_ptr(), self.ws.data_ptr(), self.ws_n]
        self._args = (stream, args, sp)

    def step(self, stream, ev=None):
        """One decode step through the C ABI; `ev` (begin, end) events bracket the partials kernel."""
        if getattr(self, "_args", (None,))[0] is not stream:
            self._marshal(stream)
        lib = self.tq._lib
        if self.append:
            handles = [None, None] if ev is None else [e.cuda_event for e in ev]
            st = lib.tq_append_decode_ex(*self._args[1], *handles)
            if st != 0:
                raise self.tq.TQError("tq_append_decode_ex", st)
            return
        args, sp = self._args[1], self._args[2]
        if ev is None:                   # the whole decode in one call, as a user makes it
            st = lib.tq_decode_attention_ex(*args, self.tq.TQ_STAGE_ALL, sp)
            if st != 0:
                raise self.tq.TQError("tq_decode_attention_ex", st)
            return
        for stage in (self.tq.TQ_STAGE_QPREP, self.tq.TQ_STAGE_PARTIALS, self.tq.TQ_STAGE_MERGE):
            if ev is not None and stage == self.tq.TQ_STAGE_PARTIALS:
                ev[0].record(stream)
            st = lib.tq_decode_attention_ex(*args, stage, sp)
            if st != 0:
                raise self.tq.TQError("tq_decode_attention_ex", st)
            if ev is not None and stage == self.tq.TQ_STAGE_PARTIALS:
                ev[1].record(stream)

    def step_e2e(self, stream):
        """One step through the public call, inputs from pinned host memory, output back to host."""
        w, tq = self.w, self.tq
        self.in_d.copy_(self.in_h, non_blocking=True)          # query and new K/V: one transfer
        if self.append:
            tq.tq_append_decode(self.ctx, self.knew, self.vnew, self.q, self.dt, w.batch, w.q_heads, w.kv_heads,
                                self.start, self.max_len, self.bt_d, self.pps, self.num_pages, self.kc, self.vc,
                                self.chunk, 1.0 / math.sqrt(128), self.out, self.ws, self.ws_n, stream)
        else:
            tq.tq_decode_attention(self.ctx, self.q, self.dt, w.batch, w.q_heads, w.kv_heads, self.start,
                                   self.max_len, self.bt_d, self.pps, self.num_pages, self.kc, self.vc, self.chunk,
                                   1.0 / math.sqrt(128), self.out, self.ws, self.ws_n, stream)
        self.out_h.copy_(self.out, non_blocking=True)

    def e2e_bytes(self):
        h2d = self.in_h.numel() * self.in_h.element_size()
        return h2d, self.out.numel() * 4

    def close(self):
        self.tq.tq_destroy(self.ctx)


class QuantizeBench:
    def __init__(self, w, torch, tq):
        self.w, self.torch, self.tq = w, torch, tq
        dev = torch.device("cuda", torch.cuda.current_device())
        cfg = tq.make_config(k_bits=w.k_bits, v_bits=w.v_bits, m=w.m, seed=w.seed, k_qjl=w.qjl)
        self.ctx = tq.tq_create_ex(cfg)
        B, H, T = w.batch, w.kv_heads, w.seq_len
        self.bt = wl.block_table(w)
        self.pps = self.bt.shape[1]
        self.num_pages = B * self.pps
        kpb, vpb = tq.tq_cache_layout(self.ctx, H)
        self.kc = torch.empty(self.num_pages * kpb, dtype=torch.uint8, device=dev)
        self.vc = torch.empty(self.num_pages * vpb, dtype=torch.uint8, device=dev)
        self.K = torch.empty(B, T, H, 128, dtype=torch.bfloat16, device=dev)
        self.V = torch.empty(B, T, H, 128, dtype=torch.bfloat16, device=dev)
        for b in range(B):
            self.K[b] = torch.from_numpy(wl.kv_tokens(w, "k", b)).to(dev).to(torch.bfloat16)
            self.V[b] = torch.from_numpy(wl.kv_tokens(w, "v", b)).to(dev).to(torch.bfloat16)
        self.bt_d = torch.from_numpy(self.bt).to(dev)
        self.start = torch.zeros(B, dtype=torch.int32, device=dev)
        self.vectors = 2 * B * T * H
        self.bytes_in = self.vectors * 128 * 2
        self.bytes_out = B * T * H * (kpb + vpb) // (16 * H)

    def step(self, stream):
        w, tq = self.w, self.tq
        tq.tq_quantize(self.ctx, self.K, self.V, tq.TQ_BF16, w.batch, w.seq_len, w.kv_heads, self.start, self.bt_d,
                       self.pps, self.num_pages, self.kc, self.vc, stream)

    def close(self):
        self.tq.tq_destroy(self.ctx)


def max_over_ranks(ms, dist, device):
    """The slowest rank's time (all ranks return it); `ms` unchanged on a single process."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([float(ms)], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def timed(torch, stream, fn, steps, warmup, dist=None, flush=None):
    """Device time of `steps` calls of fn(i) after `warmup` untimed ones, barrier + sync on both sides, max over
    ranks.  With `flush` (a callable that evicts L2), it runs before every call and each call is timed alone."""
    for _ in range(warmup):
        if flush is not None:
            flush()
        fn()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    if flush is None:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(steps):
            fn(i)
        end.record(stream)
        torch.cuda.synchronize()
        ms = start.elapsed_time(end)
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(steps):
            flush()
            evs[i][0].record(stream)
            fn(i)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        ms = sum(e0.elapsed_time(e1) for e0, e1 in evs)
    ms = max_over_ranks(ms, dist, "cuda")
    if dist is not None:
        dist.barrier()
    return ms


def l2_flusher(torch, bytes_step):
    """(callable or None, description): inputs below twice the L2 size get a flush between timed steps."""
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    if bytes_step >= 2 * l2:
        return None, f"packed cache {bytes_step / 2**20:.0f} MiB > 2x L2 ({l2 / 2**20:.0f} MiB): no flush"
    buf = torch.empty(4 * l2 // 4, dtype=torch.int32, device="cuda")
    return (lambda: buf.zero_()), (f"packed cache {bytes_step / 2**20:.0f} MiB < 2x L2 ({l2 / 2**20:.0f} MiB): "
                                   f"a {4 * l2 / 2**20:.0f} MiB buffer is written before every timed step, "
                                   f"each step timed alone")


def decode_measure(torch, tq, w, stream, steps, warmup, dist, peak, peak_kind, world, profile=False):
    """One decode workload: `steps` timed steps after `warmup` (CUDA events on the launch stream), the same steps
    again with the partials kernel bracketed by events, then the same steps end to end from pinned host memory."""
    db = DecodeBench(w, torch, tq)
    ev = [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(steps)]
    for pair in ev:                      # create the CUDA events (the library records them inside the step)
        for e in pair:
            e.record(stream)
    for _ in range(warmup):
        db.step(stream)
    torch.cuda.synchronize()
    flush, l2_note = l2_flusher(torch, db.bytes_step)
    sampler = ClockSampler(torch)
    with sampler:                        # clocks over the timed steps and the end-to-end steps
        # the step as a user runs it (no events inside: an event between two launches would stop the next
        # kernel from starting while the previous one finishes), then the same steps with the partials kernel
        # bracketed by events, for its own duration
        ms = timed(torch, stream, lambda i=None: db.step(stream), steps, 0, dist, flush)
        ms_ev = timed(torch, stream, lambda i=None: db.step(stream, ev[i] if i is not None else None), steps, 0,
                      dist, flush)
        ms_e2e = timed(torch, stream, lambda i=None: db.step_e2e(stream), steps, warmup, dist, flush)
    kern_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    ms_step = ms / steps
    value = db.bytes_step * world / (ms_step * 1e-3) / 1e9
    achieved = db.bytes_step / (kern_ms * 1e-3) / 1e9
    h2d, d2h = db.e2e_bytes()
    e2e_value = db.bytes_step * world / (ms_e2e / steps * 1e-3) / 1e9
    flags = tq.tq_check_device_status(db.ctx)
    ctx_desc = f"context {int(db.lens.max())}" if w.len_range is None else \
        f"context uniform in [{w.len_range[0]}, {w.len_range[1]}] (sum {int(db.lens.sum())})"
    step_desc = "append 1 token + attention" if w.append else "attention over the cached tokens (no append)"
    rec = {
        "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(ms_step, 5), "steps": steps,
        "warmup": warmup, "hbm_fraction": round(value / world / peak, 4),
        "config": {"workload": f"{w.name}: decode step = {step_desc}, batch {w.batch}, {w.q_heads}/{w.kv_heads} "
                               f"heads, head_dim 128, {ctx_desc}{'+1' if w.append else ''}, "
                               f"K {w.k_bits} bits{' + QJL m=%d' % w.m if w.qjl else ''}, V {w.v_bits} bits, "
                               f"{'fp32' if w.dtype == 'f32' else 'bf16'} inputs",
                   "split_k_chunk_tokens": db.chunk, "packed_bytes_per_step": db.bytes_step, "l2": l2_note},
        "roofline": {"kernel": "lut_partials_kernel (split-K partials: scoring, online softmax, value sums)",
                     "bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": db.bytes_step, "avg_launch_ms": round(kern_ms, 5),
                     "timed_in": "a second pass of the same timed steps with events around the partials launch "
                                 f"({ms_ev / steps:.5f} ms per step in that pass)",
                     "traffic": None if profile else traffic_for("tq_decode_lut.cu", "lut_partials_kernel", w.name)},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": steps * db.launches_per_step,
        "clocks": sampler.result(),
        "device_flags": flags,
    }
    db.close()
    del db
    torch.cuda.empty_cache()
    return rec


CAUSAL_B, CAUSAL_L, CAUSAL_T = 4, 8192, 64


def causal_measure(torch, tq, stream, steps, warmup, dist, peak, peak_kind, world):
    """Multi-query causal attention (a prefill chunk): c3's shapes (32/8 heads, 3.5-bit K + QJL, 3.5-bit V) with
    4 sequences of 8192 cached tokens and 64 new tokens each; a step quantize-appends the new tokens' K/V and runs
    tq_causal_attention (token t attends over its prefix).  value = packed bytes of the attended cache / step time."""
    w = wl.WORKLOADS["c3"].scaled(batch=CAUSAL_B, seq_len=CAUSAL_L)
    dev = torch.device("cuda", torch.cuda.current_device())
    ctx = tq.tq_create_ex(tq.make_config(k_bits=w.k_bits, v_bits=w.v_bits, m=w.m, seed=w.seed, k_qjl=w.qjl))
    B, H, Hq, T, L = CAUSAL_B, w.kv_heads, w.q_heads, CAUSAL_T, CAUSAL_L
    pps = (L + T + 15) // 16
    bt = torch.randperm(B * pps, generator=torch.Generator().manual_seed(w.seed)).to(torch.int32).view(B, pps).to(dev)
    kpb, vpb = tq.tq_cache_layout(ctx, H)
    kc = torch.empty(B * pps * kpb, dtype=torch.uint8, device=dev)
    vc = torch.empty(B * pps * vpb, dtype=torch.uint8, device=dev)
    zero = torch.zeros(1, dtype=torch.int32, device=dev)
    for b in range(B):
        for s0 in range(0, L, 8192):
            n = min(8192, L - s0)
            K = torch.from_numpy(wl.kv_tokens(w, "k", b, s0, n)).to(dev).to(torch.bfloat16)
            V = torch.from_numpy(wl.kv_tokens(w, "v", b, s0, n)).to(dev).to(torch.bfloat16)
            zero.fill_(s0)
            tq.tq_quantize(ctx, K, V, tq.TQ_BF16, 1, n, H, zero, bt[b], pps, B * pps, kc, vc)
    g = torch.Generator(device=dev).manual_seed(w.seed + 1)
    knew = torch.randn(B, T, H, 128, device=dev, generator=g).to(torch.bfloat16)
    vnew = torch.randn(B, T, H, 128, device=dev, generator=g).to(torch.bfloat16)
    q = torch.randn(B, T, Hq, 128, device=dev, generator=g).to(torch.bfloat16)
    start = torch.full((B,), L, dtype=torch.int32, device=dev)
    ws_n = tq.tq_causal_workspace_size(ctx, B, T, Hq, L + T, 0)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=dev)
    out = torch.empty(B, T, Hq, 128, dtype=torch.float32, device=dev)

    def step(i=None):
        tq.tq_quantize(ctx, knew, vnew, tq.TQ_BF16, B, T, H, start, bt, pps, B * pps, kc, vc, stream)
        tq.tq_causal_attention(ctx, q, tq.TQ_BF16, B, T, Hq, H, start, L + T, bt, pps, B * pps, kc, vc, 0,
                               1.0 / math.sqrt(128), out, ws, ws_n, stream)

    def attend(i=None):
        tq.tq_causal_attention(ctx, q, tq.TQ_BF16, B, T, Hq, H, start, L + T, bt, pps, B * pps, kc, vc, 0,
                               1.0 / math.sqrt(128), out, ws, ws_n, stream)

    step()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch)
    with sampler:
        ms = timed(torch, stream, step, steps, warmup, dist) / steps
        ms_att = timed(torch, stream, attend, steps, warmup, dist) / steps
    bytes_step = B * H * (L + T) * wl.packed_bytes_per_token_head(w)     # every token up to the last new one
    # algorithmic flops: every attended (query row, token) pair costs <q~, k^> + <u, signs> + p v, 2 (d + m + d)
    pairs = B * Hq * sum(L + t + 1 for t in range(T))
    flops = pairs * 2 * (128 + w.m + 128)
    tpk, tpk_kind = tensor_peak()
    tflops = flops * world / (ms_att * 1e-3) / 1e12
    flags = tq.tq_check_device_status(ctx)
    tq.tq_destroy(ctx)
    value = bytes_step * world / (ms * 1e-3) / 1e9
    return {"workload": f"causal: {B} seq x ({L} cached + {T} new tokens), {Hq}/{H} heads, K {w.k_bits} bits + QJL "
                        f"m={w.m}, V {w.v_bits} bits; step = quantize-append the {T} new tokens + causal attention "
                        f"(token t over its prefix)",
            "value": round(value, 2), "unit": "GB/s of attended packed cache", "ms_per_step": round(ms, 5),
            "queries_per_s": round(B * T * Hq * world / (ms * 1e-3), 1), "steps": steps,
            "l2": f"packed cache {bytes_step / 2**20:.0f} MiB > 2x L2: no flush",
            "roofline": {"kernel": "whole step (quantize-append + qprep + causal partials + merge)", "bound": "hbm",
                         "achieved": round(value, 2), "peak": peak, "unit": "GB/s", "frac": round(value / peak, 4),
                         "peak_source": peak_kind, "algorithmic_bytes_per_launch": bytes_step, "traffic": None},
            "attention_only": {"ms": round(ms_att, 5), "launches": "qprep_rows + causal_tc + merge_blk",
                               "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": tpk,
                                            "unit": "TFLOP/s", "frac": round(tflops / tpk, 4), "peak_source": tpk_kind,
                                            "algorithmic_flops_per_call": flops,
                                            "note": "768 flops per attended (query row, token) pair"}},
            "gpu_launches": 7 * steps, "clocks": sampler.result(), "device_flags": flags}


def quantize_measure(torch, tq, qw, stream, qsteps, warmup, dist, peak, peak_kind, world):
    """The quantize-append workload (c2 shape): one launch per step quantizes every K and V vector."""
    qb = QuantizeBench(qw, torch, tq)
    qs = ClockSampler(torch)
    with qs:
        qms = timed(torch, stream, lambda i=None: qb.step(stream), qsteps, warmup, dist)
    qstep = qms / qsteps
    qbytes = qb.bytes_in + qb.bytes_out
    full = qw == wl.WORKLOADS["c2"]
    rec = {
        "workload": f"{qw.name}: quantize-append {qw.batch} seq x {qw.kv_heads} KV heads x {qw.seq_len} tokens bf16, "
                    f"K {qw.k_bits} bits + QJL m={qw.m} / V {qw.v_bits} bits, random block-table permutation",
        "value": round(qb.vectors * world / (qstep * 1e-3), 1), "unit": "KV vectors/s", "ms_per_step": round(qstep, 4),
        "steps": qsteps,
        "l2": f"{qb.bytes_in / 2**20:.0f} MiB of bf16 input per step > 2x L2: no flush",
        "roofline": {"kernel": "quantize_pipe_kernel (K and V tiles in one launch)", "bound": "hbm",
                     "achieved": round(qbytes / (qstep * 1e-3) / 1e9, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(qbytes / (qstep * 1e-3) / 1e9 / peak, 4), "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": qbytes,
                     "traffic": traffic_for("tq_quantize_pipe.cu", "quantize_pipe_kernel", "c2") if full else None},
        "refined": tq.tq_refine_counters(qb.ctx),
        "clocks": qs.result(),
    }
    qb.close()
    return rec


SEARCH_N, SEARCH_NQ, SEARCH_K = 1 << 20, 64, 10


def search_measure(torch, tq, stream, steps, warmup, peak, peak_kind):
    """Inner-product search: 2^20 database vectors (one KV head's K cache, 3-bit + QJL, N(0,1) bf16 with
    channels 0-3 x10, quantized by tq_quantize), 64 bf16 queries, the 10 best each; value = database bytes
    read per search / time."""
    dev = torch.device("cuda")
    ctx = tq.tq_create_ex(tq.make_config(k_bits=(3, 3), v_bits=(3, 3), seed=4))
    kpb, _ = tq.tq_cache_layout(ctx, 1)
    npg = SEARCH_N // 16
    gen = torch.Generator(device=dev)
    gen.manual_seed(4)
    kc = torch.zeros(npg * kpb, dtype=torch.uint8, device=dev)
    bt = torch.randperm(npg, device=dev, generator=gen).to(torch.int32)
    X = torch.randn(1, SEARCH_N, 1, 128, device=dev, generator=gen)
    X[..., :4] *= 10
    X = X.to(torch.bfloat16)
    tq.tq_quantize(ctx, X, None, tq.TQ_BF16, 1, SEARCH_N, 1, torch.zeros(1, dtype=torch.int32, device=dev),
                   bt.view(1, -1), npg, npg, kc, None, stream)
    del X
    q_h = torch.randn(SEARCH_NQ, 128, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).pin_memory()
    q = q_h.to(dev)
    ws_n = tq.tq_search_workspace_size(ctx, SEARCH_NQ, SEARCH_N, SEARCH_K)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=dev)
    ts = torch.empty(SEARCH_NQ, SEARCH_K, device=dev)
    ti = torch.empty(SEARCH_NQ, SEARCH_K, dtype=torch.int32, device=dev)
    ts_h, ti_h = torch.empty_like(ts, device="cpu").pin_memory(), torch.empty_like(ti, device="cpu").pin_memory()
    run = lambda: tq.tq_search(ctx, q, tq.TQ_BF16, SEARCH_NQ, kc, bt, npg, SEARCH_N, SEARCH_K, ts, ti, ws, ws_n,
                               stream)

    def run_e2e():
        q.copy_(q_h, non_blocking=True)
        run()
        ts_h.copy_(ts, non_blocking=True)
        ti_h.copy_(ti, non_blocking=True)

    flush, l2_note = l2_flusher(torch, npg * kpb)
    sampler = ClockSampler(torch)
    with sampler:
        ms = timed(torch, stream, lambda i=None: run(), steps, warmup, None, flush) / steps
    ms_e2e = timed(torch, stream, lambda i=None: run_e2e(), steps, warmup, None, flush) / steps
    db_bytes = npg * kpb
    value = db_bytes / (ms * 1e-3) / 1e9
    flags = tq.tq_check_device_status(ctx)
    tq.tq_destroy(ctx)
    return {
        "metric": "inner-product search: quantized database GB/s per query batch",
        "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(ms, 4), "steps": steps, "warmup": warmup,
        "higher_is_better": True,
        "dtype": "packed 3-bit codes + QJL signs; fp16 tensor-core products (tcgen05), fp32 accumulation",
        "data": "synthetic (seeded N(0,1), channels 0-3 x10)",
        "config": {"workload": f"search: {SEARCH_N} database vectors (one KV head, K 3-bit + QJL m=128), "
                               f"{SEARCH_NQ} bf16 queries, top {SEARCH_K}",
                   "database_bytes": db_bytes, "scores_per_s": round(SEARCH_NQ * SEARCH_N / (ms * 1e-3), 1),
                   "l2": l2_note},
        "roofline": {"kernel": "tq_search: qprep, search_tc_kernel (scores + per-thread top 16), merge; "
                               "timed as the whole call", "bound": "hbm",
                     "achieved": round(value, 2), "peak": peak, "unit": "GB/s", "frac": round(value / peak, 5),
                     "peak_source": peak_kind, "algorithmic_bytes_per_launch": db_bytes, "traffic": None},
        "e2e": {"value": round(db_bytes / (ms_e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": q_h.numel() * 2, "d2h_bytes_per_step": ts.numel() * 4 + ti.numel() * 4},
        "gpu_launches": 3 * steps, "clocks": sampler.result(), "device_flags": flags,
    }


def oracle_search_sample(seconds=10.0):
    """The oracle's search (fp64) on a database sample: database bytes per second on one core."""
    import oracle
    p = oracle.make_params(k_bits=(3, 3), v_bits=(3, 3), seed=4)
    rng = np.random.default_rng(4)
    n = 4096
    X = rng.standard_normal((n, 128))
    X[:, :4] *= 10
    Q = rng.standard_normal((SEARCH_NQ, 128))
    row = np.arange(n // 16)
    cache = np.zeros((n // 16) * oracle.cache_block_bytes(p, "k"), dtype=np.uint8)
    rec = oracle.pack_k_records(p, oracle.quantize_vectors(p, X, "k"))
    oracle.write_paged(p, "k", cache, rec, row[np.arange(n) // 16], np.arange(n) % 16, np.zeros(n, dtype=np.int64), 1)
    reps, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds or reps == 0:
        oracle.search(p, Q, row, cache, n, SEARCH_K)
        reps += 1
    el = time.perf_counter() - t0
    return {"value": round(cache.size * reps / el / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{reps} fp64 searches of {SEARCH_NQ} queries over {n} database vectors (3-bit + QJL)"}


def run_ours(args):
    import torch
    from online_kv_cache_02_gb300 import tq

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    # the oracle's worker processes start before the first GPU call (spawn)
    pool = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.only:
        pool = OraclePool(wl.WORKLOADS[args.config], cpu_workers(args.cpu_workers))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
        dist = tdist
    stream = torch.cuda.current_stream()
    peak, peak_kind = peaks()
    warmup = max(3, args.warmup)

    if args.only == "search":
        line = search_measure(torch, tq, stream, args.steps, warmup, peak, peak_kind)
        line.update({"n_gpus": world, "scaling": "weak", "vs_baseline": None})
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = oracle_search_sample()
        if rank == 0:
            print(json.dumps(line), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return
    if args.only == "causal":
        line = {"metric": "causal attention over the compressed cache: GB/s of attended packed cache"}
        line.update(causal_measure(torch, tq, stream, args.steps, warmup, dist, peak, peak_kind, world))
        if rank == 0:
            print(json.dumps(line), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return
    if args.only == "quantize":
        qw = wl.WORKLOADS["c2"].scaled(batch=args.batch) if args.batch else wl.WORKLOADS["c2"]
        line = {"metric": "KV vectors quantized/s (quantize only)"}
        line.update(quantize_measure(torch, tq, qw, stream, args.steps, warmup, dist, peak, peak_kind, world))
        if rank == 0:
            print(json.dumps(line), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return
    w = wl.WORKLOADS[args.config]
    if args.batch:
        w = w.scaled(batch=args.batch)
    head = decode_measure(torch, tq, w, stream, args.steps, warmup, dist, peak, peak_kind, world,
                          profile=bool(args.batch))
    line = {
        "metric": "quantized-KV decode attention GB/s (% of HBM peak); KV vectors quantized/s",
        "value": head["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": warmup,
        "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "packed 2-4 bit codes + QJL signs, fp32 accumulation",
        "data": "synthetic (seeded N(0,1), outlier channels)",
        "config": dict(head["config"], hbm_fraction=head["hbm_fraction"],
                       parallelism=f"replicas x{world}, no collective"),
        "roofline": head["roofline"], "e2e": head["e2e"], "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"], "device_flags": head["device_flags"],
    }
    if not args.no_others and not args.batch:
        for name in ("c4", "c5", "c1"):
            if name == args.config:
                continue
            rec = decode_measure(torch, tq, wl.WORKLOADS[name], stream, args.steps, warmup, dist, peak, peak_kind,
                                 world)
            line[name] = rec
            line["gpu_launches"] += rec["gpu_launches"]
    if not args.no_others and not args.batch:
        line["causal"] = causal_measure(torch, tq, stream, args.steps, warmup, dist, peak, peak_kind, world)
        line["gpu_launches"] += line["causal"]["gpu_launches"]
    if not args.no_quantize:
        line["quantize"] = quantize_measure(torch, tq, wl.WORKLOADS["c2"], stream, max(3, min(args.steps, 20)),
                                            warmup, dist, peak, peak_kind, world)
        line["gpu_launches"] += line["quantize"]["steps"]
    if pool is not None:
        line["cpu_baseline"] = cpu_baseline(pool, w)
        line["quantize"]["cpu_baseline"] = pool.quantize_rates() if "quantize" in line else None
        pool.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

def cpu_workers(requested=0):
    """Host cores this process may run on (or `requested`, if smaller and positive)."""
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return min(n, requested) if requested > 0 else n


def cpu_model():
    """lscpu's model name (with the vendor where lscpu gives one), else /proc/cpuinfo's, else the machine."""
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        f = {k.strip(): v.strip() for k, _, v in (ln.partition(":") for ln in out.splitlines())}
        name = f.get("Model name", "")
        if name:
            vendor = f.get("Vendor ID", "")
            return f"{vendor} {name}".strip() if vendor and vendor not in name else name
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for ln in fh:
                k, _, v = ln.partition(":")
                if k.strip().lower() in ("model name", "cpu model"):
                    return v.strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


class OracleDecode:
    """One (sequence, KV head) of the workload, quantized and decoded by the fp64 oracle."""

    def __init__(self, w, b=0, h=0):
        import oracle
        from oracle import turboquant as otq
        self.o, self.otq = oracle, otq
        self.w, self.b, self.h = w, b, h
        self.p = oracle.make_params(d=128, m=w.m, k_bits=w.k_bits, v_bits=w.v_bits, seed=w.seed, k_qjl=w.qjl)
        L = int(wl.seq_lens(w)[b])
        self.L = L
        K = wl.kv_tokens(w, "k", b)[:, h].astype(np.float64)
        V = wl.kv_tokens(w, "v", b)[:, h].astype(np.float64)
        self.kraw = oracle.pack_k_records(self.p, oracle.quantize_vectors(self.p, K, "k"))
        self.vraw = oracle.pack_v_records(self.p, oracle.quantize_vectors(self.p, V, "v"))
        self.append = w.append
        if w.append:
            self.knew = wl.new_tokens(w, "k")[b, :, h].astype(np.float64)
            self.vnew = wl.new_tokens(w, "v")[b, :, h].astype(np.float64)
        G = w.q_heads // w.kv_heads
        self.Q = wl.queries(w)[b, h * G:(h + 1) * G].astype(np.float64)
        self.bytes = (L + (1 if w.append else 0)) * wl.packed_bytes_per_token_head(w)

    def step(self):
        o, p = self.o, self.p
        kraw, vraw = self.kraw, self.vraw
        if self.append:
            kn = o.pack_k_records(p, o.quantize_vectors(p, self.knew, "k"))
            vn = o.pack_v_records(p, o.quantize_vectors(p, self.vnew, "v"))
            kraw = {k: np.concatenate([kraw[k], kn[k]]) for k in kn}
            vraw = {k: np.concatenate([vraw[k], vn[k]]) for k in vn}
        kr = o.unpack_k_records(p, kraw)
        vr = o.unpack_v_records(p, vraw)
        return [self.otq.attend_one(p, q, kr, vr, 1.0 / math.sqrt(128)) for q in self.Q]


def _oracle_quantize_slice(w, b):
    """The oracle's quantize of sequence b of a quantize workload (every KV head, K and V): (vectors, seconds)."""
    import oracle
    p = oracle.make_params(d=128, m=w.m, k_bits=w.k_bits, v_bits=w.v_bits, seed=w.seed, k_qjl=w.qjl)
    K = wl.kv_tokens(w, "k", b).reshape(-1, 128).astype(np.float64)
    V = wl.kv_tokens(w, "v", b).reshape(-1, 128).astype(np.float64)
    bt = wl.block_table(w)
    H, T = w.kv_heads, w.seq_len
    kc = np.zeros(bt.size * oracle.cache_block_bytes(p, "k") * H, np.uint8)
    vc = np.zeros(bt.size * oracle.cache_block_bytes(p, "v") * H, np.uint8)
    ti, hi = np.meshgrid(np.arange(T), np.arange(H), indexing="ij")
    pages, slots = bt[b, ti.ravel() // 16], ti.ravel() % 16
    t0 = time.perf_counter()
    oracle.write_paged(p, "k", kc, oracle.pack_k_records(p, oracle.quantize_vectors(p, K, "k")), pages, slots,
                       hi.ravel(), H)
    oracle.write_paged(p, "v", vc, oracle.pack_v_records(p, oracle.quantize_vectors(p, V, "v")), pages, slots,
                       hi.ravel(), H)
    return len(K) + len(V), time.perf_counter() - t0


def _oracle_worker(conn, w, b, h):
    """Worker process: holds one (sequence, KV head) of the decode workload; runs oracle steps on request.
    It builds its oracle cache only when asked (so it stays idle while the GPU is being timed)."""
    if conn.recv()[0] != "init":
        return
    od = OracleDecode(w, b, h)
    conn.send(("ready", od.bytes, od.L))
    while True:
        cmd = conn.recv()
        if cmd[0] == "step":
            t0 = time.perf_counter()
            for _ in range(cmd[1]):
                od.step()
            conn.send(("done", time.perf_counter() - t0))
        elif cmd[0] == "quantize":
            conn.send(("done",) + _oracle_quantize_slice(wl.WORKLOADS["c2"], cmd[1]))
        else:
            break


class OraclePool:
    """One spawn-started process per host core, each holding its own (sequence, KV head) of the decode workload
    (the first `n` of its units).  Started before the first GPU call; each worker runs numpy with one BLAS
    thread."""

    def __init__(self, w, n):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        units = [(b, h) for b in range(w.batch) for h in range(w.kv_heads)]
        self.n = max(1, min(n, len(units)))
        self.w = w
        self.conns, self.procs = [], []
        for b, h in units[:self.n]:
            a, bconn = ctx.Pipe()
            pr = ctx.Process(target=_oracle_worker, args=(bconn, w, b, h), daemon=True)
            pr.start()
            self.conns.append(a)
            self.procs.append(pr)
        self._ready = None

    def ready(self):
        if self._ready is None:
            for c in self.conns:
                c.send(("init",))
            self._ready = [c.recv() for c in self.conns]
        return self._ready

    def step(self, workers, reps=1):
        """`reps` oracle steps on each of the first `workers` workers at once: (bytes, wall seconds)."""
        info = self.ready()
        t0 = time.perf_counter()
        for c in self.conns[:workers]:
            c.send(("step", reps))
        for c in self.conns[:workers]:
            c.recv()
        return sum(i[1] for i in info[:workers]) * reps, time.perf_counter() - t0

    def quantize_rates(self):
        """The oracle's quantize of c2 slices (one sequence = 1/32 of the workload each): one core, then every
        worker on its own sequence at once; vectors/s, extrapolated from the slices to the whole workload."""
        self.ready()
        qw = wl.WORKLOADS["c2"]
        self.conns[0].send(("quantize", 0))
        _, nv1, s1 = self.conns[0].recv()
        k = min(self.n, qw.batch)
        t0 = time.perf_counter()
        for i, c in enumerate(self.conns[:k]):
            c.send(("quantize", i))
        nv = sum(c.recv()[1] for c in self.conns[:k])
        wall = time.perf_counter() - t0
        total = 2 * qw.batch * qw.seq_len * qw.kv_heads
        return {"value": round(nv / wall, 1), "unit": "KV vectors/s", "cores": k, "kind": "oracle",
                "sample": f"{k} of the 32 sequences of c2 (each 1/32 of the workload: {nv1} K+V vectors) quantized, "
                          f"packed and written through the block table at once; extrapolated to the "
                          f"{total}-vector workload: {total / (nv / wall):.1f} s",
                "single_core": {"value": round(nv1 / s1, 1), "unit": "KV vectors/s", "cores": 1,
                                "sample": f"sequence 0 of c2 (1/32 of the workload, {nv1} vectors) in {s1:.2f} s; "
                                          f"extrapolated to the workload: {total / (nv1 / s1):.1f} s"},
                "cpu_model": cpu_model()}

    def close(self):
        for c in self.conns:
            try:
                c.send(("quit",))
            except (BrokenPipeError, OSError):
                pass
        for pr in self.procs:
            pr.join(timeout=30)
            if pr.is_alive():
                pr.kill()


def cpu_baseline(pool, w, seconds=8.0):
    """The oracle on the host cores: every pool worker stepping its own (sequence, KV head) at once, and one
    worker alone; decode GB/s of packed cache read (the GPU metric's bytes)."""
    info = pool.ready()
    b1, s1 = pool.step(1)
    reps1 = max(1, int(seconds / max(s1, 1e-3)) - 1)
    b1r, s1r = pool.step(1, reps1)
    b1, s1 = b1 + b1r, s1 + s1r
    bn, sn = pool.step(pool.n)
    repsn = max(1, int(seconds / max(sn, 1e-3)) - 1)
    bnr, snr = pool.step(pool.n, repsn)
    bn, sn = bn + bnr, sn + snr
    L = info[0][2]
    G = w.q_heads // w.kv_heads
    return {"value": round(bn / sn / 1e9, 6), "unit": "GB/s", "cores": pool.n, "kind": "oracle",
            "sample": f"{pool.n} worker processes, each its own (sequence, KV head) of {w.name} ({G} query heads, "
                      f"{L}{'+1' if w.append else ''} tokens: append + fp64 decode per step), all stepping at once; "
                      f"{1 + repsn} steps each; numpy with 1 BLAS thread per worker",
            "single_core": {"value": round(b1 / s1 / 1e9, 6), "unit": "GB/s", "cores": 1,
                            "sample": f"one worker alone, {1 + reps1} steps"},
            "cpu_model": cpu_model(), "host_cores": cpu_workers()}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = wl.WORKLOADS[args.config]
    pool = OraclePool(w, cpu_workers(args.cpu_workers))
    try:
        pool.ready()
        for _ in range(args.warmup):
            pool.step(pool.n)
        tot_b, tot_s = 0, 0.0
        for _ in range(args.steps):
            b, s = pool.step(pool.n)
            tot_b += b
            tot_s += s
    finally:
        pool.close()
    value = tot_b / tot_s / 1e9
    G = w.q_heads // w.kv_heads
    sample = (f"each step: {pool.n} worker processes, each its own (sequence, KV head) of {w.name} ({G} query heads),"
              f" append 1 token + fp64 decode over {pool.ready()[0][2] + 1} tokens, all at once; 1 BLAS thread each")
    line = {
        "impl": "reference",
        "metric": "quantized-KV decode attention GB/s (% of HBM peak); KV vectors quantized/s",
        "value": round(value, 6), "unit": "GB/s", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_s / max(args.steps, 1) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name}: oracle sample of the decode step ({pool.n} of its "
                               f"{w.batch * w.kv_heads} (sequence, KV head) units per step)"},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": pool.n, "kind": "oracle",
                         "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
