"""Throughput of the mixed-head attention hot path on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl duo|reference]
                    [--workload NAME] [--no-decode] [--no-e2e] [--no-cpu-baseline]

Default workload: one-shot prefill of 32768 tokens shaped like one Llama-3-8B
layer (batch 1, 32 query / 8 KV heads, head_dim 128, 4 retrieval KV heads chosen
by a seeded permutation, sink 64 / recent 256). One step = the whole hot path for
that input: one prefill launch over all heads, then the append of the 32768
tokens' K/V into the retrieval and sink + ring caches. ``value`` = algorithmic
prefill FLOPs (4 D per visible pair per query head) / step time, inputs already
in HBM. The per-step inputs (Q 256 MiB, K/V 64 MiB each) exceed the 129 MB L2, so
no separate L2 flush is done.

The line also carries the decode half of the metric on the million-token decode
workload (batch 1, 1,048,576 context tokens, 2 retrieval KV heads; each step
appends one token and decodes it): KV bytes the method must read / decode
kernel time, and the retrieval-only prefill throughput (a launch over the
retrieval heads alone).

Under torchrun (N > 1) every rank runs the same workload on its own GPU (the
path shards over sequences and heads with no exchange); rank 0 prints
value = all ranks' FLOPs / the slowest rank's time.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefill attn TFLOP/s & decode KV-read GB/s, as % of GB300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from the ncu
# captures summarised in profiles/, valid only for the kernel sources they were taken on
# (the decode records were re-keyed after a comment-only edit to the 4-bit consumer).
L2_BYTES = 129e6  # GB300 L2 capacity

MEASURED_TRAFFIC = {
    "prefill": {"src": ("prefill.cu", "duo_device.cuh", "duo_internal.h"), "sha1": "7a550e89e096f3fb",
                "bytes": 471.982e6 + 233.347e6},
    # the 8 prefill launches of one chunked-prefill step (Llama-2-7B shape, 8 x 4096 tokens)
    "prefill_chunked": {"src": ("prefill.cu", "duo_device.cuh", "duo_internal.h"), "sha1": "7a550e89e096f3fb",
                        "bytes": 1305.004e6 + 96.197e6},
    # the same against 4-bit caches (codes + pairs read and dequantized in the kernel)
    "prefill_chunked_kv4": {"src": ("prefill.cu", "duo_device.cuh", "duo_internal.h"), "sha1": "7a550e89e096f3fb",
                            "bytes": 940.968e6 + 84.545e6},
    # one decode launch of the batched 8 x 128K workload (device lengths, graph replay)
    "decode_batched": {"src": ("decode.cu", "duo_device.cuh", "duo_internal.h"), "sha1": "2a2b52e1174c6bc6",
                       "bytes": 1.081919e9 + 1.479e6},
    "decode": {"src": ("decode.cu", "duo_device.cuh", "duo_internal.h"), "sha1": "2a2b52e1174c6bc6",
               "bytes": 1.074810e9 + 1.485e6},
    # one decode launch of the million-token decode over 4-bit caches (stored bytes read)
    "decode_kv4": {"src": ("decode.cu", "duo_device.cuh", "duo_internal.h"), "sha1": "2a2b52e1174c6bc6",
                   "bytes": 285.598976e6 + 3.443456e6},
}


def measured_traffic(kernel):
    """Traffic of the last ncu capture of `kernel`, or None if its sources changed since."""
    import hashlib
    rec = MEASURED_TRAFFIC.get(kernel)
    if rec is None:
        return None
    m = hashlib.sha1()
    for f in rec["src"]:
        with open(os.path.join(ROOT, "streaming_kv_cache_duo_gb300", "csrc", f), "rb") as fh:
            m.update(fh.read())
    return rec["bytes"] if m.hexdigest()[:16] == rec["sha1"] else None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """SM clock and throttle reasons sampled every 5 ms (NVML through ctypes) while a
    timed region runs, with one sample as it starts and one as it ends."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int):
        self.cuda_index = cuda_index
        self.samples = []
        self.max_mhz = None
        self.stop_flag = threading.Event()
        self.thread = None
        self.nvml = None
        self.handle = None
        self.how = None

    def _open_nvml(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        bus = _pci_bus_id(self.cuda_index)
        if bus is not None and nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0:
            self.how = "nvml by PCI bus id"
        else:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            ids = [x for x in vis.split(",") if x.strip().isdigit()]
            idx = int(ids[self.cuda_index]) if self.cuda_index < len(ids) else self.cuda_index
            if nv.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(h)) != 0:
                return False
            self.how = f"nvml index {idx}"
        self.nvml, self.handle = nv, h
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        return True

    def _loop(self):
        import ctypes
        nv, h = self.nvml, self.handle
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        get_r = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while True:
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and get_r(h, ctypes.byref(rs)) == 0:
                self.samples.append((float(clk.value), int(rs.value)))
            if self.stop_flag.is_set():  # one last sample after the region ends
                break
            time.sleep(0.005)

    def start(self):
        try:
            ok = self._open_nvml()
        except OSError:
            ok = False
        if not ok:
            self.how = None
            return
        self.thread = threading.Thread(target=self._loop, daemon=True)
        self.thread.start()

    def stop(self):
        if self.thread is None:
            return None
        self.stop_flag.set()
        self.thread.join(timeout=2)
        if not self.samples:
            return None
        sm = sorted(c for c, _ in self.samples)
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(sm), "source": self.how}


def _pci_bus_id(cuda_index):
    """NVML-style PCI bus id ("0000:XX:00.0") of a CUDA device, from torch's properties."""
    try:
        import torch
        p = torch.cuda.get_device_properties(cuda_index)
        return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
    except Exception:
        return None


# ----------------------------------------------------------------------------- helpers
def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
    if torch.cuda.is_available() and local < torch.cuda.device_count():
        torch.cuda.set_device(local)
    return rank, world, local


def dist_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def events_ms(pairs):
    return [a.elapsed_time(b) for a, b in pairs]


# ----------------------------------------------------------------------------- our arm
def bench_prefill(w, steps, warmup, world, peaks, want_e2e):
    import torch

    import duo_synth as ds
    from streaming_kv_cache_duo_gb300 import DuoLayer, duo_attn_prefill_select, duo_device_error, workload as wl

    dev = torch.device("cuda", torch.cuda.current_device())
    L = w.prefill_len
    kinds = w.is_retrieval
    layer = DuoLayer(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, L, kinds, device=dev)
    q = ds.stream_torch(w.seed, ds.STREAM_Q, w.B, 0, L, w.Hq, w.D, device=dev)
    k = ds.stream_torch(w.seed, ds.STREAM_K, w.B, 0, L, w.Hkv, w.D, device=dev)
    v = ds.stream_torch(w.seed, ds.STREAM_V, w.B, 0, L, w.Hkv, w.D, device=dev)
    o = torch.empty_like(q)
    fr, fs = wl.prefill_flops(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, kinds, L)
    flops = fr + fs
    stream = torch.cuda.current_stream()

    def step():
        layer.reset()
        duo_attn_prefill_select(layer.handle, layer.cache, q, k, v, L, o, 3, stream)
        layer.append(k, v)

    for _ in range(warmup):
        step()
    # inputs that fit in L2 are flushed out of it before every step (a 256 MiB write
    # outside the per-step events, which then give the step time)
    in_bytes = (q.numel() + k.numel() + v.numel()) * 2
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if in_bytes < L2_BYTES else None
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    clocks = ClockSampler(dev.index)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(steps):
        layer.reset()
        if flush is not None:
            flush.fill_(i & 255)
        ev[i][0].record(stream)
        duo_attn_prefill_select(layer.handle, layer.cache, q, k, v, L, o, 3, stream)
        ev[i][1].record(stream)
        layer.append(k, v)
        ev[i][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    total_ms = dist_max(t_start.elapsed_time(t_end), world)
    prefill_ms = [a.elapsed_time(b) for a, b, _ in ev]
    append_ms = [b.elapsed_time(c) for _, b, c in ev]
    avg_prefill = sum(prefill_ms) / steps
    ms_step = total_ms / steps
    if flush is not None:  # the flushes are not part of a step
        ms_step = dist_max(sum(prefill_ms) + sum(append_ms), world) / steps
    value = flops * world / (ms_step * 1e-3) / 1e12

    # retrieval heads alone (the tensor-core figure of merit), one-shot: empty cache
    layer.reset()
    sel = []
    for _ in range(max(3, warmup)):
        duo_attn_prefill_select(layer.handle, layer.cache, q, k, v, L, o, 2, stream)
    torch.cuda.synchronize()
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        duo_attn_prefill_select(layer.handle, layer.cache, q, k, v, L, o, 2, stream)
        b.record(stream)
        sel.append((a, b))
    torch.cuda.synchronize()
    sel_ms = sum(events_ms(sel)) / steps
    if duo_device_error():
        raise RuntimeError("a kernel gave up a bounded wait")

    peak = peaks["bf16_tflops"]
    achieved = flops / (avg_prefill * 1e-3) / 1e12
    res = {
        "value": value, "ms_per_step": ms_step, "flops": flops,
        "prefill_ms": avg_prefill, "append_ms": sum(append_ms) / steps,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": measured_traffic("prefill"),
                     "kernel": f"prefill_kernel<{w.D}>", "flops_per_launch": flops},
        "prefill_retrieval_only": {"tflops": round(fr / (sel_ms * 1e-3) / 1e12, 2), "ms": round(sel_ms, 4),
                                   "flops": fr, "frac_of_bf16_peak": round(fr / (sel_ms * 1e-3) / 1e12 / peak, 4)},
        "clocks": clk, "launches": 2 * steps,
        "l2": (f"L2 flushed before every step (inputs {in_bytes / 2**20:.1f} MiB fit in the 129 MB L2; "
               "256 MiB write outside the step's events)") if flush is not None else
              (f"no flush: per-step inputs (Q {q.numel() * 2 / 2**20:.0f} MiB, K/V {k.numel() * 2 / 2**20:.0f} MiB "
               "each) exceed the 129 MB L2"),
    }
    if want_e2e:
        res["e2e"] = e2e_prefill(w, layer, q, k, v, o, flops, steps, warmup, world)
    layer.close()
    return res


def e2e_prefill(w, layer, q, k, v, o, flops, steps, warmup, world):
    """The same step through the public API with host buffers: every step copies its
    Q/K/V in from pinned host memory, runs prefill + append, and copies O out, all
    inside the timed region. Copies run on their own streams, double-buffered, so the
    upload of step i+1 and the readback of step i-1 overlap step i's kernels."""
    import torch
    from streaming_kv_cache_duo_gb300 import duo_attn_prefill_select
    hq = q.cpu().pin_memory()
    hk = k.cpu().pin_memory()
    hv = v.cpu().pin_memory()
    ho = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    dq = [q, torch.empty_like(q)]
    dk = [k, torch.empty_like(k)]
    dv = [v, torch.empty_like(v)]
    do = [o, torch.empty_like(o)]
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    L = w.prefill_len

    def run(n):
        ev = lambda: torch.cuda.Event()
        uploaded, computed, read = [None] * n, [None] * n, [None] * n

        def upload(i):
            x = i % 2
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(computed[i - 2])  # buffer x is free once step i-2 used it
                dq[x].copy_(hq, non_blocking=True)
                dk[x].copy_(hk, non_blocking=True)
                dv[x].copy_(hv, non_blocking=True)
                uploaded[i] = ev()
                uploaded[i].record(up)

        upload(0)
        for i in range(n):
            x = i % 2
            if i + 1 < n:
                upload(i + 1)
            comp.wait_event(uploaded[i])
            if i >= 2:
                comp.wait_event(read[i - 2])  # O buffer x has been read back
            layer.reset(stream=comp)
            duo_attn_prefill_select(layer.handle, layer.cache, dq[x], dk[x], dv[x], L, do[x], 3, comp)
            layer.append(dk[x], dv[x], stream=comp)
            computed[i] = ev()
            computed[i].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(computed[i])
                ho[x].copy_(do[x], non_blocking=True)
                read[i] = ev()
                read[i].record(down)
        comp.wait_event(read[n - 1])
        comp.wait_event(uploaded[n - 1])

    run(warmup)
    torch.cuda.synchronize()
    barrier(world)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    run(steps)
    b.record(comp)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = dist_max(a.elapsed_time(b), world) / steps
    h2d = (hq.numel() + hk.numel() + hv.numel()) * 2
    return {"value": round(flops * world / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": ho[0].numel() * 2,
            "how": "pinned host Q/K/V in, O out, every step; copies on two side streams, double-buffered, "
                   "overlapping the neighbouring steps' kernels", "clocks": clk}


def make_layer(w, cap, dev, paged_block, pool=False, kv4=False):
    """A DuoLayer, or with paged_block > 0 a DuoPagedLayer whose retrieval blocks are
    scattered over the pool in a seeded random order; with `pool` the streaming heads
    live in the same pool too (every block of their table allocated: the ones that
    fall out of the window are simply never touched again)."""
    import numpy as np
    import torch

    from streaming_kv_cache_duo_gb300 import DuoKv4Layer, DuoKv4PagedLayer, DuoLayer, DuoPagedLayer
    kinds = w.is_retrieval
    if kv4 and paged_block <= 0:
        return DuoKv4Layer(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, cap, kinds, device=dev)
    if paged_block <= 0:
        return DuoLayer(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, cap, kinds, device=dev)
    n_ret = sum(kinds)
    n_str = len(kinds) - n_ret
    max_blocks = -(-cap // paged_block)
    planes = n_ret + (n_str if pool else 0)
    num_blocks = w.B * planes * max_blocks
    ids = np.random.default_rng(w.seed).permutation(num_blocks).reshape(w.B, planes, max_blocks)
    table = torch.tensor(ids[:, :n_ret], dtype=torch.int32, device=dev) if n_ret else None
    if kv4:  # 4-bit rows in the pool; streaming heads keep their 4-bit ring arrays
        return DuoKv4PagedLayer(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, paged_block, max_blocks, num_blocks, table, kinds,
                                device=dev)
    stream = torch.tensor(ids[:, n_ret:], dtype=torch.int32, device=dev) if pool else None
    return DuoPagedLayer(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, paged_block, max_blocks, num_blocks, table, kinds,
                         device=dev, stream_table=stream)


def bench_decode(w, steps_cap, peaks, paged_block=0, pool=False, kv4=False):
    """Million-token decode: build the cache by appends, then time (append 1 token + decode)."""
    import torch

    import duo_synth as ds
    from streaming_kv_cache_duo_gb300 import DuoLayer, duo_attn_decode, duo_device_error, workload as wl

    dev = torch.device("cuda", torch.cuda.current_device())
    kinds = w.is_retrieval
    steps = min(w.decode_steps, steps_cap)
    layer = make_layer(w, w.context + w.decode_steps, dev, paged_block, pool, kv4)
    chunk = 65536
    for c0 in range(0, w.context, chunk):
        kk = ds.stream_torch(w.seed, ds.STREAM_K, w.B, c0, chunk, w.Hkv, w.D, device=dev)
        vv = ds.stream_torch(w.seed, ds.STREAM_V, w.B, c0, chunk, w.Hkv, w.D, device=dev)
        layer.append(kk, vv)
    del kk, vv
    q = ds.stream_torch(w.seed, ds.STREAM_Q, w.B, w.context, w.decode_steps, w.Hq, w.D, device=dev)
    kn = ds.stream_torch(w.seed, ds.STREAM_K, w.B, w.context, w.decode_steps, w.Hkv, w.D, device=dev)
    vn = ds.stream_torch(w.seed, ds.STREAM_V, w.B, w.context, w.decode_steps, w.Hkv, w.D, device=dev)
    qs = [q[:, s].contiguous() for s in range(w.decode_steps)]
    ks = [kn[:, s:s + 1].contiguous() for s in range(w.decode_steps)]
    vs = [vn[:, s:s + 1].contiguous() for s in range(w.decode_steps)]
    o = torch.empty_like(qs[0])
    stream = torch.cuda.current_stream()
    layer.decode(qs[0], out=o, stream=stream)  # the decode kernel loaded before the timed loop
    torch.cuda.synchronize()
    ev = []
    clocks = ClockSampler(dev.index)
    clocks.start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(steps):
        layer.append(ks[s], vs[s])
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        layer.decode(qs[s], out=o, stream=stream)
        b.record(stream)
        ev.append((a, b, layer.n))
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if duo_device_error():
        raise RuntimeError("a kernel gave up a bounded wait")
    # the first steps warm up; report the rest
    warm = min(3, steps - 1)
    times = [a.elapsed_time(b) for a, b, _ in ev][warm:]
    count = wl.decode_bytes_kv4 if kv4 else wl.decode_bytes
    nbytes = [sum(count(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, kinds, n)) for _, _, n in ev][warm:]
    avg_ms = sum(times) / len(times)
    gbs = sum(nbytes) / (sum(times) * 1e-3) / 1e9
    step_ms = t0.elapsed_time(t1) / steps
    peak = peaks["hbm_gbs"]
    layer.close()
    return {"workload": w.name, "value": round(gbs, 1), "unit": "GB/s", "decode_ms": round(avg_ms, 4),
            "step_ms_with_append": round(step_ms, 4), "bytes_per_step": int(sum(nbytes) / len(nbytes)),
            "steps_timed": len(times), "steps_run": steps,
            # append, decode, merge (a million-token decode is always split over CTAs)
            "gpu_launches": 3 * steps,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4),
                         "traffic": None if paged_block else measured_traffic("decode_kv4" if kv4 else "decode"),
                         "kernel": f"decode_kernel<{w.D},{w.Hq // w.Hkv},"
                                   f"{('kv4' if kv4 else 'plain') + (' paged' if paged_block else '')}>"},
            "tokens_per_s": round(1e3 / (sum(times) / len(times)), 1), "clocks": clk}


def bench_decode_graph(w, peaks):
    """Batched decode with per-sequence lengths held on the device: one step (append one
    token to every sequence, then decode) is captured once in a CUDA graph and replayed
    for every decode step of the workload."""
    import torch

    import duo_synth as ds
    from streaming_kv_cache_duo_gb300 import DuoLayer, duo_device_error, workload as wl

    dev = torch.device("cuda", torch.cuda.current_device())
    kinds = w.is_retrieval
    max_len = w.context + w.decode_steps
    layer = DuoLayer(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, max_len, kinds, device=dev)
    chunk = 65536
    for c0 in range(0, w.context, chunk):
        T = min(chunk, w.context - c0)
        kk = ds.stream_torch(w.seed, ds.STREAM_K, w.B, c0, T, w.Hkv, w.D, device=dev)
        vv = ds.stream_torch(w.seed, ds.STREAM_V, w.B, c0, T, w.Hkv, w.D, device=dev)
        layer.append(kk, vv)
        del kk, vv
    q = ds.stream_torch(w.seed, ds.STREAM_Q, w.B, w.context, w.decode_steps, w.Hq, w.D, device=dev)
    kn = ds.stream_torch(w.seed, ds.STREAM_K, w.B, w.context, w.decode_steps, w.Hkv, w.D, device=dev)
    vn = ds.stream_torch(w.seed, ds.STREAM_V, w.B, w.context, w.decode_steps, w.Hkv, w.D, device=dev)
    seq_lens = torch.full((w.B,), w.context, dtype=torch.int32, device=dev)
    # one step's inputs (q, then the new token's k and v) side by side in one buffer, as an
    # engine would hand them over, so that staging a step is one copy
    nq, nk = w.B * w.Hq * w.D, w.B * w.Hkv * w.D
    steps_in = torch.cat([q.permute(1, 0, 2, 3).reshape(w.decode_steps, nq),
                          kn.permute(1, 0, 2, 3).reshape(w.decode_steps, nk),
                          vn.permute(1, 0, 2, 3).reshape(w.decode_steps, nk)], dim=1).contiguous()
    del q, kn, vn
    stage = torch.empty(nq + 2 * nk, dtype=torch.bfloat16, device=dev)
    sq = stage[:nq].view(w.B, w.Hq, w.D)
    sk = stage[nq:nq + nk].view(w.B, 1, w.Hkv, w.D)
    sv = stage[nq + nk:].view(w.B, 1, w.Hkv, w.D)
    so = torch.empty_like(sq)
    stage.copy_(steps_in[0])
    layer.append_varlen(sk, sv, seq_lens)  # eager step 0 (loads the kernels before capture)
    layer.decode_varlen(sq, seq_lens, max_len, out=so)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.append_varlen(sk, sv, seq_lens)
        layer.decode_varlen(sq, seq_lens, max_len, out=so)
    stream = torch.cuda.current_stream()
    steps = w.decode_steps - 1
    clocks = ClockSampler(dev.index)
    clocks.start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s_ in range(1, w.decode_steps):
        stage.copy_(steps_in[s_])
        graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if duo_device_error():
        raise RuntimeError("a kernel reported an error")
    ms = t0.elapsed_time(t1) / steps
    nbytes = sum(sum(wl.decode_bytes(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, kinds, w.context + s_ + 1))
                 for s_ in range(1, w.decode_steps)) / steps
    gbs = nbytes / (ms * 1e-3) / 1e9
    layer.close()
    return {"workload": w.name, "value": round(gbs, 1), "unit": "GB/s", "step_ms": round(ms, 4),
            "bytes_per_step": int(nbytes), "steps_timed": steps,
            "how": "device-held sequence lengths; (append + decode) captured once in a CUDA graph and "
                   "replayed; step time includes the copy staging the step's q, k and v",
            "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4), "clocks": clk,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": measured_traffic("decode_batched"),
                         "kernel": f"decode_kernel<{w.D},{w.Hq // w.Hkv},plain> (device lengths)"},
            "gpu_launches_per_step": 3}  # append, decode, merge of the split units


def bench_chunked(w, steps, warmup, peaks, paged_block=0, pool=False, kv4=False):
    """Chunked prefill against the growing cache: one step = for each chunk, prefill of
    the chunk (keys: cache before it + the chunk) then its append."""
    import torch

    import duo_synth as ds
    from streaming_kv_cache_duo_gb300 import DuoLayer, duo_attn_prefill_select, duo_device_error, workload as wl

    dev = torch.device("cuda", torch.cuda.current_device())
    L, C = w.prefill_len, w.chunk
    kinds = w.is_retrieval
    layer = make_layer(w, L, dev, paged_block, pool, kv4)
    q = ds.stream_torch(w.seed, ds.STREAM_Q, w.B, 0, L, w.Hq, w.D, device=dev)
    k = ds.stream_torch(w.seed, ds.STREAM_K, w.B, 0, L, w.Hkv, w.D, device=dev)
    v = ds.stream_torch(w.seed, ds.STREAM_V, w.B, 0, L, w.Hkv, w.D, device=dev)
    chunks = [(c0, min(C, L - c0)) for c0 in range(0, L, C)]
    qs = [q[:, c0:c0 + T].contiguous() for c0, T in chunks]
    ks = [k[:, c0:c0 + T].contiguous() for c0, T in chunks]
    vs = [v[:, c0:c0 + T].contiguous() for c0, T in chunks]
    os_ = [torch.empty_like(x) for x in qs]
    flops = sum(sum(wl.prefill_flops(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, kinds, T, c0)) for c0, T in chunks)
    fr = sum(wl.prefill_flops(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, kinds, T, c0)[0] for c0, T in chunks)
    stream = torch.cuda.current_stream()
    pre = []

    def step(record):
        layer.reset()
        for i, (c0, T) in enumerate(chunks):
            a = torch.cuda.Event(enable_timing=True) if record else None
            b = torch.cuda.Event(enable_timing=True) if record else None
            if record:
                a.record(stream)
            layer.prefill(qs[i], ks[i], vs[i], out=os_[i], stream=stream)
            if record:
                b.record(stream)
                pre.append((a, b))
            layer.append(ks[i], vs[i])

    for _ in range(warmup):
        step(False)
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    clocks.start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step(True)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if duo_device_error():
        raise RuntimeError("a kernel reported an error")
    ms = t0.elapsed_time(t1) / steps
    pre_ms = sum(a.elapsed_time(b) for a, b in pre) / steps
    layer.close()
    # traffic of one step's prefill launches, from the ncu capture of the contiguous layouts
    traffic = None if paged_block else measured_traffic("prefill_chunked_kv4" if kv4 else "prefill_chunked")
    return {"value": flops / (ms * 1e-3) / 1e12, "ms_per_step": ms, "flops": flops, "retrieval_flops": fr,
            "prefill_ms": pre_ms, "append_ms": ms - pre_ms, "launches": 2 * len(chunks) * steps, "clocks": clk,
            "roofline": {"bound": "tensor", "achieved": round(flops / (pre_ms * 1e-3) / 1e12, 2),
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(flops / (pre_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                         "traffic": traffic, "traffic_is": "sum over the step's 8 prefill launches",
                         "kernel": f"prefill_kernel<{w.D}> ({len(chunks)} launches per step)",
                         "flops_per_step": flops}}


def bench_tiny(w, steps, warmup, peaks):
    """The tiny workload end to end on the device: one step = reset the caches, prefill
    the 256-token prompt (all heads, one launch), append it, then 16 decode steps (append
    one token, decode it). Timed eagerly (every call launched from the host) and as one
    CUDA graph of the whole step replayed; both are launch-bound, so the figure of
    merit is microseconds per step."""
    import torch

    import duo_synth as ds
    from streaming_kv_cache_duo_gb300 import DuoLayer, duo_device_error, workload as wl

    dev = torch.device("cuda", torch.cuda.current_device())
    L, n_dec = w.prefill_len, w.decode_steps
    kinds = w.is_retrieval
    layer = DuoLayer(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, L + n_dec, kinds, device=dev)
    gen = lambda st, H: ds.stream_torch(w.seed, st, w.B, 0, L + n_dec, H, w.D, device=dev)
    q, k, v = gen(ds.STREAM_Q, w.Hq), gen(ds.STREAM_K, w.Hkv), gen(ds.STREAM_V, w.Hkv)
    qp, kp, vp = (x[:, :L].contiguous() for x in (q, k, v))
    qd = [q[:, L + s].contiguous() for s in range(n_dec)]
    kd = [k[:, L + s:L + s + 1].contiguous() for s in range(n_dec)]
    vd = [v[:, L + s:L + s + 1].contiguous() for s in range(n_dec)]
    op = torch.empty_like(qp)
    od = torch.empty_like(qd[0])

    def step():
        stream = torch.cuda.current_stream()  # the capture stream while a graph is captured
        layer.reset(stream=stream)
        layer.prefill(qp, kp, vp, out=op, stream=stream)
        layer.append(kp, vp, stream=stream)
        for s_ in range(n_dec):
            layer.append(kd[s_], vd[s_], stream=stream)
            layer.decode(qd[s_], out=od, stream=stream)

    stream = torch.cuda.current_stream()

    def timed(fn, n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clocks = ClockSampler(dev.index)
        clocks.start()
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / n, clocks.stop()

    n = max(steps, 20)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    eager_us, clk = timed(step, n)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    graph_us, clk_g = timed(graph.replay, n)
    if duo_device_error():
        raise RuntimeError("a kernel reported an error")
    layer.close()
    fr, fs = wl.prefill_flops(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, kinds, L)
    dec_bytes = sum(sum(wl.decode_bytes(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, kinds, L + s_ + 1)) for s_ in range(n_dec))
    return {"workload": w.name, "us_per_step": round(eager_us, 2), "us_per_step_graph": round(graph_us, 2),
            "steps_timed": n, "prefill_flops": fr + fs, "decode_bytes_per_step": dec_bytes,
            "gpu_launches_per_step": 3 + 2 * n_dec, "clocks": clk, "clocks_graph": clk_g,
            "how": "reset + prefill (256 tokens) + append + 16 x (append 1, decode 1); eager launches, and the "
                   "same step captured once as a CUDA graph and replayed; launch-bound"}


def oracle_decode_sample(w, steps_pick, batches, budget_s):
    """Time the CPU oracle's decode (what the caches hold after the step's append, the
    float64 softmax over it) for the picked decode steps and sequences, every KV head:
    retrieval heads read every stored key, streaming heads their sink + ring slots.
    Inputs are regenerated on the host (excluded from the time). Stops after the step
    that passes `budget_s` of oracle time."""
    import numpy as np

    import duo_synth as ds
    import oracle
    from streaming_kv_cache_duo_gb300 import workload as wl

    g = w.Hq // w.Hkv
    kinds = w.is_retrieval
    spent, nbytes, done = 0.0, 0, []
    for s_ in steps_pick:
        p = w.context + s_
        for b in batches:
            Qp = ds.stream_f64(w.seed, ds.STREAM_Q, w.B, p, 1, w.Hq, w.D, batches=[b])[0, 0]
            for h in range(w.Hkv):
                if kinds[h]:
                    K = ds.head_stream_f64(w.seed, ds.STREAM_K, b, h, 0, p + 1, w.D, workers=8)
                    V = ds.head_stream_f64(w.seed, ds.STREAM_V, b, h, 0, p + 1, w.D, workers=8)
                    kpos = np.arange(p + 1)
                else:
                    sim = oracle.RingCacheSim(w.S, w.R)
                    sim.append(p + 1)
                    kpos = np.array([x for x in sim.positions() if x >= 0])
                    K = np.stack([ds.stream_f64(w.seed, ds.STREAM_K, w.B, int(t), 1, w.Hkv, w.D,
                                                heads=[h], batches=[b])[0, 0, 0] for t in kpos])
                    V = np.stack([ds.stream_f64(w.seed, ds.STREAM_V, w.B, int(t), 1, w.Hkv, w.D,
                                                heads=[h], batches=[b])[0, 0, 0] for t in kpos])
                t0 = time.perf_counter()
                oracle.attend_rows(Qp[h * g:(h + 1) * g], [p] * g, K, V, kpos, kinds[h], w.S, w.R)
                spent += time.perf_counter() - t0
            r, st, _ = wl.decode_bytes(1, w.Hq, w.Hkv, w.D, w.S, w.R, kinds, p + 1)
            nbytes += r + st
            done.append((s_, b))
        if spent > budget_s:
            break
    return {"value": round(nbytes / spent / 1e9, 3), "unit": "GB/s", "cores": _threads_used(), "kind": "oracle",
            "s_per_sequence_step": round(spent / len(done), 3),
            "sample": f"{len(done)} (step, sequence) decodes of {w.name}, steps {sorted({d[0] for d in done})}, "
                      f"sequences {sorted({d[1] for d in done})}, every KV head ({spent:.1f} s of attention "
                      f"work, input generation excluded); GB/s = KV bytes the method reads / oracle time"}


# ----------------------------------------------------------------------------- oracle arm
def oracle_prefill_sample(w, budget_s):
    """Time the CPU oracle on sampled rows of the prefill (rows of every head kind)."""
    import numpy as np

    import duo_synth as ds
    import oracle
    from streaming_kv_cache_duo_gb300 import workload as wl

    L = w.prefill_len
    g = w.Hq // w.Hkv
    rng = np.random.default_rng(0)
    kinds = w.is_retrieval
    t_begin = time.perf_counter()
    flops = 0
    rows_done = 0
    cache = {}
    gen_s = 0.0
    while time.perf_counter() - t_begin < budget_s:
        hq = int(rng.integers(0, w.Hq))
        hk = hq // g
        if hk not in cache:
            t = time.perf_counter()
            cache[hk] = (ds.head_stream_f64(w.seed, ds.STREAM_K, 0, hk, 0, L, w.D, workers=4),
                         ds.head_stream_f64(w.seed, ds.STREAM_V, 0, hk, 0, L, w.D, workers=4))
            gen_s += time.perf_counter() - t
        rows = rng.integers(0, L, 8)
        Q = ds.stream_f64(w.seed, ds.STREAM_Q, 1, 0, L, w.Hq, w.D, heads=[hq])[0, rows, 0]
        oracle.attend_rows(Q, rows, cache[hk][0], cache[hk][1], np.arange(L), kinds[hk], w.S, w.R)
        for i in rows:
            pairs = (i + 1) if kinds[hk] else min(int(i) + 1, w.S + w.R)
            flops += 4 * w.D * pairs
        rows_done += len(rows)
    elapsed = time.perf_counter() - t_begin - gen_s
    total_flops = sum(wl.prefill_flops(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, kinds, L))
    return {"value": flops / elapsed / 1e12, "unit": "TFLOP/s", "cores": _threads_used(), "kind": "oracle",
            "sample": f"{rows_done} random query rows of random heads of the 32768-token prefill "
                      f"({elapsed:.1f} s of attention work, input generation excluded); full prefill "
                      f"extrapolates to {total_flops / (flops / elapsed) / 3600:.1f} h"}


def _threads_used():
    try:
        from threadpoolctl import threadpool_info
        return max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
    except Exception:
        v = os.environ.get("OMP_NUM_THREADS")
        return int(v) if v else (os.cpu_count() or 1)


def prefill_config(w, world):
    """`config` of the one-shot prefill line, the same for both arms."""
    in_bytes = w.B * w.prefill_len * (w.Hq + 2 * w.Hkv) * w.D * 2
    l2 = ((f"L2 flushed before every step (inputs {in_bytes / 2**20:.1f} MiB fit in the 129 MB L2; "
           "256 MiB write outside the step's events)") if in_bytes < L2_BYTES else
          (f"no flush: per-step inputs (Q {w.B * w.prefill_len * w.Hq * w.D * 2 / 2**20:.0f} MiB, K/V "
           f"{w.B * w.prefill_len * w.Hkv * w.D * 2 / 2**20:.0f} MiB each) exceed the 129 MB L2"))
    return {"workload": w.name, "batch": w.B, "seq_len": w.prefill_len, "q_heads": w.Hq,
            "kv_heads": w.Hkv, "head_dim": w.D, "retrieval_kv_heads": sum(w.is_retrieval),
            "sink": w.S, "recent": w.R, "parallelism": f"replicas{world}", "l2": l2,
            "step": f"prefill (all heads, one launch) + append of the {w.prefill_len} tokens"}


def run_reference(args, w, world, rank):
    if rank != 0:
        return
    peaks, _ = load_peaks()
    budget = 4.0
    times, vals = [], []
    for _ in range(args.warmup):
        oracle_prefill_sample(w, 1.0)
    for _ in range(args.steps):
        r = oracle_prefill_sample(w, budget)
        vals.append(r["value"])
    value = sum(vals) / len(vals)
    from streaming_kv_cache_duo_gb300 import workload as wl
    full = sum(wl.prefill_flops(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, w.is_retrieval, w.prefill_len))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            # the oracle times a bounded sample of each step; a whole step at its rate:
            "ms_per_step": round(full / (value * 1e12) * 1e3, 1), "ms_per_step_is": "extrapolated from the sample",
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded counter-based generator)",
            "config": prefill_config(w, world),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": r["cores"], "kind": "oracle",
                             "sample": f"each step: {r['sample']}"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ----------------------------------------------------------------------------- main
def bench_dca(w, steps, warmup, peaks):
    """Dual Chunk Attention: one-shot prefill of the prompt (all heads full attention,
    query vector chosen by the key's chunk, per-position mscale), timed per launch;
    then the prompt's keys are appended and decode steps timed. The plain causal
    prefill of the same shape is timed beside it to show what the three query vectors
    cost."""
    import torch

    import duo_synth as ds
    from streaming_kv_cache_duo_gb300 import DuoLayer, duo_device_error, workload as wl

    dev = torch.device("cuda", torch.cuda.current_device())
    L, CL = w.prefill_len, w.dca_chunk
    kinds = [1] * w.Hkv
    layer = DuoLayer(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, L + w.decode_steps, kinds, device=dev)
    gen = lambda s, pos0, T, H: ds.stream_torch(w.seed, s, w.B, pos0, T, H, w.D, device=dev)
    q, qs, qi = gen(ds.STREAM_Q, 0, L, w.Hq), gen(ds.STREAM_Q_SUCC, 0, L, w.Hq), gen(ds.STREAM_Q_INTER, 0, L, w.Hq)
    k, v = gen(ds.STREAM_K, 0, L, w.Hkv), gen(ds.STREAM_V, 0, L, w.Hkv)
    ms_all = torch.from_numpy(ds.dca_mscale(w.B, L + w.decode_steps, CL)).to(dev)
    ms = ms_all[:, :L].contiguous()
    o = torch.empty_like(q)
    stream = torch.cuda.current_stream()
    fr, _ = wl.prefill_flops(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, kinds, L)

    def timed(fn, n):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in ev:
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / n

    n = max(3, min(steps, 10))
    for _ in range(warmup):
        layer.dca_prefill(q, qs, qi, k, v, CL, mscale=ms, out=o, stream=stream)
    torch.cuda.synchronize()
    dca_ms = timed(lambda: layer.dca_prefill(q, qs, qi, k, v, CL, mscale=ms, out=o, stream=stream), n)
    plain_ms = timed(lambda: layer.prefill(q, k, v, out=o, stream=stream), n)
    # decode: the prompt's keys into the cache, then one token per step
    layer.reset()
    layer.append(k, v)
    del q, qs, qi, o
    qd, qsd, qid = (gen(s, L, w.decode_steps, w.Hq) for s in (ds.STREAM_Q, ds.STREAM_Q_SUCC, ds.STREAM_Q_INTER))
    kd, vd = gen(ds.STREAM_K, L, w.decode_steps, w.Hkv), gen(ds.STREAM_V, L, w.decode_steps, w.Hkv)
    od = torch.empty_like(qd[:, 0])
    dec, plain_dec = [], []
    for s in range(w.decode_steps):
        layer.append(kd[:, s:s + 1].contiguous(), vd[:, s:s + 1].contiguous(), stream=stream)
        args = [x[:, s].contiguous() for x in (qd, qsd, qid)]
        m1 = ms_all[:, L + s].contiguous()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        layer.dca_decode(*args, CL, mscale=m1, out=od, stream=stream)
        b.record(stream)
        dec.append((a, b, L + s + 1))
        c, d = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c.record(stream)
        layer.decode(args[0], out=od, stream=stream)  # the plain decode of the same step, for comparison
        d.record(stream)
        plain_dec.append((c, d))
    torch.cuda.synchronize()
    if duo_device_error():
        raise RuntimeError("a kernel gave up a bounded wait")
    warm = min(3, len(dec) - 1)
    dt = [a.elapsed_time(b) for a, b, _ in dec][warm:]
    pdt = [c.elapsed_time(d) for c, d in plain_dec][warm:]
    nb = [sum(wl.decode_bytes(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, kinds, nn)) for _, _, nn in dec][warm:]
    layer.close()
    peak = peaks["bf16_tflops"]
    ach = fr / (dca_ms * 1e-3) / 1e12
    return {"value": ach, "ms": dca_ms, "plain_causal_ms": plain_ms, "flops": fr, "launches": n,
            "roofline": {"bound": "tensor", "achieved": round(ach, 2), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(ach / peak, 4), "traffic": None, "kernel": f"prefill_kernel<{w.D},dca>"},
            "decode": {"decode_ms": round(sum(dt) / len(dt), 4),
                       "gbs": round(sum(nb) / (sum(dt) * 1e-3) / 1e9, 1),
                       "frac_of_hbm": round(sum(nb) / (sum(dt) * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                       "kernel": f"decode_kernel<{w.D},{w.Hq // w.Hkv},dca>", "steps_timed": len(dt),
                       "plain_decode_ms": round(sum(pdt) / len(pdt), 4)}}


def other_workload(args, w, world, rank, peaks):
    """JSON line for the workloads other than the one-shot prefill: decode (GB/s) or
    chunked prefill (TFLOP/s)."""
    base = {"metric": METRIC, "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "higher_is_better": True,
            "data": "synthetic (seeded counter-based generator, bf16 values of mean 0, variance 1)",
            "config": {"workload": w.name, "batch": w.B, "q_heads": w.Hq, "kv_heads": w.Hkv, "head_dim": w.D,
                       "retrieval_kv_heads": sum(w.is_retrieval), "sink": w.S, "recent": w.R,
                       "parallelism": f"replicas{world}"}}
    if args.kv4:
        base["config"]["cache"] = "4-bit codes + fp16 (scale, zero) per row; bytes counted as stored"
    if args.paged:
        base["config"]["paged_block"] = args.paged
        base["config"]["streaming_heads"] = "paged pool" if args.pool else "sink + ring cache"
    if w.prefill_len and w.decode_steps and not w.dca_chunk:
        # the tiny workload: prefill then decode steps, launch-bound, microseconds per step
        r = bench_tiny(w, args.steps, args.warmup, peaks)
        base["config"].update(seq_len=w.prefill_len, decode_steps=w.decode_steps,
                              step="reset, prefill, append, 16 x (append 1, decode 1); one CUDA graph")
        line = dict(base, value=round(r["us_per_step_graph"], 2), unit="us/step", higher_is_better=False,
                    ms_per_step=round(r["us_per_step_graph"] / 1e3, 5), tiny=r,
                    gpu_launches=r["gpu_launches_per_step"] * 2 * r["steps_timed"])
    elif w.dca_chunk:
        r = bench_dca(w, args.steps, args.warmup, peaks)
        base["config"].update(seq_len=w.prefill_len, dca_chunk_len=w.dca_chunk, decode_steps=w.decode_steps,
                              step="one Dual Chunk Attention prefill launch of the prompt (all heads)")
        line = dict(base, value=round(r["value"] * world, 2), unit="TFLOP/s", ms_per_step=round(r["ms"], 4),
                    roofline=r["roofline"], gpu_launches=r["launches"],
                    plain_causal_prefill_ms=round(r["plain_causal_ms"], 4), decode=r["decode"])
    elif w.chunk:
        r = bench_chunked(w, args.steps, args.warmup, peaks, args.paged, args.pool, args.kv4)
        base["config"].update(seq_len=w.prefill_len, chunk=w.chunk,
                              step="8 x (prefill of a 4096-token chunk against the cache, append)")
        line = dict(base, value=round(r["value"] * world, 2), unit="TFLOP/s", ms_per_step=round(r["ms_per_step"], 4),
                    roofline=r["roofline"], gpu_launches=r["launches"],
                    breakdown_ms={"prefill": round(r["prefill_ms"], 4)})
    else:
        if args.paged or args.kv4 or w.B == 1:
            r = bench_decode(w, w.decode_steps, peaks, args.paged, args.pool, args.kv4)
        else:
            r = bench_decode_graph(w, peaks)
        base["config"].update(context=w.context, decode_steps=w.decode_steps)
        line = dict(base, value=round(r["value"] * world, 1), unit="GB/s", ms_per_step=r.get("step_ms",
                    r.get("step_ms_with_append")), decode=r,
                    gpu_launches=r.get("gpu_launches", 3 * r["steps_timed"]))  # append, decode, merge
    if rank == 0:
        print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="duo", choices=["duo", "reference"])
    ap.add_argument("--workload", default="llama3_8b_prefill32k")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--kv4", action="store_true",
                    help="decode and chunked workloads: caches stored as 4-bit codes with an fp16 (scale, zero) "
                         "per row (chunked prefill then dequantizes the cache tiles in the kernel)")
    ap.add_argument("--pool", action="store_true",
                    help="with --paged: streaming heads in the paged pool too (block-granular eviction)")
    ap.add_argument("--paged", type=int, default=0,
                    help="decode / chunked workloads: retrieval caches in blocks of this many tokens, scattered")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import duo_synth as ds
    w = ds.WORKLOADS[args.workload]
    rank, world, local = dist_setup()
    if args.impl == "reference":
        if w.prefill_len == 0 or w.chunk or w.dca_chunk or w.decode_steps:
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable": "the oracle arm times the one-shot "
                                  "prefill workloads only"}))
            return
        run_reference(args, w, world, rank)
        return

    import __graft_entry__
    __graft_entry__.build()
    peaks, peak_src = load_peaks()
    if w.prefill_len == 0 or w.chunk or w.dca_chunk or w.decode_steps:
        other_workload(args, w, world, rank, peaks)
        return
    res = bench_prefill(w, args.steps, args.warmup, world, peaks, not args.no_e2e)
    dec = dec_graph = chunked = tiny = None
    if not args.no_decode:
        # the other workloads, each in its own timed region with its own clock record
        dec = bench_decode(ds.WORKLOADS["decode_ctx1m"], 64, peaks)
        dec_graph = bench_decode_graph(ds.WORKLOADS["batched_decode_ctx128k"], peaks)
        wc = ds.WORKLOADS["llama2_7b_chunked_prefill32k"]
        r = bench_chunked(wc, args.steps, args.warmup, peaks)
        chunked = {"workload": wc.name, "value": round(r["value"], 2), "unit": "TFLOP/s",
                   "ms_per_step": round(r["ms_per_step"], 4), "prefill_ms": round(r["prefill_ms"], 4),
                   "append_ms": round(r["append_ms"], 4), "roofline": r["roofline"],
                   "retrieval_flops": r["retrieval_flops"], "gpu_launches": r["launches"], "clocks": r["clocks"],
                   "step": "8 x (prefill of a 4096-token chunk against the cache, append)"}
        tiny = bench_tiny(ds.WORKLOADS["tiny_prefill256_decode16"], args.steps, args.warmup, peaks)
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = oracle_prefill_sample(w, args.cpu_budget)
        if not args.no_decode:
            w5, w3 = ds.WORKLOADS["decode_ctx1m"], ds.WORKLOADS["batched_decode_ctx128k"]
            cpu["decode"] = {
                w5.name: oracle_decode_sample(w5, [0, w5.decode_steps - 1, 17], [0], args.cpu_budget / 3),
                w3.name: oracle_decode_sample(w3, [0, w3.decode_steps - 1, 101], [0, w3.B - 1, 3],
                                              args.cpu_budget / 3)}
    res["roofline"]["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json bf16_tflops, burst)" \
        if peak_src == "measured" else "fallback 1.9 PFLOP/s"
    line = {
        "metric": METRIC, "value": round(res["value"], 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["ms_per_step"], 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded counter-based generator, bf16 values of mean 0, variance 1)",
        "config": prefill_config(w, world),
        "roofline": res["roofline"],
        "prefill_retrieval_only": res["prefill_retrieval_only"],
        "decode": dec,
        "decode_batched_graph": dec_graph,
        "chunked_prefill": chunked,
        "tiny": tiny,
        "cpu_baseline": cpu,
        "e2e": res.get("e2e"),
        "clocks": res["clocks"],
        "gpu_launches": res["launches"],
        "gpu_launches_is": "prefill + append launches of the main timed region; each sub-record counts its own",
        "breakdown_ms": {"prefill": round(res["prefill_ms"], 4), "append": round(res["append_ms"], 4)},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
