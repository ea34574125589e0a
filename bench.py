#!/usr/bin/env python
"""Benchmark of the exact attention forward library on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step = one call of the hot path over one batch of synthetic input:
attn_fwd for the prefill / training workloads (one kernel launch),
attn_fwd_window for the sliding-window workload (one kernel launch), or
attn_fwd_splitkv for the decode workload (split kernel + combine kernel).
Default workload: the training shape B=4, H=16, N=4096, d=128, causal.

value: device-resident throughput (inputs already in HBM), CUDA events around
each step on the launching stream, L2 flushed (256 MB write) before every
timed step, summed over K steps, max over ranks; whole-job aggregate.
sustained: the same step back to back for about two seconds (no flush; the
inputs exceed L2), with its own clock samples.
e2e: the same metric through the same C-ABI call with host buffers: every
step copies the inputs from pinned host memory and the outputs back; the
copies of consecutive steps overlap the compute on their own streams
(e2e_serial: the same with copy in, compute and copy out one after another).
For N > 1 (torchrun) every rank runs an independent replica of the workload
(weak scaling; the path has no exchange step).

--impl reference times the fp64 CPU oracle (the correctness reference) on
the host cores, each step a bounded sample of the same workload, and prints
the same line with "impl": "reference".
"""
import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s and % of GB300 BF16 peak; decode GB/s and % of HBM peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLUSH_BYTES = 256 << 20


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def profiled_traffic(workload_name):
    """DRAM bytes per launch of the dominant kernel from the ncu summary under
    profiles/, or None when there is none or the kernel source changed since."""
    import glob
    import hashlib
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        fields = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith((" ", "|", "#")):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("workload") != workload_name or "traffic_bytes_per_launch" not in fields:
            continue
        src, _, sha = fields.get("kernel_source", "").partition(" sha256:")
        try:
            with open(os.path.join(ROOT, src), "rb") as f:
                cur = hashlib.sha256(f.read()).hexdigest()[:16]
        except OSError:
            return None
        return int(fields["traffic_bytes_per_launch"]) if cur == sha else None
    return None


# --------------------------------------------------------------------------- clocks (NVML via ctypes)
class ClockSampler:
    """Samples SM clock and clock-event reasons every few ms while running."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, torch_device_index):
        self.ok = False
        self.samples = []
        self.reason_bits = 0
        self.max_mhz = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            self.nv = nv
            self.h = ctypes.c_void_p()
            import torch
            bus = None
            try:
                props = torch.cuda.get_device_properties(torch_device_index)
                bus = "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
            except Exception:
                bus = None
            rc = 1
            if bus is not None:
                rc = nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h))
            if rc != 0:
                rc = nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(0), ctypes.byref(self.h))
            if rc != 0:
                return
            m = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(m)) == 0:
                self.max_mhz = m.value
            self.get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ok = True
        except OSError:
            self.ok = False

    def _run(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) == 0:
                self.samples.append(c.value)
            if self.get_reasons(self.h, ctypes.byref(r)) == 0:
                self.reason_bits |= r.value
            time.sleep(0.002)

    def __enter__(self):
        if self.ok:
            self._stop = threading.Event()
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "source": "unavailable"}
        reasons = [n for bit, n in sorted(self.REASONS.items()) if self.reason_bits & bit and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(self.samples), "source": "nvml"}


# --------------------------------------------------------------------------- workloads
def get_workload(name):
    from exact_io_aware_14_gb300 import workloads as W
    table = {"tiny": W.TINY, "train_causal": W.TRAIN_CAUSAL, "train": W.TRAIN, "gqa": W.GQA, "long": W.LONG,
             "window": W.WINDOW, "decode": W.DECODE, "decode_paged": W.DECODE_PAGED}
    return table[name]


def config_of(w, n_gpus):
    from exact_io_aware_14_gb300 import workloads as W
    if isinstance(w, W.Decode):
        cfg = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "max_seqlen": w.max_seqlen, "d": w.d,
               "chunk": w.chunk, "seqlens": "U[%d,%d] int32, seed %d" % (w.len_lo, w.len_hi, w.seed)}
        if w.page_size:
            cfg["page_size"] = w.page_size
            cfg["pages"] = "shuffled page pool, block table [B, max_seqlen/page_size]"
    else:
        cfg = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Nq": w.N, "Nk": w.N, "d": w.d,
               "causal": w.causal, "scale": "1/sqrt(d)"}
        if w.window is not None:
            cfg["window"] = list(w.window)
            cfg["flops"] = "4*d per visible (row, key) pair"
    cfg["l2"] = "flushed before every timed step (256 MB write)"
    cfg["parallelism"] = "replicas x%d (independent, no exchange)" % n_gpus if n_gpus > 1 else "single GPU"
    return cfg


def decode_bytes(w, seqlens):
    kv = sum(2 * int(L) * w.Hkv * w.d * 2 for L in seqlens)
    return kv + 2 * (w.B * w.Hq * w.d * 2) + w.B * w.Hq * 4


# --------------------------------------------------------------------------- CPU oracle timing
def oracle_sample_rate(w, q, k, v, seqlens, budget_s, seed):
    """Times the fp64 oracle on a seeded sample of rows sized to ~budget_s.
    Returns (value in the metric's unit, seconds, description, threads)."""
    import numpy as np
    import oracle
    from exact_io_aware_14_gb300 import workloads as W
    threads = oracle.host_threads()
    dec = isinstance(w, W.Decode)
    Nq = 1 if dec else w.N
    keys = None if dec else w.keys_per_row().tolist()

    def rows_and_work(n):
        rows = W.sample_rows(w.B, w.Hq, Nq, n, seed=seed)
        if dec:
            work = sum(2 * int(seqlens[b]) * w.d * 2 for b, _, _ in rows)   # bytes of K and V rows read
        else:
            work = sum(4.0 * keys[i] * w.d for _, _, i in rows)  # FLOPs
        return rows, work

    def run(n):
        rows, work = rows_and_work(n)
        t0 = time.perf_counter()
        oracle.attn_rows(q, k, v, rows, False if dec else w.causal, w.scale,
                         kv_len=(seqlens if dec else None), n_threads=threads,
                         window=(None if dec else w.window))
        return work, time.perf_counter() - t0, len(rows)

    n = max(threads, 16)
    work, dt, _ = run(n)
    while dt < 0.2 and n < (w.B * w.Hq * Nq):
        n *= 4
        work, dt, _ = run(n)
    n_target = int(min(w.B * w.Hq * Nq, max(n, n * budget_s / max(dt, 1e-6))))
    work, dt, nrows = run(n_target)
    whole = nrows >= w.B * w.Hq * Nq
    if dec:
        value = work / dt / 1e9
        desc = "%s%d seeded (b, hq) rows of the decode workload, all valid keys each (%.1f s)" % (
            "all " if whole else "", nrows, dt)
    else:
        value = work / dt / 1e12
        desc = "%s%d seeded query rows of the workload, every visible key (%.1f s)" % (
            "all " if whole else "", nrows, dt)
    if whole:
        desc += ": the whole workload"
    return value, dt, desc, threads


# --------------------------------------------------------------------------- our arm
def max_over_ranks(x, world):
    """Largest value of x over all ranks: the whole job is as slow as its
    slowest rank.  Works under NCCL (device tensor) and gloo (host tensor)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    if dist.get_backend() == "gloo":
        dev = torch.device("cpu")
    else:
        dev = torch.device("cuda", torch.cuda.current_device())
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def whole_job_rate(work_per_rank, ms_per_step, world, scale_unit):
    """Units every rank processed in one step over the (slowest) step time:
    N independent replicas each do `work_per_rank` per step (weak scaling)."""
    return world * work_per_rank / (ms_per_step * 1e-3) / scale_unit


def setup_workload(w, dev, rank, library=None):
    """Inputs of workload w drawn on the device (seeded CUDA generator, the
    recipe of workloads.py), outputs and workspace allocated, and one step of
    the hot path as a closure.  Returns a dict."""
    import torch
    from exact_io_aware_14_gb300 import _native, workloads as W

    stream = torch.cuda.current_stream()
    gen = torch.Generator(device=dev).manual_seed(1234 + w.seed + rank)
    dec = isinstance(w, W.Decode)

    def randn(shape, amp=1.0):
        x = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)
        if amp != 1.0:
            x.mul_(amp)
        return x.to(torch.bfloat16)

    if dec:
        q = randn((w.B, 1, w.Hq, w.d))
        k = randn((w.B, w.max_seqlen, w.Hkv, w.d))
        v = randn((w.B, w.max_seqlen, w.Hkv, w.d))
        seqlens = torch.randint(w.len_lo, w.len_hi + 1, (w.B,), generator=gen, device=dev, dtype=torch.int32)
        pos = torch.arange(w.max_seqlen, device=dev)[None, :, None, None]
        bad = pos >= seqlens.long()[:, None, None, None]
        k.masked_fill_(bad, float("nan"))
        v.masked_fill_(bad, float("nan"))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq, 1), dtype=torch.float32, device=dev)
        ws = torch.empty(_native.attn_splitkv_workspace_size(w.B, w.Hq, w.max_seqlen, w.d, w.chunk),
                         dtype=torch.uint8, device=dev)
        L_host = seqlens.cpu().tolist()
        work = decode_bytes(w, L_host)
        unit, scale_unit = "GB/s", 1e9
        launches_per_step = 2
        if w.page_size:
            # the same logical cache in a shuffled page pool (one spare page)
            mb = w.max_seqlen // w.page_size
            n_pages = w.B * mb + 1
            block_table = torch.randperm(n_pages, generator=gen, device=dev)[: w.B * mb].to(torch.int32)
            block_table = block_table.reshape(w.B, mb).contiguous()
            k_pages = torch.empty((n_pages, w.page_size, w.Hkv, w.d), dtype=torch.bfloat16, device=dev)
            v_pages = torch.empty_like(k_pages)
            idx = block_table.reshape(-1).long()
            k_pages[idx] = k.reshape(w.B * mb, w.page_size, w.Hkv, w.d)
            v_pages[idx] = v.reshape(w.B * mb, w.page_size, w.Hkv, w.d)
            dev_inputs = [q, k_pages, v_pages, block_table, seqlens]

            def step():
                rc = _native.attn_fwd_splitkv_paged(q, k_pages, v_pages, block_table, seqlens, o, lse, w.scale,
                                                    w.chunk, ws, stream)
                if rc != 0:
                    raise RuntimeError("attn_fwd_splitkv_paged: %s" % _native.status_string(rc))
        else:
            dev_inputs = [q, k, v, seqlens]

            def step():
                rc = _native.attn_fwd_splitkv(q, k, v, seqlens, o, lse, w.scale, w.chunk, ws, stream)
                if rc != 0:
                    raise RuntimeError("attn_fwd_splitkv: %s" % _native.status_string(rc))
    else:
        q = randn((w.B, w.N, w.Hq, w.d), w.amp)
        k = randn((w.B, w.N, w.Hkv, w.d), w.amp)
        v = randn((w.B, w.N, w.Hkv, w.d), w.amp)
        seqlens = None
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device=dev)
        work = w.flops()
        unit, scale_unit = "TFLOP/s", 1e12
        launches_per_step = 1
        dev_inputs = [q, k, v]

        if w.window is None:
            def step():
                rc = _native.attn_fwd(q, k, v, o, lse, w.causal, w.scale, stream, library)
                if rc != 0:
                    raise RuntimeError("attn_fwd: %s" % _native.status_string(rc))
        else:
            def step():
                rc = _native.attn_fwd_window(q, k, v, o, lse, w.causal, w.window, w.scale, stream)
                if rc != 0:
                    raise RuntimeError("attn_fwd_window: %s" % _native.status_string(rc))
    return {"step": step, "dev_inputs": dev_inputs, "oracle_inputs": (q, k, v), "outputs": (o, lse),
            "work": work, "unit": unit,
            "scale_unit": scale_unit, "launches_per_step": launches_per_step, "dec": dec, "seqlens": seqlens,
            "stream": stream}


def time_steps(st, steps, warmup, flush, local_rank, world):
    """W untimed warm-up steps, then K steps each timed with CUDA events on the
    launching stream, L2 flushed before every step, clocks sampled meanwhile.
    Returns (per-step ms list, clock summary, wall seconds)."""
    import torch
    from exact_io_aware_14_gb300 import _native

    step, stream = st["step"], st["stream"]
    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if _native.attn_get_device_status(stream) != 0:
        raise RuntimeError("device status error after warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    sampler = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    with sampler:
        for i in range(steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    wall1 = time.perf_counter()
    if world > 1:
        torch.distributed.barrier()
    if _native.attn_get_device_status(stream) != 0:
        raise RuntimeError("device status error in the timed region")
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], sampler.summary(), wall1 - wall0


def roofline_of(w, st, kernel_rate, peaks, peak_src):
    if st["dec"]:
        peak = float(peaks["hbm_gbs"])
        return {"bound": "hbm", "achieved": kernel_rate, "peak": peak, "unit": "GB/s",
                "frac": kernel_rate / peak, "traffic": profiled_traffic(w.name),
                "peak_source": "%s hbm_gbs (copy)" % peak_src,
                "kernel": "decode split + combine (one step, both launches)",
                "algorithmic_bytes_per_step": st["work"]}
    peak = float(peaks["bf16_tflops"])
    return {"bound": "tensor", "achieved": kernel_rate, "peak": peak, "unit": "TFLOP/s",
            "frac": kernel_rate / peak, "traffic": profiled_traffic(w.name),
            "peak_source": "%s bf16_tflops (burst cuBLAS)" % peak_src,
            "kernel": "prefill_fwd_kernel<%d>" % w.d, "algorithmic_flops_per_launch": st["work"]}


def read_rate_gbs(dev, nbytes=4 << 30, reps=5):
    """HBM read rate of a plain streaming read (the library's read probe: 16-byte
    loads over nbytes, several in flight per thread), best of reps, CUDA events
    on the launching stream: the read-only counterpart of the copy rate, for
    memory-bound kernels that read far more than they write."""
    import torch
    from exact_io_aware_14_gb300 import _native
    buf = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    sink = torch.zeros(1, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream()
    if _native.attn_probe_read_bandwidth(buf, sink, stream) != 0:
        raise RuntimeError("read probe failed to launch")
    torch.cuda.synchronize()
    best = None
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        _native.attn_probe_read_bandwidth(buf, sink, stream)
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        best = ms if best is None else min(best, ms)
    del buf
    return nbytes / (best * 1e-3) / 1e9


def e2e_pipelined(sets, h_in, h_out, steps, comp):
    """Milliseconds for `steps` steps, each copying its inputs from pinned host
    memory and its results back, double-buffered across three streams
    (copy in, compute on `comp`, copy out).  sets: two setup_workload dicts;
    h_in: host inputs; h_out: two lists of host outputs."""
    import torch
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event(enable_timing=False)
    comp_done, out_done = [None] * steps, [None] * steps

    def run(n):
        for i in range(n):
            st = sets[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[i - 2])  # the set's inputs were consumed
                for d_t, h_t in zip(st["dev_inputs"], h_in):
                    d_t.copy_(h_t, non_blocking=True)
                in_done = ev()
                in_done.record(s_in)
            comp.wait_event(in_done)
            if i >= 2:
                comp.wait_event(out_done[i - 2])  # the set's outputs were copied out
            st["step"]()
            comp_done[i] = ev()
            comp_done[i].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[i])
                for h_t, d_t in zip(h_out[i % 2], st["outputs"]):
                    h_t.copy_(d_t, non_blocking=True)
                out_done[i] = ev()
                out_done[i].record(s_out)

    run(2)  # warm-up
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    comp.wait_event(start)
    s_out.wait_event(start)
    run(steps)
    for i in range(max(0, steps - 2), steps):
        s_out.wait_event(out_done[i])
    end.record(s_out)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


EXTRA_WORKLOADS = ("train", "gqa", "long", "window", "decode", "decode_paged")


def run_ours(args, w, rank, world, local_rank):
    import torch
    from exact_io_aware_14_gb300 import _native, build as native_build, workloads as W

    if rank == 0:
        native_build.build()
        if args.exp2_poly:
            native_build.build_variant("exp2poly%d" % args.exp2_poly)
    if world > 1:
        torch.distributed.barrier()
        native_build.build()  # no-op once rank 0 has built it
    _native.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peaks, peak_src = load_peaks()

    library = None
    if args.exp2_poly:
        if isinstance(w, W.Decode) or w.window is not None:
            raise SystemExit("--exp2-poly applies to the attn_fwd workloads")
        library = _native.variant_lib("exp2poly%d" % args.exp2_poly)
    st = setup_workload(w, dev, rank, library)
    step, work, unit, scale_unit, dec = st["step"], st["work"], st["unit"], st["scale_unit"], st["dec"]
    stream = st["stream"]
    launches_per_step = st["launches_per_step"]
    step_ms, clocks, timed_wall = time_steps(st, args.steps, args.warmup, flush, local_rank, world)
    total_ms = max_over_ranks(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(work, ms_per_step, world, scale_unit)
    kernel_rate = work / (statistics.mean(step_ms) * 1e-3) / scale_unit

    # ---- sustained: the same step back to back for about two seconds, one
    # event pair around the block, clocks sampled meanwhile (inputs larger
    # than L2 stand in for the flush)
    sustained = None
    if not args.no_sustained and not args.no_workloads:
        in_bytes = sum(x.numel() * x.element_size() for x in st["dev_inputs"])
        n_sus = max(10, int(args.sustained_seconds * 1e3 / max(statistics.mean(step_ms), 1e-3)))
        a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sus_sampler = ClockSampler(local_rank)
        torch.cuda.synchronize()
        with sus_sampler:
            a_ev.record(stream)
            for _ in range(n_sus):
                step()
            b_ev.record(stream)
            torch.cuda.synchronize()
        if _native.attn_get_device_status(stream) != 0:
            raise RuntimeError("device status error in the sustained block")
        sus_ms = max_over_ranks(a_ev.elapsed_time(b_ev), world) / n_sus
        sustained = {"value": whole_job_rate(work, sus_ms, world, scale_unit), "unit": unit, "steps": n_sus,
                     "ms_per_step": sus_ms, "clocks": sus_sampler.summary(),
                     "l2": "not flushed: inputs of %.0f MB, larger than L2" % (in_bytes / 1e6)
                     if in_bytes > 129e6 else "not flushed; inputs of %.0f MB fit L2" % (in_bytes / 1e6)}

    # ---- e2e through host buffers (pinned), copies inside the timed region
    o, lse = st["outputs"]
    d_in = st["dev_inputs"]
    h_in = [x.cpu().pin_memory() for x in d_in]
    h_out = [[torch.empty_like(x, device="cpu").pin_memory() for x in (o, lse)] for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in h_in)
    d2h = sum(x.numel() * x.element_size() for x in h_out[0])
    e2e_steps = max(3, min(args.steps, 20))

    # serial: each step copies its inputs in, runs, and copies its result out
    # on the launching stream, one after the other
    def e2e_step():
        for d_t, h_t in zip(d_in, h_in):
            d_t.copy_(h_t, non_blocking=True)
        step()
        h_out[0][0].copy_(o, non_blocking=True)
        h_out[0][1].copy_(lse, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    es = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    for i in range(e2e_steps):
        es[i].record(stream)
        e2e_step()
        ee[i].record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(es, ee)) / e2e_steps, world)

    # pipelined: two device buffer sets; step i's input copy (its own stream)
    # overlaps step i-1's compute and step i-2's result copy (a third stream),
    # as a caller streaming batches through the same call would run it
    st_b = setup_workload(w, dev, rank, library)
    sets = [st, st_b]
    e2e_ms = max_over_ranks(e2e_pipelined(sets, h_in, h_out, e2e_steps, stream) / e2e_steps, world)
    e2e_value = whole_job_rate(work, e2e_ms, world, scale_unit)
    e2e_serial_value = whole_job_rate(work, e2e_serial_ms, world, scale_unit)
    del h_in, h_out, sets, st_b

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        qc, kc, vc = (x.cpu() for x in st["oracle_inputs"])  # the paged workload: its contiguous cache
        sl = st["seqlens"].cpu().numpy() if dec else None
        val, dt, desc, thr = oracle_sample_rate(w, qc, kc, vc, sl, args.cpu_seconds, seed=w.seed)
        cpu = {"value": val, "unit": unit, "cores": thr, "kind": "oracle", "sample": desc}
        del qc, kc, vc
    del st, d_in, o, lse

    # ---- every other workload, timed the same way in this process
    extra = {}
    if not args.no_workloads:
        read_gbs = read_rate_gbs(dev) if rank == 0 else None
        for name in EXTRA_WORKLOADS:
            w2 = get_workload(name)
            if w2.name == w.name:
                continue
            st2 = setup_workload(w2, dev, rank)
            ms2, clocks2, wall2 = time_steps(st2, args.workload_steps, args.warmup, flush, local_rank, world)
            tot2 = max_over_ranks(sum(ms2), world)
            mps2 = tot2 / args.workload_steps
            rate2 = st2["work"] / (statistics.mean(ms2) * 1e-3) / st2["scale_unit"]
            entry = {"workload": w2.name, "value": whole_job_rate(st2["work"], mps2, world, st2["scale_unit"]),
                     "unit": st2["unit"], "ms_per_step": mps2, "steps": args.workload_steps,
                     "warmup": args.warmup, "gpu_launches": st2["launches_per_step"] * args.workload_steps,
                     "roofline": roofline_of(w2, st2, rate2, peaks, peak_src), "clocks": clocks2,
                     "timed_wall_s": wall2, "config": config_of(w2, world)}
            entry["frac"] = entry["roofline"]["frac"]
            if st2["dec"] and read_gbs:
                entry["read_gbs"] = read_gbs
                entry["frac_of_read"] = rate2 / read_gbs
            extra[name] = entry
            del st2
            torch.cuda.empty_cache()
        if rank == 0 and read_gbs:
            extra["read_probe"] = {"read_gbs": read_gbs,
                                   "how": "attn_probe_read_bandwidth: one streaming read of 4 GiB with 16-byte loads, "
                                          "best of 5, CUDA events"}

    if rank != 0:
        return None
    config = config_of(w, world)
    if args.exp2_poly:
        config["exp2"] = "software exp2 for every %d-th pair of a row's exponentials (build variant exp2poly%d)" % (
            args.exp2_poly, args.exp2_poly)
    return {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) fp32 draws rounded to bf16, generated on the device",
        "config": config,
        "roofline": roofline_of(w, {"dec": dec, "work": work}, kernel_rate, peaks, peak_src),
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "ms_per_step": e2e_ms,
                "how": "pinned host buffers; step i's H2D copy (own stream) overlaps step i-1's compute and "
                       "step i-2's D2H copy (own stream), two device buffer sets; one clock from the first "
                       "copy to the last result"},
        "e2e_serial": {"value": e2e_serial_value, "unit": unit, "ms_per_step": e2e_serial_ms,
                       "how": "H2D copy, compute and D2H copy of each step one after the other on one stream"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "timed_wall_s": timed_wall,
        "sustained": sustained,
        "workloads": extra,
    }


# --------------------------------------------------------------------------- reference arm (CPU oracle)
def run_reference(args, w):
    import torch
    from exact_io_aware_14_gb300 import workloads as W
    dec = isinstance(w, W.Decode)
    # a bounded slice of the same workload on the CPU (same seeds and recipe)
    if dec:
        q, k, v, L = W.workload_decode_inputs(w)
        sl = L.numpy()
        unit = "GB/s"
    else:
        q, k, v = W.workload_inputs(w)
        sl = None
        unit = "TFLOP/s"
    per_step = max(0.2, min(8.0, args.reference_seconds / max(1, args.steps + args.warmup)))
    vals, secs, desc, thr = [], [], "", 1
    for i in range(args.warmup + args.steps):
        val, dt, desc, thr = oracle_sample_rate(w, q, k, v, sl, per_step, seed=w.seed + 17 * i)
        if i >= args.warmup:
            vals.append(val)
            secs.append(dt)
    value = statistics.mean(vals)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded N(0,1) fp32 draws rounded to bf16 (CPU generator)",
        "config": config_of(w, 1),
        "cpu_baseline": {"value": value, "unit": unit, "cores": thr, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="train_causal",
                    choices=["tiny", "train_causal", "train", "gqa", "long", "window", "decode", "decode_paged"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-oracle sample budget")
    ap.add_argument("--reference-seconds", type=float, default=90.0, help="whole reference-arm budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time only the K steps of the selected workload (no other workloads, no sustained block)")
    ap.add_argument("--no-sustained", action="store_true", help="skip the two-second back-to-back block")
    ap.add_argument("--sustained-seconds", type=float, default=2.0)
    ap.add_argument("--workload-steps", type=int, default=20, help="timed steps of each other workload")
    ap.add_argument("--exp2-poly", type=int, default=0, choices=[0, 2, 4, 8, 16],
                    help="time the build variant whose softmax computes every K-th pair of exponentials in "
                         "software (attn_fwd workloads; implies --no-workloads)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = get_workload(args.workload)
    if args.exp2_poly:
        args.no_workloads = True
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, w)), flush=True)
        return 0

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        line = run_ours(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
