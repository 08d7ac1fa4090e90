#!/usr/bin/env python3
"""Benchmark of libfattn on one GB300 (or N independent replicas).

One step = one fused attention forward through the C ABI on the workload the
headline metric is quoted on: bf16, B=2, H=32, N=M=8192, d=128, causal
(FLOPs = 4*B*H*N*M*d / 2).  Inputs (403 MB) are larger than the 129 MB L2, so
no flush is needed between steps.  The row-softmax workload (bf16
[4096, 32768], one read + one write, 537 MB) is the second headline and is
timed in its own loop on the same device; the LSE-only kernel and the fp32
attention path are timed alongside for completeness.

Prints ONE JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
on a bounded sample of the same workload instead (the reference arm).
Multi-GPU: every rank runs the full workload on its own GPU (weak scaling, no
collective on the data path); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s and % of GB300 dense BF16 peak; row-softmax GB/s vs HBM"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def recorded_traffic(kernel: str):
    """DRAM bytes per benchmark launch from profiles/traffic.json, or None when
    the kernel's sources changed since the capture (hash mismatch)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[kernel]
        h = hashlib.sha256()
        for src in rec["sources"]:
            with open(os.path.join(ROOT, "online_softmax_10_gb300", "csrc", src), "rb") as f:
                h.update(f.read())
        if h.hexdigest()[:16] != rec["sha256_16"]:
            return None
        return (rec["dram_read_bytes"] + rec["dram_write_bytes"]) * rec["scale_to_benchmark_workload"]
    except Exception:
        return None


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, world_size: int, device=None) -> float:
    """Max of a float over all ranks (identity when world_size == 1)."""
    if world_size <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, world_size: int, max_seconds: float) -> float:
    """Whole-job throughput: the units all ranks processed / the slowest rank's time."""
    return units_per_rank * world_size / max_seconds


def barrier(world_size: int):
    if world_size > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.out is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        self.out.flush()
        with open(self.out.name) as f:
            lines = [l.strip() for l in f if l.strip()]
        os.unlink(self.out.name)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        # samples under load: the upper half by power draw
        cut = statistics.median(power)
        loaded = [s for s, p in zip(sm, power) if p >= cut] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


def gpu_uuid():
    try:
        import torch
        u = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ------------------------------------------------------------------ timing
def time_launches(fn, steps: int, warmup: int, world_size: int):
    """Warm up, then time `steps` calls of fn() with CUDA events on the current
    stream: returns (total seconds, max over ranks; mean per-launch seconds)."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world_size)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start.record(stream)
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world_size)
    total = start.elapsed_time(end) / 1e3
    per = statistics.mean(a.elapsed_time(b) for a, b in evs) / 1e3
    return max_over_ranks(total, world_size, device="cuda"), per


def time_for(fn, seconds: float, warmup: int = 3, flush=None, max_launches: int = 20000):
    """Mean device seconds per fn() call over about `seconds` of launches,
    each bracketed by its own pair of CUDA events on the current stream
    (`flush`, if given, runs between launches outside the events).
    Returns (mean seconds per launch, launches)."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    fn()
    b.record(stream)
    torch.cuda.synchronize()
    est = max(a.elapsed_time(b) / 1e3, 1e-6)
    n = int(max(10, min(max_launches, math.ceil(seconds / est))))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for x, y in evs:
        if flush is not None:
            flush()
        x.record(stream)
        fn()
        y.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(x.elapsed_time(y) for x, y in evs) / 1e3, n


def time_batched(fn, launches: int, warmup: int = 3):
    """Mean device seconds per fn() call over `launches` back-to-back calls
    between one pair of CUDA events on the current stream (so the figure
    holds the gaps between launches but no per-launch event records)."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(launches):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3 / launches


def link_bandwidth(host_in, dev_in, host_out, dev_out, reps: int = 5):
    """Pinned host <-> device copy rates on the tensors one end-to-end step
    moves (one cudaMemcpyAsync per tensor): host-to-device alone,
    device-to-host alone, and both directions at once on two streams.
    Returns a dict of GB/s and the both-ways time of one step's copies."""
    import torch
    up = torch.cuda.Stream()
    down = torch.cuda.Stream()
    bi = sum(t.numel() * t.element_size() for t in host_in)
    bo = sum(t.numel() * t.element_size() for t in host_out)

    def h2d():
        with torch.cuda.stream(up):
            for d, h in zip(dev_in, host_in):
                d.copy_(h, non_blocking=True)

    def d2h():
        with torch.cuda.stream(down):
            for h, d in zip(host_out, dev_out):
                h.copy_(d, non_blocking=True)

    def timed(fn):
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            best = min(best, time.perf_counter() - t0)
        return best

    timed(h2d)
    timed(d2h)
    t_in, t_out = timed(h2d), timed(d2h)
    t_both = timed(lambda: (h2d(), d2h()))
    return {"h2d_gbs": bi / t_in / 1e9, "d2h_gbs": bo / t_out / 1e9, "both_gbs": (bi + bo) / t_both / 1e9,
            "step_copies_ms": t_both * 1e3, "h2d_bytes": bi, "d2h_bytes": bo, "reps": reps,
            "how": "best of reps, host clock around a synchronised burst; one cudaMemcpyAsync per tensor"}


def time_graph(fn, calls: int, reps: int):
    """Mean device seconds per fn() call: `calls` calls captured in one CUDA
    graph, replayed `reps` times between CUDA events (launches back to back,
    no host work between them)."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(calls):
            fn()
    g.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(reps):
        g.replay()
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3 / (calls * reps)


# ------------------------------------------------------------------ CPU oracle
def cpu_oracle_sample(w, target_s: float = 10.0, max_rows: int | None = None):
    """Time the fp64 oracle on a seeded sample of the workload's query rows.
    Returns (TFLOP/s by the workload's FLOP convention, seconds, rows, threads)."""
    import numpy as np
    import oracle
    from online_softmax_10_gb300 import inputs
    q, k, v = inputs.workload_attn_inputs(w)
    Q, K, V = oracle.as_f64(q), oracle.as_f64(k), oracle.as_f64(v)
    threads = oracle.default_threads()
    total_rows = w.B * w.H * w.N

    def flops(rows):
        i = rows % w.N
        kept = np.minimum(i + 1, w.M) if w.causal else np.full_like(i, w.M)
        return float(np.sum(4.0 * kept * w.d))

    probe = inputs.sample_rows(total_rows, 256, seed=99).numpy()
    t0 = time.perf_counter()
    oracle.attn_fwd(Q, K, V, w.scale, w.causal, rows=probe, nthreads=threads)
    tp = time.perf_counter() - t0
    n = int(len(probe) * target_s / max(tp, 1e-3))
    n = max(256, min(n, total_rows if max_rows is None else max_rows))
    rows = inputs.sample_rows(total_rows, n, seed=100).numpy()
    t0 = time.perf_counter()
    oracle.attn_fwd(Q, K, V, w.scale, w.causal, rows=rows, nthreads=threads)
    dt = time.perf_counter() - t0
    return flops(rows) / dt / 1e12, dt, len(rows), threads, flops(rows)


# ------------------------------------------------------------------ arms
def run_reference(args, world_size, rank):
    """The reference arm: the fp64 CPU oracle as it stands, on the host cores."""
    if rank != 0:
        return
    from online_softmax_10_gb300 import inputs
    import numpy as np
    import oracle
    w = inputs.ATTN_B2H32_8192_D128_CAUSAL
    q, k, v = inputs.workload_attn_inputs(w)
    Q, K, V = oracle.as_f64(q), oracle.as_f64(k), oracle.as_f64(v)
    threads = oracle.default_threads()
    total_rows = w.B * w.H * w.N
    # size one step so that warmup + steps stay within about two minutes
    probe = inputs.sample_rows(total_rows, 128, seed=99).numpy()
    t0 = time.perf_counter()
    oracle.attn_fwd(Q, K, V, w.scale, w.causal, rows=probe, nthreads=threads)
    tp = time.perf_counter() - t0
    per_step_target = min(10.0, 120.0 / max(1, args.steps + args.warmup))
    n = max(64, min(total_rows, int(len(probe) * per_step_target / max(tp, 1e-3))))
    samples = [inputs.sample_rows(total_rows, n, seed=1000 + s).numpy() for s in range(args.warmup + args.steps)]

    def fl(rows):
        i = rows % w.N
        return float(np.sum(4.0 * np.minimum(i + 1, w.M) * w.d))

    for s in range(args.warmup):
        oracle.attn_fwd(Q, K, V, w.scale, w.causal, rows=samples[s], nthreads=threads)
    t0 = time.perf_counter()
    work = 0.0
    for s in range(args.warmup, args.warmup + args.steps):
        oracle.attn_fwd(Q, K, V, w.scale, w.causal, rows=samples[s], nthreads=threads)
        work += fl(samples[s])
    dt = time.perf_counter() - t0
    value = work / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "M": w.M, "d": w.d, "causal": w.causal,
                   "sample_rows_per_step": n},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n} seeded query rows of {total_rows} per step (fp64, three-pass softmax)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world_size, rank, local_rank):
    import torch
    from online_softmax_10_gb300 import build as fbuild
    from online_softmax_10_gb300 import fattn, inputs

    torch.cuda.set_device(local_rank)
    fbuild.build()
    peaks, peak_src = load_peaks()
    w = inputs.ATTN_B2H32_8192_D128_CAUSAL
    q_h, k_h, v_h = inputs.workload_attn_inputs(w)
    q, k, v = q_h.cuda(), k_h.cuda(), v_h.cuda()
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device="cuda")

    def step():
        fattn.attn_fwd(q, k, v, w.scale, w.causal, out=o, lse=lse)

    step()
    assert fattn.device_status() == fattn.FA_OK
    # The sampler covers the contract loop and, right after it, a loop of the
    # same launches long enough (>= roofline_seconds) for the clock record and
    # the roofline's mean launch duration to rest on many samples.
    with ClockSampler(gpu_uuid()) as clk:
        total_s, per_launch_s = time_launches(step, args.steps, args.warmup, world_size)
        roof_per_s, roof_n = time_for(step, args.roofline_seconds, warmup=0)
    clocks = clk.summary()
    assert fattn.device_status() == fattn.FA_OK
    flops = w.flops()
    value = aggregate_throughput(flops, world_size, total_s / args.steps) / 1e12
    achieved = flops / roof_per_s / 1e12

    # ---- end to end through the public API with host buffers: every step
    # copies its Q, K, V in from pinned host memory and its O, LSE back out.
    # Two device input sets let step i+1's upload (copy stream) overlap step
    # i's kernel and download (compute stream); events order the hand-offs.
    qp, kp, vp = (t.pin_memory() for t in (q_h, k_h, v_h))
    op = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lp = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    dev_in = [tuple(torch.empty_like(t) for t in (q, k, v)) for _ in range(2)]
    copy_stream = torch.cuda.Stream()
    comp = torch.cuda.current_stream()
    uploaded = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    for ev in consumed:
        ev.record(comp)

    def upload(slot):
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(consumed[slot])
            for dst, src in zip(dev_in[slot], (qp, kp, vp)):
                dst.copy_(src, non_blocking=True)
            uploaded[slot].record(copy_stream)

    e2e_state = {"i": 0}

    def e2e_step():
        i = e2e_state["i"]
        slot = i % 2
        if i == 0:
            upload(0)
        upload(1 - slot)  # the next step's inputs, while this step computes
        comp.wait_event(uploaded[slot])
        qd, kd, vd = dev_in[slot]
        fattn.attn_fwd(qd, kd, vd, w.scale, w.causal, out=o, lse=lse)
        consumed[slot].record(comp)
        op.copy_(o, non_blocking=True)
        lp.copy_(lse, non_blocking=True)
        e2e_state["i"] = i + 1

    e2e_steps = max(3, min(args.steps, 30))
    e2e_total, _ = time_launches(e2e_step, e2e_steps, 2, world_size)
    torch.cuda.synchronize()
    e2e_value = aggregate_throughput(flops, world_size, e2e_total / e2e_steps) / 1e12
    h2d = sum(t.numel() * t.element_size() for t in (q_h, k_h, v_h))
    d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()
    # the host link alone, on the same pinned buffers and device tensors
    link = link_bandwidth([qp, kp, vp], list(dev_in[0]), [op, lp], [o, lse])
    # an end-to-end step can go no faster than its copies (both directions at
    # once) or its kernel, whichever is longer
    e2e_bound = flops / max(link["step_copies_ms"] / 1e3, per_launch_s) / 1e12
    del dev_in, qp, kp, vp

    # ---- row softmax workload (second headline): bf16 [4096, 32768] -> bf16 P + fp32 LSE
    rw = inputs.ROWS_4096x32768
    x = inputs.workload_rows_inputs(rw).cuda()
    p = torch.empty_like(x)
    plse = torch.empty(rw.rows, dtype=torch.float32, device="cuda")
    r_per, rsteps = time_for(lambda: fattn.softmax_rows(x, out=p, lse=plse), args.extra_seconds,
                             warmup=max(3, args.warmup))
    r_bytes = rw.rows * rw.cols * 2 * 2 + rw.rows * 4
    r_gbs = r_bytes / r_per / 1e9
    l_per, lsteps = time_for(lambda: fattn.logsumexp_rows(x, out=plse), args.extra_seconds)
    l_bytes = rw.rows * rw.cols * 2 + rw.rows * 4
    r_batch = time_batched(lambda: fattn.softmax_rows(x, out=p, lse=plse), rsteps)
    l_batch = time_batched(lambda: fattn.logsumexp_rows(x, out=plse), lsteps)
    del x, p

    # ---- split-KV on a decode-like shape (few query rows, long keys): the
    # (head, query block) units alone cover 8 of the SMs
    sq, sk, sv = (t.cuda() for t in inputs.attn_inputs(1, 8, 256, 65536, 128, torch.bfloat16, seed=6))
    s_flops = 4.0 * 8 * 256 * 65536 * 128
    nsplit = fattn.splitkv_num_splits(1, 8, 256, 65536, 128, False)
    ws = torch.empty(max(1, fattn.splitkv_workspace_bytes(1, 8, 256, 128, nsplit)), dtype=torch.uint8, device="cuda")
    so = torch.empty_like(sq)
    sl = torch.empty((1, 8, 256), dtype=torch.float32, device="cuda")
    _, s_per = time_launches(lambda: fattn.attn_fwd_splitkv(sq, sk, sv, 128 ** -0.5, False, num_splits=nsplit,
                                                           workspace=ws, out=so, lse=sl), 50, 5, world_size)
    _, u_per = time_launches(lambda: fattn.attn_fwd(sq, sk, sv, 128 ** -0.5, False, out=so, lse=sl), 20, 3,
                             world_size)
    del sq, sk, sv, ws

    # ---- the other two bf16 attention workloads: d = 64 (inputs 67 MB fit in
    # L2, so L2 is flushed between launches) and the 32768-key causal one
    peak_t = peaks["bf16_tflops"]
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    extra_attn = {}
    for ew, flush in ((inputs.ATTN_B4H16_2048_D64, lambda: flush_buf.zero_()),
                      (inputs.ATTN_B1H16_32768_D128_CAUSAL, None)):
        eq, ek, ev = (t.cuda() for t in inputs.workload_attn_inputs(ew))
        eo = torch.empty_like(eq)
        el = torch.empty((ew.B, ew.H, ew.N), dtype=torch.float32, device="cuda")
        e_per, e_n = time_for(lambda: fattn.attn_fwd(eq, ek, ev, ew.scale, ew.causal, out=eo, lse=el),
                              args.extra_seconds, flush=flush)
        assert fattn.device_status() == fattn.FA_OK
        extra_attn[ew.name] = {"value": ew.flops() / e_per / 1e12, "unit": "TFLOP/s", "us_per_launch": e_per * 1e6,
                               "frac": ew.flops() / e_per / 1e12 / peak_t, "launches": e_n,
                               "l2": "flushed (256 MB write) between launches" if flush else
                                     "inputs 403 MB > 129 MB L2, no flush"}
        del eq, ek, ev, eo, el
    del flush_buf

    # ---- fp32 attention workload (N = M = 64, d = 64): launch-latency bound
    fw = inputs.ATTN_F32_64
    fq, fk, fv = (t.cuda() for t in inputs.workload_attn_inputs(fw))
    f_total, f_per = time_launches(lambda: fattn.attn_fwd(fq, fk, fv, fw.scale, fw.causal), 200, 10, world_size)
    assert fattn.device_status() == fattn.FA_OK
    # the kernel's own time: the same call (outputs preallocated) captured 50
    # times in a CUDA graph and replayed, so no host work paces the launches
    fo, fl = torch.empty_like(fq), torch.empty(fq.shape[:3], dtype=torch.float32, device=fq.device)
    f_dev = time_graph(lambda: fattn.attn_fwd(fq, fk, fv, fw.scale, fw.causal, out=fo, lse=fl), 50, 5)
    assert fattn.device_status() == fattn.FA_OK

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        tf, dt, nrows, threads, _ = cpu_oracle_sample(w, target_s=args.cpu_seconds)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{nrows} seeded query rows of {w.B * w.H * w.N} ({dt:.1f} s, fp64 three-pass softmax, "
                         f"FLOPs by the same 4*kept*d convention)"}

    peak_sus = peaks["bf16_tflops_sustained"]
    alg_bytes = (q.numel() + k.numel() + v.numel() + o.numel()) * 2 + lse.numel() * 4
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world_size, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_s / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "M": w.M, "d": w.d, "causal": w.causal,
                   "inputs": "Q,K,V i.i.d. N(0,1) seed 3, bf16", "l2": "inputs 403 MB > 129 MB L2, no flush",
                   "parallelism": f"replicas x{world_size}"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_sus, "unit": "TFLOP/s",
                     "frac": achieved / peak_sus, "frac_of_burst": achieved / peak_t,
                     "traffic": args.traffic if args.traffic is not None else recorded_traffic("attn_bf16_tc"),
                     "algorithmic_bytes": alg_bytes,
                     "peak_source": f"bf16_tflops_sustained ({peak_src}): the kernel is timed over a "
                                    f"{args.roofline_seconds:g} s back-to-back loop; burst {peak_t:g} beside it",
                     "launches": roof_n, "us_per_launch": roof_per_s * 1e6,
                     "timed": f"{roof_n} back-to-back launches after the contract loop, one event pair each",
                     "clocks_samples": clocks.get("samples"), "sm_mhz": clocks.get("sm_mhz")},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipelining": "step i+1's host-to-device copy overlaps step i's kernel and device-to-host copy",
                "link": link, "bound": e2e_bound, "frac_of_bound": e2e_value / e2e_bound},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "row_softmax": {"workload": rw.name, "value": r_gbs, "unit": "GB/s", "us_per_launch": r_per * 1e6,
                        "roofline": {"bound": "hbm", "achieved": r_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                     "frac": r_gbs / peaks["hbm_gbs"],
                                     "traffic": args.rows_traffic if args.rows_traffic is not None
                                     else recorded_traffic("softmax_rows_tma"),
                                     "bytes_per_launch": r_bytes, "peak_source": f"hbm_gbs, {peak_src}"},
                        "launches": rsteps, "l2": "input 268 MB > 129 MB L2, no flush",
                        "timed": "one event pair per launch",
                        "batched": {"us_per_launch": r_batch * 1e6, "value": r_bytes / r_batch / 1e9,
                                    "frac": r_bytes / r_batch / 1e9 / peaks["hbm_gbs"], "launches": rsteps,
                                    "timed": "one event pair around the launches, back to back"}},
        "logsumexp_rows": {"workload": rw.name, "value": l_bytes / l_per / 1e9, "unit": "GB/s",
                           "us_per_launch": l_per * 1e6, "frac": l_bytes / l_per / 1e9 / peaks["hbm_gbs"],
                           "traffic": recorded_traffic("logsumexp_rows_tma"), "bytes_per_launch": l_bytes,
                           "launches": lsteps, "timed": "one event pair per launch",
                           "batched": {"us_per_launch": l_batch * 1e6, "value": l_bytes / l_batch / 1e9,
                                       "frac": l_bytes / l_batch / 1e9 / peaks["hbm_gbs"], "launches": lsteps,
                                       "timed": "one event pair around the launches, back to back"}},
        "attn_b4_h16_n2048_d64": extra_attn[inputs.ATTN_B4H16_2048_D64.name],
        "attn_b1_h16_n32768_d128_causal": extra_attn[inputs.ATTN_B1H16_32768_D128_CAUSAL.name],
        "attn_splitkv": {"workload": "attn_bf16_B1_H8_N256_M65536_d128 (decode-like)", "splits": nsplit,
                         "value": s_flops / s_per / 1e12, "unit": "TFLOP/s", "us_per_launch": s_per * 1e6,
                         "unsplit_value": s_flops / u_per / 1e12},
        "attn_f32": {"workload": fw.name, "us_per_launch": f_per * 1e6,
                     "value": fw.flops() / f_per / 1e12, "unit": "TFLOP/s",
                     "device_us_per_launch": f_dev * 1e6},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_only(args):
    """One kernel on one shape, for profiling captures (prints a short JSON
    line that is not the benchmark's contract line)."""
    import torch
    from online_softmax_10_gb300 import build as fbuild
    from online_softmax_10_gb300 import fattn, inputs
    fbuild.build()
    torch.cuda.set_device(0)
    if args.only in ("attn", "splitkv"):
        B, H, N, M, d, causal = (int(x) for x in args.shape.split(","))
        dt = torch.float32 if args.f32 else torch.bfloat16
        q, k, v = (t.cuda() for t in inputs.attn_inputs(B, H, N, M, d, dt, seed=3))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        if args.only == "attn":
            fn = lambda: fattn.attn_fwd(q, k, v, 1.0 / math.sqrt(d), bool(causal), out=o, lse=lse)
        else:
            S = fattn.splitkv_num_splits(B, H, N, M, d, bool(causal))
            ws = torch.empty(max(1, fattn.splitkv_workspace_bytes(B, H, N, d, S)), dtype=torch.uint8, device="cuda")
            fn = lambda: fattn.attn_fwd_splitkv(q, k, v, 1.0 / math.sqrt(d), bool(causal), num_splits=S,
                                                workspace=ws, out=o, lse=lse)
        work = 4.0 * B * H * N * M * d / (2 if causal else 1)
        unit, scale = "TFLOP/s", 1e12
    else:
        rows, cols = (int(x) for x in args.shape.split(","))
        x = inputs.rows_inputs(rows, cols, torch.bfloat16, seed=1).cuda()
        lse = torch.empty(rows, dtype=torch.float32, device="cuda")
        if args.only == "rows":
            p = torch.empty_like(x)
            fn = lambda: fattn.softmax_rows(x, out=p, lse=lse)
            work = rows * cols * 4.0 + rows * 4
        else:
            fn = lambda: fattn.logsumexp_rows(x, out=lse)
            work = rows * cols * 2.0 + rows * 4
        unit, scale = "GB/s", 1e9
    with ClockSampler(gpu_uuid()) as clk:
        total, per = time_launches(fn, args.steps, args.warmup, 1)
    clocks = clk.summary()
    assert fattn.device_status() == fattn.FA_OK
    print(json.dumps({"only": args.only, "shape": args.shape, "launches": args.steps,
                      "us_per_launch": per * 1e6, "value": work / per / scale, "unit": unit,
                      "sm_mhz": clocks.get("sm_mhz"), "clock_samples": clocks.get("samples"),
                      "reasons": clocks.get("reasons")}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--roofline-seconds", type=float, default=1.5,
                    help="length of the back-to-back loop the roofline's launch duration is taken from")
    ap.add_argument("--extra-seconds", type=float, default=0.5,
                    help="seconds of launches for each of the other attention workloads")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per attention launch, if captured for the current kernel")
    ap.add_argument("--rows-traffic", type=float, default=None,
                    help="ncu dram bytes per row-softmax launch, if captured for the current kernel")
    ap.add_argument("--only", choices=["attn", "splitkv", "rows", "lse"], default=None,
                    help="time one kernel on --shape only (profiling aid; not the contract line)")
    ap.add_argument("--shape", default=None, help="attn/splitkv: B,H,N,M,d,causal   rows/lse: rows,cols")
    ap.add_argument("--f32", action="store_true", help="with --only attn: fp32 inputs")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.only:
        run_only(args)
        return
    world_size, rank, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, world_size, rank)
        return
    if world_size > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, world_size, rank, local_rank)
    finally:
        if world_size > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
