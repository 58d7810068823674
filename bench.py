#!/usr/bin/env python
"""Throughput of continuity-aware draft-tree construction on GB300.

One step = one dart_tree_build call over a batch: every logit row streamed
once (log-softmax + top-k), then every tree grown depth by depth (expand,
n-gram score, top-W), with token/parent/depth ids and ancestor masks written.

Prints one JSON line: trees/s over the whole job (value), the streaming
kernel's achieved HBM bandwidth against the measured copy peak (roofline),
the same metric end to end with host buffers (e2e), and the CPU oracle on a
bounded sample of the same workload (cpu_baseline).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 2] [--impl ours|reference]

Under torchrun every rank builds its own batch (weak scaling, no collective
on the data path); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

DEFAULT_CONFIG = 2
METRIC = "draft trees/sec and achieved HBM GB/s (% of GB300 peak) at 1 GPU vs CPU oracle"


def workload_name(i: int) -> str:
    c = synth.CONFIGS[i]
    return (f"config {i}: B={c['B']} d={c['d']} V={c['V']} {c['dtype']} logits {c['recipe'][0]}, "
            f"T={c['T']} k={c['k']} W={c['W']}, {c['n']}-gram table {c['M']} keys, "
            f"lambda={c['lam']} beta={c['beta']}")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--config", type=int, default=DEFAULT_CONFIG)
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the CPU-baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-per-config", action="store_true", help="skip the other configs' records")
    p.add_argument("--probe-sfu", action="store_true",
                   help="only measure the exponential unit's throughput (one JSON line)")
    p.add_argument("--probe-stream", action="store_true",
                   help="only sweep the streaming-read probes (one JSON line per shape)")
    return p.parse_args()


# ------------------------------------------------------------------ ranks

def dist_setup():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, local):
    import torch
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- clocks

CLOCK_QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def clocks_start(gpu_index: int):
    """Starts nvidia-smi sampling every 20 ms; waits (up to 3 s) for its first line."""
    try:
        f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        p = subprocess.Popen(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={CLOCK_QUERY}",
                              "--format=csv,noheader,nounits", "-lms", "20"],
                             stdout=f, stderr=subprocess.DEVNULL)
    except (OSError, FileNotFoundError):
        return None, None
    t0 = time.time()
    while time.time() - t0 < 3.0 and os.path.getsize(f.name) == 0:
        time.sleep(0.02)
    return p, f.name


def _stamp(text: str):
    for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
        try:
            return datetime.datetime.strptime(text, fmt).timestamp()
        except ValueError:
            pass
    return None


def clocks_stop(handle, window):
    """Median SM clock and throttle reasons of the samples inside `window`
    (wall-clock start, end of the timed regions); if none fall inside it, of
    every sample since warm-up, and the result says so."""
    p, path = handle
    if p is None:
        return None
    p.terminate()
    try:
        p.wait(timeout=5)
    except subprocess.TimeoutExpired:
        p.kill()
    rows = []
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in open(path):
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            rows.append((_stamp(parts[0]), float(parts[2]), float(parts[3]),
                         {n for n, v in zip(names, parts[6:10]) if v.lower() == "active"}))
        except ValueError:
            continue
    os.unlink(path)
    inside = [r for r in rows if r[0] is not None and window[0] - 0.02 <= r[0] <= window[1] + 0.02]
    used, where = (inside, "timed region") if inside else (rows, "warm-up through timed region")
    if not used:
        return None
    reasons = set().union(*[r[3] for r in used])
    return {"sm_mhz": statistics.median(r[1] for r in used), "sm_max_mhz": max(r[2] for r in used),
            "reasons": sorted(reasons), "samples": len(used), "window": where}


# ------------------------------------------------------------ measured peaks

def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in ("dart_rows.cu", "dart_common.cuh"):
        with open(os.path.join(ROOT, "draft_tree_construction_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def k1_traffic(config: int):
    """DRAM bytes (read + write) of one launch of the streaming kernel on `config`
    from the committed ncu capture of that config, or None when there is none or
    the kernel source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "row_stream_dram.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != kernel_source_hash():
        return None
    c = rec.get("configs", {}).get(str(config))
    if not c:
        return None
    return c["dram_bytes_read"] + c["dram_bytes_write"]


# -------------------------------------------------------------- CPU oracle

def _sub_case(case, S):
    return synth.Case(name=case.name, B=S, d=case.d, V=case.V, dtype=case.dtype, T=case.T,
                      k=case.k, W=case.W, n=case.n, lam=case.lam, beta=case.beta,
                      logits=case.logits[:S], ctx=case.ctx[:S], ng_keys=case.ng_keys,
                      ng_vals=case.ng_vals)


def oracle_sample(case, budget_s: float, ngram=None):
    """Times the oracle on the first S trees of `case` (S sized to the budget)."""
    import oracle
    if ngram is None and case.n >= 2:
        ngram = oracle.NGram(case.n, case.ng_keys, case.ng_vals)
    threads = os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle.tree_build(_sub_case(case, 1), ngram=ngram, threads=threads)
    t1 = time.perf_counter() - t0
    S = int(max(1, min(case.B, math.floor(budget_s / max(t1, 1e-6)))))
    t0 = time.perf_counter()
    oracle.tree_build(_sub_case(case, S), ngram=ngram, threads=threads)
    dt = time.perf_counter() - t0
    return S, dt, threads, ngram


def oracle_single_core(case, budget_s: float, ngram):
    """Times the oracle on one host core (S trees sized to the budget)."""
    import oracle
    t0 = time.perf_counter()
    oracle.tree_build(_sub_case(case, 1), ngram=ngram, threads=1)
    t1 = time.perf_counter() - t0
    S = int(max(1, min(case.B, math.floor(budget_s / max(t1, 1e-6)))))
    t0 = time.perf_counter()
    oracle.tree_build(_sub_case(case, S), ngram=ngram, threads=1)
    return S, time.perf_counter() - t0


def run_probe_sfu(args):
    """Exponentials per second the GPU sustains (ex2.approx, the row pass's
    exponential), against what the row pass needs at 70% of the measured copy
    bandwidth on 2-byte logits (one exponential per logit)."""
    import ctypes as C
    import torch
    import draft_tree_construction_gb300 as D
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    D.build()
    L = D.lib()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks, threads, iters = sms * 4, 512, 4096
    out = torch.empty(blocks * threads, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def go():
        rc = L.dart_probe_ex2(blocks, threads, iters, C.c_void_p(out.data_ptr()), C.c_void_p(stream.cuda_stream))
        assert rc == 0, rc

    for _ in range(3):
        go()
    torch.cuda.synchronize(dev)
    clk = clocks_start(0)
    t0 = time.time()
    times = []
    for _ in range(10):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        go()
        b.record(stream)
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b))
    clocks = clocks_stop(clk, (t0, time.time()))
    ms = statistics.median(times)
    rate = blocks * threads * iters * 8 / (ms / 1e3)
    mhz = clocks.get("sm_mhz") or 2070.0
    peaks, src = measured_peaks()
    need = 0.7 * peaks["hbm_gbs"] * 1e9 / 2.0
    print(json.dumps({"probe": "ex2.approx throughput", "exp2_per_s": rate,
                      "per_sm_per_clock": rate / sms / (mhz * 1e6), "sms": sms, "ms_per_launch": ms,
                      "exps_per_launch": blocks * threads * iters * 8,
                      "row_pass_need_at_70pct_copy_peak_2byte_logits": need, "need_over_probe": need / rate,
                      "peak_source": src, "clocks": clocks}), flush=True)
    return 0


def hold_gpu(stream, steps, us_per_step=80.0):
    """Queues a spin kernel on `stream` long enough for the host to queue the
    `steps` timed steps behind it, so that no timed step waits for the host
    (Python needs tens of microseconds to queue one step)."""
    import torch
    if hasattr(torch.cuda, "_sleep"):
        ms = min(60.0, 1.0 + steps * us_per_step / 1e3)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(int(ms * 2.0e6))   # cycles, about 1 ms per 2e6 at 2 GHz


def stream_probe(L, buf, mode, ctas, warps, stages, stream, steps=20, flush=None):
    """Mean GB/s of dart_probe_stream over `steps` launches (L2 flushed before each)."""
    import ctypes as C
    import torch
    dev = buf.device
    out = torch.empty(ctas * warps * 32, dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    nbytes = buf.numel() * buf.element_size()

    def go():
        rc = L.dart_probe_stream(C.c_void_p(buf.data_ptr()), nbytes, mode, ctas, warps, stages,
                                 C.c_void_p(out.data_ptr()), C.c_void_p(err.data_ptr()),
                                 C.c_void_p(stream.cuda_stream))
        assert rc == 0, rc

    for _ in range(3):
        go()
    times = []
    hold_gpu(stream, steps)
    for _ in range(steps):
        if flush is not None:
            flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        go()
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize(dev)
    ms = statistics.mean(a.elapsed_time(b) for a, b in times)
    assert int(err.item()) == 0, "stream probe: a bulk wait ran out"
    return nbytes / (ms / 1e3) / 1e9, ms


def run_probe_stream(args):
    """Sweeps the streaming-read probe over loader kinds and launch shapes on a
    buffer the size of the chosen config's logits (config 2: 155.6 MB)."""
    import torch
    import draft_tree_construction_gb300 as D
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    D.build()
    L = D.lib()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    c = synth.CONFIGS[args.config]
    nbytes = c["B"] * c["d"] * c["V"] * synth.ELEM_BYTES[c["dtype"]]
    buf = (torch.randn(nbytes // 2, device=dev) * 3).to(torch.bfloat16)
    flush_buf = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    peaks, src = measured_peaks()
    shapes = []
    # the row pass's shape in one, two and three waves of CTAs
    for waves in (1, 2, 3):
        shapes.append((1, waves, 12, 3))
    for math_ in (0, 2):
        for warps in (8, 12, 16):
            shapes.append((math_, 1, warps, 0))
        shapes.append((math_, 2, 8, 0))
        for warps, stages in ((8, 4), (8, 6), (12, 3), (12, 4), (16, 3), (6, 8)):
            shapes.append((math_ | 1, 1, warps, stages))
        # the CTA's warps interleaved over one span
        for warps, stages in ((8, 4), (12, 3), (16, 3)):
            shapes.append((math_ | 5, 1, warps, stages))
    clk = clocks_start(0)
    t0 = time.time()
    rows = []
    for mode, per_sm, warps, stages in shapes:
        gbs, ms = stream_probe(L, buf, mode, sms * per_sm, warps, stages, stream, steps=args.steps,
                               flush=lambda: flush_buf.sum())
        rows.append({"loader": ("bulk ring, warps interleaved" if mode & 4 else "bulk ring") if mode & 1 else "direct",
                     "math": bool(mode & 2),
                     "ctas_per_sm": per_sm, "warps_per_cta": warps, "stages": stages,
                     "gbs": gbs, "us": ms * 1e3, "frac_of_peak": gbs / peaks["hbm_gbs"]})
    clocks = clocks_stop(clk, (t0, time.time()))
    # torch's own read of the same buffer, for comparison
    times = []
    for _ in range(args.steps):
        flush_buf.sum()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        buf.sum()
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize(dev)
    tms = statistics.mean(a.elapsed_time(b) for a, b in times)
    for r in rows:
        print(json.dumps({"probe": "stream", "bytes": nbytes, **r}), flush=True)
    print(json.dumps({"probe": "stream torch.sum", "bytes": nbytes, "gbs": nbytes / (tms / 1e3) / 1e9,
                      "peak": peaks["hbm_gbs"], "peak_source": src, "clocks": clocks}), flush=True)
    return 0


# ------------------------------------------------------------------ arms

def run_reference(args):
    rank, world, local = dist_setup()
    if rank != 0:
        return 0
    import oracle
    case = synth.make_config(args.config, seed=args.seed)
    ngram = oracle.NGram(case.n, case.ng_keys, case.ng_vals) if case.n >= 2 else None
    per_step = min(10.0, 150.0 / max(1, args.steps + args.warmup))
    S, _, threads, _ = oracle_sample(case, per_step, ngram)
    sub = _sub_case(case, S)
    for _ in range(args.warmup):
        oracle.tree_build(sub, ngram=ngram, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.tree_build(sub, ngram=ngram, threads=threads)
    dt = time.perf_counter() - t0
    value = S * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "trees/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_name(args.config), "sample_trees_per_step": S},
        "cpu_baseline": {"value": value, "unit": "trees/s", "cores": threads, "kind": "oracle",
                         "sample": f"first {S} of {case.B} trees per step, full vocabulary and table"},
        "e2e": {"value": value, "unit": "trees/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def measure(L, D, torch, case, dev, stream, steps, warmup, world, with_select=False):
    """One config: whole steps (row pass + row merge + tree kernel), the row
    pass alone (the dominant kernel, for the roofline), the row merge alone;
    CUDA events on `stream`, L2 flushed before every timed launch."""
    import ctypes as C
    B, d, V, k = case.B, case.d, case.V, case.k
    if case.dtype == "bf16":
        host = torch.from_numpy(case.logits.view(np.int16).copy()).view(torch.bfloat16)
    else:
        host = torch.from_numpy(case.logits.copy())
    z = host.to(dev)
    tab = D.NGramTable(case.n, case.ng_keys, case.ng_vals, device=dev) if case.n >= 2 else None
    ctx = torch.from_numpy(np.ascontiguousarray(case.ctx)).to(dev) if tab is not None else None
    builder = D.TreeBuilder(B, d, V, z.dtype, case.T, k, case.W, case.lam, case.beta,
                            table=tab, ctx=ctx, device=dev)
    # L2 flush between timed launches: a read-only sweep of 256 MB (twice the
    # L2) evicts the logits, the n-gram table and the workspace without
    # leaving dirty lines to be written back inside the next timed window
    flush_buf = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.sum()

    def timed(fn, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        hold_gpu(stream, n)
        for i in range(n):
            flush()
            evs[i][0].record(stream)
            fn(i)
            evs[i][1].record(stream)
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b) for a, b in evs]

    for _ in range(max(3, warmup)):
        flush()
        builder(z)
    torch.cuda.synchronize(dev)
    assert D.device_error(builder.ws) == 0, "device error during warm-up"
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    step_times = timed(lambda i: builder(z), steps)
    t1 = time.time()
    barrier(world)
    # the same steps with a direct dart_tree_build call each (three launches
    # from the host instead of one graph replay): the reference for the
    # per-kernel breakdown below, whose parts are direct launches too
    builder.graph = False
    direct_times = timed(lambda i: builder(z), steps)
    builder.graph = True
    code = D.DTYPE_CODES()[z.dtype]
    ws = builder.ws
    sp = C.c_void_p(stream.cuda_stream)

    def row_pass(i):
        assert L.dart_row_pass(C.c_void_p(z.data_ptr()), B * d, V, V, code, float(case.T), k,
                               C.c_void_p(ws.data_ptr()), ws.numel(), sp) == 0

    def row_finish(i):
        assert L.dart_row_finish(B * d, V, V, code, float(case.T), k, None, None, None,
                                 C.c_void_p(ws.data_ptr()), ws.numel(), sp) == 0

    pass_times = timed(row_pass, steps)
    merge_times = timed(row_finish, steps)
    assert D.device_error(builder.ws) == 0, "device error during the timed steps"
    res = {
        "step_ms": max_over_ranks(statistics.mean(step_times), world),
        "row_pass_ms": max_over_ranks(statistics.mean(pass_times), world),
        "row_merge_ms": max_over_ranks(statistics.mean(merge_times), world),
        "direct_step_ms": max_over_ranks(statistics.mean(direct_times), world),
        "step_p10_p50_p90": [float(np.percentile(step_times, q)) for q in (10, 50, 90)],
        "row_pass_p10_p50_p90": [float(np.percentile(pass_times, q)) for q in (10, 50, 90)],
        "window": (t0, t1), "host": host, "z": z, "builder": builder,
    }
    res["tree_ms_by_difference"] = res["direct_step_ms"] - res["row_pass_ms"] - res["row_merge_ms"]
    if with_select and builder.out.get("scores") is not None:
        # the verification tree chosen best-first from the step's candidate
        # trees, budget 16 (one of the verification budgets PCTree quotes)
        o = builder.out
        budget = min(16, o["parents"].shape[1])
        sel_err = torch.zeros(1, dtype=torch.int32, device=dev)

        def select_only(i):
            D.tree_select(o["tokens"], o["parents"], o["pos"], o["scores"], budget, device_err=sel_err,
                          stream=stream)

        sel_times = timed(select_only, min(steps, 200))
        sel_ms = max_over_ranks(statistics.mean(sel_times), world)
        torch.cuda.synchronize(dev)
        res["select"] = {"budget": budget, "us_per_call": sel_ms * 1e3, "trees_per_s": B * world / (sel_ms / 1e3),
                         "kernel": "select_kernel (best-first verification tree)", "calls": len(sel_times),
                         "device_error": int(sel_err.item())}
        # the same verification tree chosen inside the tree kernel
        # (dart_tree_build_verify): the whole step with it, against without
        Mp = budget
        vout = [torch.empty((B, Mp), dtype=torch.int32, device=dev) for _ in range(4)]
        vmask = torch.empty((B, Mp, (Mp + 31) // 32), dtype=torch.int32, device=dev)
        vsc = torch.empty((B, Mp), dtype=torch.float32, device=dev)
        tab = builder.table
        P = lambda t: C.c_void_p(t.data_ptr())

        def build_verify(i):
            assert L.dart_tree_build_verify(
                P(z), B, d, V, V, code, float(case.T), k, case.W, float(case.lam), float(case.beta),
                C.byref(tab.desc) if tab is not None else None, P(builder.ctx) if tab is not None else None,
                P(o["tokens"]), P(o["parents"]), P(o["pos"]), P(o["mask"]), P(o["scores"]), Mp,
                P(vout[0]), P(vout[1]), P(vout[2]), P(vout[3]), P(vmask), P(vsc), P(ws), ws.numel(), sp) == 0

        ver_times = timed(build_verify, min(steps, 200))
        ver_ms = max_over_ranks(statistics.mean(ver_times), world)
        assert D.device_error(builder.ws) == 0, "device error in the verify steps"
        res["select"]["fused_in_tree_kernel"] = {
            "entry": "dart_tree_build_verify", "step_ms": ver_ms,
            "extra_us_over_direct_step": (ver_ms - res["direct_step_ms"]) * 1e3, "calls": len(ver_times)}
    return res


def numa_placement(index: int) -> dict:
    """NUMA node of the GPU (from its PCI device in sysfs) and the nodes of the
    CPUs this process may run on (the pinned host buffers are first touched
    there), so the host link's rate can be read against their placement."""
    out = {"gpu_numa_node": None, "process_cpu_numa_nodes": None, "gpu_pci_bus_id": None}
    try:
        bus = subprocess.run(["nvidia-smi", "-i", str(index), "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout.strip()
        out["gpu_pci_bus_id"] = bus or None
        if bus:
            path = f"/sys/bus/pci/devices/{bus[-12:].lower()}/numa_node"
            out["gpu_numa_node"] = int(open(path).read().strip())
    except (OSError, ValueError, subprocess.SubprocessError):
        pass
    try:
        cpus = os.sched_getaffinity(0)
        nodes = []
        base = "/sys/devices/system/node"
        for name in sorted(os.listdir(base)):
            if not name.startswith("node") or not name[4:].isdigit():
                continue
            ids = set()
            for part in open(os.path.join(base, name, "cpulist")).read().strip().split(","):
                if "-" in part:
                    a, b = part.split("-")
                    ids.update(range(int(a), int(b) + 1))
                elif part:
                    ids.add(int(part))
            if ids & cpus:
                nodes.append(int(name[4:]))
        out["process_cpu_numa_nodes"] = nodes
    except (OSError, ValueError):
        pass
    return out


def stream_ceiling(L, torch, nbytes, dev, stream, steps):
    """The bulk-copy ring of the row pass (twelve warps x three 4 KiB stages
    per SM) with no arithmetic, on a buffer of the logits' size: the
    bandwidth any row pass of this shape can reach at this size."""
    buf = torch.empty(nbytes // 2, dtype=torch.bfloat16, device=dev).normal_()
    flush_buf = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    gbs, ms = stream_probe(L, buf, 1, sms, 12, 3, stream, steps=steps, flush=lambda: flush_buf.sum())
    del buf
    return {"gbs": gbs, "us": ms * 1e3, "shape": "12 warps x 3 bulk-copy stages of 4 KiB per SM, no arithmetic"}


def run_ours(args):
    import torch
    import draft_tree_construction_gb300 as D

    rank, world, local = dist_setup()
    dist_init(world, local)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    D.build()
    L = D.lib()
    stream = torch.cuda.current_stream(dev)
    peaks, peaks_src = measured_peaks()

    case = synth.make_config(args.config, seed=args.seed + rank)
    B, d, V, k = case.B, case.d, case.V, case.k
    logit_bytes = case.logit_bytes
    clk = clocks_start(dev.index or 0)
    m = measure(L, D, torch, case, dev, stream, args.steps, args.warmup, world, with_select=True)
    clocks = clocks_stop(clk, m["window"])
    step_ms, k1_ms = m["step_ms"], m["row_pass_ms"]
    builder, z, host = m["builder"], m["z"], m["host"]

    # ---- end to end: pinned host logits in, pinned host outputs back, every step
    e2e = None
    if not args.no_e2e:
        pinned = host.pin_memory()
        outs = {key: torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                for key, v in builder.out.items() if v is not None}
        d2h = sum(v.numel() * v.element_size() for v in outs.values())
        h2d = pinned.numel() * pinned.element_size()

        def e2e_step():
            z.copy_(pinned, non_blocking=True)
            builder(z)
            for key, v in outs.items():
                v.copy_(builder.out[key], non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        barrier(world)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        hold_gpu(stream, args.steps, us_per_step=900.0)
        for a, b in evs:
            a.record(stream)
            e2e_step()
            b.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in evs), world)
        e2e = {"value": B * world / (e2e_ms / 1e3), "unit": "trees/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, **numa_placement(dev.index or 0)}

    achieved = logit_bytes / (k1_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": k1_traffic(args.config),
                "kernel": "row_stream_kernel (log-softmax + top-k stream, dart_row_pass)",
                "peak_source": f"{peaks_src} hbm_gbs",
                "k1_ms": k1_ms, "frac_of_8tbs_nominal": achieved / 8000.0}

    ceiling = None
    per_config = None
    cpu = None
    if rank == 0 and world == 1:
        ceiling = stream_ceiling(L, torch, logit_bytes, dev, stream, min(args.steps, 50))
        ceiling["frac"] = ceiling["gbs"] / peaks["hbm_gbs"]
        ceiling["row_pass_over_ceiling"] = achieved / ceiling["gbs"]
        if not args.no_per_config:
            per_config = {}
            for c2 in (1, 3, 4):
                if c2 == args.config:
                    continue
                cc = synth.make_config(c2, seed=args.seed)
                mm = measure(L, D, torch, cc, dev, stream, max(20, min(args.steps, 200)), args.warmup, world)
                ach = cc.logit_bytes / (mm["row_pass_ms"] / 1e3) / 1e9
                per_config[str(c2)] = {
                    "workload": workload_name(c2), "ms_per_step": mm["step_ms"],
                    "direct_launches_ms_per_step": mm["direct_step_ms"],
                    "trees_per_s": cc.B / (mm["step_ms"] / 1e3), "row_pass_ms": mm["row_pass_ms"],
                    "row_pass_frac": ach / peaks["hbm_gbs"], "row_pass_traffic": k1_traffic(c2),
                    "row_merge_ms": mm["row_merge_ms"],
                    "tree_ms_by_difference": mm["tree_ms_by_difference"],
                    "logit_bytes": cc.logit_bytes}
                del mm
        if not args.no_cpu_baseline:
            S, dt, threads, ng = oracle_sample(case, args.cpu_seconds)
            S1, dt1 = oracle_single_core(case, args.cpu_seconds / 3.0, ng)
            cpu = {"value": S / dt, "unit": "trees/s", "cores": threads, "kind": "oracle",
                   "sample": f"first {S} of {B} trees of the same batch, full vocabulary and table",
                   "value_1_core": S1 / dt1, "sample_1_core": f"first {S1} of {B} trees, one thread"}

    if rank == 0:
        value = B * world / (step_ms / 1e3)
        line = {
            "metric": METRIC, "value": value, "unit": "trees/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32/f64",
            "data": "synthetic",
            "config": {"workload": workload_name(args.config), "logit_dtype": case.dtype,
                       "trees_per_gpu": B, "logit_bytes_per_step": logit_bytes,
                       "l2": "flushed before every timed launch (read-only sweep of 256 MB)",
                       "step_ms_p10_p50_p90": m["step_p10_p50_p90"],
                       "row_pass_ms_p10_p50_p90": m["row_pass_p10_p50_p90"],
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "hbm_gbs_whole_step": logit_bytes / (step_ms / 1e3) / 1e9,
            "roofline": roofline,
            "stream_ceiling": ceiling,
            "step_breakdown_ms": {"launch": "one CUDA-graph replay of the three kernels a step (dart_tree_plan_launch)",
                                  "direct_launches_step": m["direct_step_ms"],
                                  "row_pass": k1_ms, "row_merge": m["row_merge_ms"],
                                  "tree_by_difference": m["tree_ms_by_difference"]},
            "per_config": per_config,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": 3 * args.steps,
            "verification_tree_select": m.get("select"),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.probe_sfu:
        return run_probe_sfu(args)
    if args.probe_stream:
        return run_probe_stream(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
