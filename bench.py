"""Benchmark of exact attention on one GB300: forward + backward at B=1, H=16, N=8192, d=128 (bf16).

One step = one forward (fa_fwd) and one backward (fa_bwd) over the same seeded synthetic batch, the
whole hot path.  Prints one JSON line (see ``main``).  ``--impl reference`` times the fp64 CPU oracle
on the host cores instead (a bounded sample of the same workload per step).
"""
from __future__ import annotations

import os

# The oracle's BLAS uses every host core; set before numpy is imported anywhere.
_NCPU = os.cpu_count() or 1
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS"):
    os.environ.setdefault(_v, str(_NCPU))

import argparse
import json
import math
import statistics
import subprocess
import sys
import threading
import time

import torch

import fa_inputs

ROOT = os.path.dirname(os.path.abspath(__file__))
L2_FLUSH_BYTES = 256 << 20


def _dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of `x` over all ranks (timings are reported for the slowest rank)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": p["bf16_tflops"], "bf16_tflops_sustained": p.get("bf16_tflops_sustained"),
                "hbm_gbs": p["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi every INTERVAL_MS while the timed region runs;
    only samples whose own timestamp falls inside the region (mark_start .. mark_end) are reported."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 20

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None
        self.t0 = self.t1 = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.INTERVAL_MS)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        return summarize_clock_lines(self.lines, self.t0, self.t1, self.INTERVAL_MS)


def _smi_time(stamp: str):
    """Seconds since the epoch of an nvidia-smi timestamp ('YYYY/MM/DD HH:MM:SS.mmm', local time)."""
    try:
        main, _, frac = stamp.strip().partition(".")
        return time.mktime(time.strptime(main, "%Y/%m/%d %H:%M:%S")) + (float("0." + frac) if frac else 0.0)
    except (ValueError, OverflowError):
        return None


def summarize_clock_lines(lines, t0, t1, interval_ms):
    """Median SM clock, maximum clock and active throttle reasons of the samples taken between t0 and t1
    (plus half a sampling interval either side); all samples if none carries a usable timestamp."""
    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            rows.append((_smi_time(parts[0]), float(parts[2]), float(parts[3]), parts[6:10]))
        except ValueError:
            continue
    slack = interval_ms / 2000.0
    timed = t0 is not None and t1 is not None and any(r[0] is not None for r in rows)
    inside = [r for r in rows if r[0] is not None and t0 - slack <= r[0] <= t1 + slack] if timed else rows
    sm = [r[1] for r in inside]
    reasons = {n for r in inside for n, v in zip(names, r[3]) if v.lower() == "active"}
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(r[2] for r in inside) if inside else None,
            "reasons": sorted(reasons), "samples": len(sm), "interval_ms": interval_ms,
            "window": "timed region" if timed else "whole run (no timestamps)"}


def _oracle_sample(w, heads: int, inp):
    """fp64 oracle forward + backward of the first `heads` heads of batch 0, full N x N each."""
    import oracle
    q, k, v, do = (inp[n][:1, :heads].double().numpy() for n in ("q", "k", "v", "do"))
    t0 = time.perf_counter()
    oracle.forward(q, k, v, w.scale)
    oracle.backward(q, k, v, do, w.scale)
    dt = time.perf_counter() - t0
    flops = 14.0 * heads * w.N * w.N * w.d
    return flops, dt


def _cpu_meta(heads, w):
    return {"kind": "oracle", "cores": _NCPU,
            "sample": f"fp64 oracle (numpy, {_NCPU} BLAS threads) forward+backward of {heads} of the {w.B * w.H} "
                      f"heads (N={w.N}, d={w.d}), all rows; flops counted as 14*heads*N^2*d"}


def run_reference(args, w):
    rank, world, _ = _dist_env()
    if rank != 0:
        return 0
    inp = fa_inputs.workload_inputs(w, with_grad=True)
    heads = args.oracle_heads_per_step
    for _ in range(args.warmup):
        _oracle_sample(w, heads, inp)
    total_f, total_t = 0.0, 0.0
    for _ in range(args.steps):
        f, t = _oracle_sample(w, heads, inp)
        total_f += f
        total_t += t
    tflops = total_f / total_t / 1e12
    meta = _cpu_meta(heads, w)
    meta["value"] = tflops
    meta["unit"] = "TFLOP/s"
    line = {"impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(w, world), "cpu_baseline": meta,
            "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


METRIC = "attention TFLOP/s fwd and fwd+bwd vs BF16 tensor peak (N=8192, d=128, 1xGB300)"


def _config(w, world, strong=False):
    if world == 1:
        par = "single-gpu"
    elif strong:
        par = f"heads{world}: the workload's B*H heads split into contiguous ranges, one per rank, no collective"
    else:
        par = f"batches{world}: each rank its own batch of the workload's shape (seed + rank), no collective"
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "dtype": w.dtype,
            "step": "fa_fwd + fa_bwd", "parallelism": par,
            "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write, untimed)"}


def run_ours(args, w):
    import exact_io_aware_17_gb300 as fa

    rank, world, local = _dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fa.load_library()

    strong = args.strong and world > 1
    if strong:
        # Strong scaling: the one workload, its heads split across the ranks (each rank holds only its own).
        from exact_io_aware_17_gb300 import shard
        full = fa_inputs.workload_inputs(w, with_grad=True)
        inp_cpu = {n: shard.local_heads(t, rank, world).contiguous() for n, t in full.items()}
        heads_here = inp_cpu["q"].shape[1]
        if heads_here == 0:
            raise SystemExit(f"--strong: rank {rank} of {world} would get no head of {w.name}")
    else:
        # One GPU, or weak scaling: every rank runs the whole workload's shape on its own batch.
        inp_cpu = fa_inputs.make_inputs(w.B, w.H, w.N, w.d, w.dtype, w.seed + rank, w.q_gain, with_grad=True)
    q, k, v, do = (inp_cpu[n].to(dev) for n in ("q", "k", "v", "do"))
    B, H, N, d = (int(x) for x in q.shape)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        fa.fa_fwd(q, k, v, w.scale, o, lse, stream=stream)
        fa.fa_bwd(q, k, v, o, do, lse, w.scale, dq, dk, dv, ws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    fa.fa_check_status(stream)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    # The backward's main kernel alone, between events the library records around it (fa_debug_time_bwd_main);
    # each event is recorded once first so that it exists.
    evm = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for pair in evm:
        for e in pair:
            e.record(stream)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = fa.fa_kernel_launches()
    clocks.mark_start()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xff)                      # evict the previous step's data from L2 (untimed)
        ev[i][0].record(stream)
        fa.fa_fwd(q, k, v, w.scale, o, lse, stream=stream)
        ev[i][1].record(stream)
        fa.fa_debug_time_bwd_main(evm[i][0], evm[i][1])
        fa.fa_bwd(q, k, v, o, do, lse, w.scale, dq, dk, dv, ws, stream=stream)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - t_wall
    clocks.mark_end()
    launches = fa.fa_kernel_launches() - launches0          # counted by the library at each launch
    clk = clocks.stop()
    fa.fa_check_status(stream)

    fwd_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    bwd_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    main_ms = [evm[i][0].elapsed_time(evm[i][1]) for i in range(args.steps)]
    step_ms = sum(fwd_ms) / args.steps + sum(bwd_ms) / args.steps
    step_ms = max_over_ranks(step_ms, dev)
    # Work of this rank's heads, and of the whole job (all ranks) per step.
    lw = fa_inputs.Workload(w.name, w.dtype, B, H, N, d, w.seed)
    total_flops = (w.fwd_flops() + w.bwd_flops()) * (1 if strong else world)
    value = total_flops / (step_ms * 1e-3) / 1e12
    fwd_avg = sum(fwd_ms) / args.steps
    bwd_avg = sum(bwd_ms) / args.steps
    fwd_tflops = lw.fwd_flops() / (fwd_avg * 1e-3) / 1e12
    bwd_tflops = lw.bwd_flops() / (bwd_avg * 1e-3) / 1e12
    peaks = _peaks()
    peak = peaks["bf16_tflops"]

    e2e_ms, h2d, d2h = _e2e(fa, lw, inp_cpu, dev, args.steps)
    e2e_ms = max_over_ranks(e2e_ms, dev)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "strong" if strong else "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded iid N(0,1), bf16)",
        "config": _config(w, world, strong),
        "fwd": {"ms": fwd_avg, "tflops": fwd_tflops, "frac_of_peak": fwd_tflops / peak},
        "bwd": {"ms": bwd_avg, "tflops": bwd_tflops, "frac_of_peak": bwd_tflops / peak},
        "fwd_bwd_frac_of_peak": value / world / peak,
        "wall_s_timed_region": wall,
        "clocks": clk,
        "gpu_launches": launches,
        "gpu_launches_counted_by": "libfa.so's own launch counter (fa_kernel_launches) across the timed loop",
        "e2e": {"value": total_flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "pinned host q,k,v,dO copied in and o,lse,dq,dk,dv copied out every step, through the "
                       "public API; one copy stream per tensor, double-buffered so that step i's transfers "
                       "overlap steps i-1 and i+1's compute"},
    }
    line["bwd"]["main_kernel_ms"] = sum(main_ms) / args.steps
    line["roofline"] = _roofline(lw, fwd_avg, bwd_avg, sum(main_ms) / args.steps, peaks, whole_workload=not strong)
    line["exp_pipe"] = _exp_pipe(lw, fwd_avg, bwd_avg)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        f, t = _oracle_sample(w, args.oracle_heads, inp_cpu)
        meta = _cpu_meta(args.oracle_heads, w)
        meta.update({"value": f / t / 1e12, "unit": "TFLOP/s", "seconds": t})
        line["cpu_baseline"] = meta
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def _e2e(fa, w, inp_cpu, dev, steps):
    """Per-step time of fa_fwd + fa_bwd fed from and drained to pinned host memory, double-buffered: step i's
    inputs are copied in while step i-1 computes, and its outputs copied out while step i+1 computes (o and
    lse already while step i's backward runs; step i's backward waits for dO, its forward does not).  Every
    tensor has a copy stream of its own, so that the copies of a step use several copy engines at once."""
    B, H, N, d = w.B, w.H, w.N, w.d
    ins, outs = ("q", "k", "v", "do"), ("o", "lse", "dq", "dk", "dv")
    host_in = {n: inp_cpu[n].pin_memory() for n in ins}
    host_out = [{n: torch.empty(B, H, N, d, dtype=inp_cpu["q"].dtype).pin_memory() for n in ("o", "dq", "dk", "dv")}
                for _ in range(2)]
    for h in host_out:
        h["lse"] = torch.empty(B, H, N, dtype=torch.float32).pin_memory()
    bufs = []
    for _ in range(2):
        b = {n: torch.empty(B, H, N, d, dtype=inp_cpu["q"].dtype, device=dev) for n in ins + ("o", "dq", "dk", "dv")}
        b["lse"] = torch.empty(B, H, N, dtype=torch.float32, device=dev)
        b["ws"] = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
        bufs.append(b)
    comp = torch.cuda.current_stream(dev)
    s_in = {n: torch.cuda.Stream(dev) for n in ins}
    s_out = {n: torch.cuda.Stream(dev) for n in outs}
    computed = [torch.cuda.Event() for _ in range(2)]          # buffer j's inputs read, outputs written
    fwd_done = [torch.cuda.Event() for _ in range(2)]          # buffer j's o and lse written
    loaded = [{n: torch.cuda.Event() for n in ins} for _ in range(2)]
    drained = [{n: torch.cuda.Event() for n in outs} for _ in range(2)]
    for j in range(2):
        computed[j].record(comp)
        for e in drained[j].values():
            e.record(comp)

    def drain(j, names, after):
        for name in names:
            st = s_out[name]
            st.wait_event(after)
            with torch.cuda.stream(st):
                host_out[j][name].copy_(bufs[j][name], non_blocking=True)
                drained[j][name].record(st)

    def run(n):
        for i in range(n):
            j = i % 2
            b = bufs[j]
            for name in ins:                               # buffer j's inputs are free once step i-2 computed
                st = s_in[name]
                st.wait_event(computed[j])
                with torch.cuda.stream(st):
                    b[name].copy_(host_in[name], non_blocking=True)
                    loaded[j][name].record(st)
            for name in ("q", "k", "v"):
                comp.wait_event(loaded[j][name])
            for name in outs:                              # ... and its outputs once step i-2's were copied out
                comp.wait_event(drained[j][name])
            fa.fa_fwd(b["q"], b["k"], b["v"], w.scale, b["o"], b["lse"], stream=comp)
            fwd_done[j].record(comp)
            drain(j, ("o", "lse"), fwd_done[j])            # final after the forward: out while the backward runs
            comp.wait_event(loaded[j]["do"])               # dO is needed only from here on
            fa.fa_bwd(b["q"], b["k"], b["v"], b["o"], b["do"], b["lse"], w.scale, b["dq"], b["dk"], b["dv"], b["ws"],
                      stream=comp)
            computed[j].record(comp)
            drain(j, ("dq", "dk", "dv"), computed[j])

    run(4)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(comp)
    for st in list(s_in.values()) + list(s_out.values()):
        st.wait_stream(comp)
    run(steps)
    for st in s_out.values():
        comp.wait_stream(st)
    end.record(comp)
    torch.cuda.synchronize(dev)
    elt = inp_cpu["q"].element_size() * inp_cpu["q"].numel()
    return start.elapsed_time(end) / steps, 4 * elt, 4 * elt + B * H * N * 4


# DRAM bytes per launch of the dominant kernel at the bench workload, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), with the profile summary that records it and the
# SHA-256 of the kernel's source files when it was taken.  If the sources differ now, the figure is
# stale: the JSON line then reports traffic null and says so.
TRAFFIC = {
    ("backward", "bf16-fwdbwd-B1-H16-N8192-d128"): {
        "bytes": 202727168 + 83696896,
        "profile": "profiles/dram_per_launch_bench_B1-H16-N8192-d128.md",
        "kernel": "bwd_tc_kernel<128>",
        "sources": ("exact_io_aware_17_gb300/csrc/fa_bwd_tc.cu", "exact_io_aware_17_gb300/csrc/fa_ptx.cuh"),
        "sha256": "7fc13617fa9cb275a4b7a52b17bff2358760e1c09fbe4b6634bd6124d7860954",
    },
}


def _sources_digest(paths):
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _traffic(name, w):
    t = TRAFFIC.get((name, w.name))
    if t is None:
        return None, "no capture for this kernel and workload"
    if t["sha256"] != _sources_digest(t["sources"]):
        return None, f"stale: {t['kernel']} sources changed since the capture in {t['profile']}"
    return t["bytes"], f"ncu capture of {t['kernel']}, {t['profile']}"


# Measured throughput of the exponential unit (ex2.approx.f32, whole GPU), the second ceiling of the
# softmax work: a recorded result of a standalone microbenchmark on this GPU model
# (profiles/mufu_ex2_peak.md).
EX2_PER_S = 9.97e12


def _exp_pipe(w, fwd_ms, bwd_ms):
    """Exponentials per second of each pass against the measured ex2 throughput: B*H*N^2 exponentials in
    the forward (P) and the same again in the backward (P recomputed)."""
    n = w.B * w.H * w.N * w.N
    fwd, bwd = n / (fwd_ms * 1e-3), n / (bwd_ms * 1e-3)
    return {"unit": "ex2/s", "fwd": fwd, "bwd": bwd, "peak": EX2_PER_S, "frac_fwd": fwd / EX2_PER_S,
            "frac_bwd": bwd / EX2_PER_S, "peak_source": "measured (ex2.approx throughput microbenchmark)"}


def _roofline(w, fwd_ms, bwd_ms, main_ms, peaks, whole_workload=True):
    """Roofline of the dominant kernel: the backward's main kernel (bwd_tc_kernel), whose time the library
    records between events around its launch, unless the forward takes longer.  Achieved = the kernel's
    algorithmic flops (10*B*H*N^2*d: the five N x N x d products) / its average event-timed duration."""
    if bwd_ms >= fwd_ms:
        name, flops, ms = "backward", w.bwd_flops(), main_ms
        kernel = "bwd_tc_kernel (the backward's main kernel, timed alone between library-recorded events)"
    else:
        name, flops, ms = "forward", w.fwd_flops(), fwd_ms
        kernel = "fwd_tc_kernel (the forward's launches)"
    achieved = flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    traffic, source = _traffic(name, w) if whole_workload else (None, "no capture for a rank's share of the heads")
    return {"kernel": kernel, "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "ms_per_launch": ms, "peak_source": f"{peaks['source']} burst bf16 (cuBLAS)",
            "traffic": traffic, "traffic_unit": "DRAM bytes per launch of the main kernel", "traffic_source": source}


def _time_call(fn, flush, iters):
    """Median CUDA-event time (ms) of fn() over `iters` calls, L2 flushed before each, after 3 warm-ups."""
    for _ in range(3):
        fn()
    ts = []
    for i in range(iters):
        flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def run_sweep(args):
    """Throughput over shapes, one JSON line per shape (not the bench contract line).

    Grid mode: B=1, d in --d, N in --N, H = --rows // N (so every shape has the same B*H*N rows), seeded
    N(0,1) bf16 inputs.  Workload mode (--workloads): the named workloads' own shapes and inputs; --bwd times
    the backward of forward-only workloads too (their upstream gradient dO is drawn after Q, K, V by the
    same seeded generator, so Q, K, V are the workload's own).  Median of --iters CUDA-event timings per call,
    L2 flushed between calls; fractions of the measured bf16 burst peak."""
    import exact_io_aware_17_gb300 as fa
    peaks = _peaks()
    peak = peaks["bf16_tflops"]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    if args.workloads:
        shapes = [(fa_inputs.WORKLOADS[n], fa_inputs.WORKLOADS[n].backward or args.bwd) for n in args.workloads]
    else:
        shapes = []
        for d in args.d:
            for N in args.N:
                H = max(1, args.rows // N)
                shapes.append((fa_inputs.Workload(f"B1-H{H}-N{N}-d{d}", "bf16", 1, H, N, d, seed=N + d), True))
    for w, with_bwd in shapes:
        if w.dtype != "bf16":
            continue
        inp = fa_inputs.workload_inputs(w, with_grad=with_bwd)
        t = {n: x.cuda() for n, x in inp.items()}
        o, lse = fa.fa_fwd(t["q"], t["k"], t["v"], w.scale)
        tf = _time_call(lambda: fa.fa_fwd(t["q"], t["k"], t["v"], w.scale, o, lse), flush, args.iters)
        line = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "fwd_ms": tf,
                "fwd_tflops": w.fwd_flops() / tf / 1e9, "fwd_frac": w.fwd_flops() / tf / 1e9 / peak}
        if with_bwd:
            dq, dk, dv = (torch.empty_like(t["q"]) for _ in range(3))
            ws = torch.empty(fa.fa_bwd_workspace_size(w.B, w.H, w.N, w.d), dtype=torch.uint8, device="cuda")
            tb = _time_call(lambda: fa.fa_bwd(t["q"], t["k"], t["v"], o, t["do"], lse, w.scale, dq, dk, dv, ws),
                            flush, args.iters)
            line.update(bwd_ms=tb, bwd_tflops=w.bwd_flops() / tb / 1e9, bwd_frac=w.bwd_flops() / tb / 1e9 / peak,
                        fwdbwd_tflops=(w.fwd_flops() + w.bwd_flops()) / (tf + tb) / 1e9,
                        fwdbwd_frac=(w.fwd_flops() + w.bwd_flops()) / (tf + tb) / 1e9 / peak)
        if args.stepnorm:
            tsn = _time_call(lambda: fa.fa_fwd_stepnorm(t["q"], t["k"], t["v"], w.scale, o, lse), flush, args.iters)
            line.update(stepnorm_fwd_ms=tsn, stepnorm_fwd_tflops=w.fwd_flops() / tsn / 1e9, stepnorm_slowdown=tsn / tf)
        if args.f32:
            # The fp32 CUDA-core forward on the same values (the bf16 inputs widened to fp32).
            q32, k32, v32 = (t[n].float() for n in ("q", "k", "v"))
            o32, l32 = fa.fa_fwd_f32(q32, k32, v32, w.scale)
            t32 = _time_call(lambda: fa.fa_fwd_f32(q32, k32, v32, w.scale, o32, l32), flush, args.iters)
            line.update(f32_fwd_ms=t32, f32_fwd_tflops=w.fwd_flops() / t32 / 1e9)
            del q32, k32, v32, o32, l32
        fa.fa_check_status()
        line.update(peak_tflops=peak, peak_source=peaks["source"])
        print(json.dumps(line), flush=True)
        del t, o, lse
        torch.cuda.empty_cache()
    return 0


def run_case(args):
    """A fixed, small command for profilers: --iters forward (and with --bwd backward) calls on one seeded
    bf16 shape B H N d, then a status check.  Prints "ok"."""
    import exact_io_aware_17_gb300 as fa
    B, H, N, d = args.case
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", seed=5, with_grad=args.bwd)
    t = {n: x.cuda() for n, x in inp.items()}
    scale = 1 / math.sqrt(d)
    for _ in range(args.iters):
        o, lse = fa.fa_fwd(t["q"], t["k"], t["v"], scale)
        if args.bwd:
            fa.fa_bwd(t["q"], t["k"], t["v"], o, t["do"], lse, scale)
    torch.cuda.synchronize()
    fa.fa_check_status()
    print("ok")
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=fa_inputs.HEADLINE, choices=sorted(fa_inputs.WORKLOADS))
    ap.add_argument("--oracle-heads", type=int, default=8,
                    help="heads of the workload the CPU baseline runs through the oracle (about 1.5 s each)")
    ap.add_argument("--oracle-heads-per-step", type=int, default=1,
                    help="heads per step of --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--strong", action="store_true",
                    help="under torchrun: split the one workload's heads across the ranks (strong scaling) "
                         "instead of giving every rank a batch of its own (weak scaling, the default)")
    g = ap.add_argument_group("other modes (their output is not the bench line)")
    g.add_argument("--sweep", action="store_true", help="throughput over a grid of shapes or named workloads")
    g.add_argument("--N", type=int, nargs="+", default=[2048, 4096, 8192, 16384, 32768], help="--sweep grid")
    g.add_argument("--d", type=int, nargs="+", default=[64, 128], help="--sweep grid")
    g.add_argument("--rows", type=int, default=131072, help="--sweep grid: B*H*N of every shape")
    g.add_argument("--workloads", nargs="+", choices=sorted(fa_inputs.WORKLOADS), help="--sweep these workloads")
    g.add_argument("--bwd", action="store_true", help="--sweep / --case: time or run the backward too")
    g.add_argument("--stepnorm", action="store_true", help="--sweep: also time fa_fwd_stepnorm")
    g.add_argument("--f32", action="store_true", help="--sweep: also time the fp32 forward fa_fwd_f32")
    g.add_argument("--iters", type=int, default=10, help="--sweep: timed calls per shape; --case: calls")
    g.add_argument("--case", type=int, nargs=4, metavar=("B", "H", "N", "d"),
                   help="run one seeded shape --iters times (a fixed command for profilers)")
    args = ap.parse_args()
    if args.sweep:
        return run_sweep(args)
    if args.case:
        return run_case(args)
    w = fa_inputs.WORKLOADS[args.workload]
    if not w.backward:
        raise SystemExit("the bench step is forward + backward: pick a workload with a backward pass")
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
