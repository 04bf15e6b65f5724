"""Throughput of fa_fwd and fa_bwd over a grid of sequence lengths and head sizes (one GPU).

    python -m exact_io_aware_17_gb300.sweep --N 2048 4096 8192 16384 32768 --d 64 128

Each shape runs B=1 with H chosen so that B*H*N = 131072 rows (the headline workload's size), seeded
N(0,1) bf16 inputs, L2 flushed between timed calls, median of --iters CUDA-event timings.  Prints one
JSON line per shape with TFLOP/s and the fraction of the measured bf16 peak.

    python -m exact_io_aware_17_gb300.sweep --workload bf16-fwd-B1-H8-N32768-d128-q4

times the forward (and the backward when the workload has one) on a named workload's own inputs.
"""
import argparse
import json
import math
import os
import statistics
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import exact_io_aware_17_gb300 as fa  # noqa: E402
import fa_inputs  # noqa: E402


def _peak():
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f)["bf16_tflops"], "measured"
    return 1900.0, "fallback"


def _time(fn, flush, iters):
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--N", type=int, nargs="+", default=[2048, 4096, 8192, 16384, 32768])
    ap.add_argument("--d", type=int, nargs="+", default=[64, 128])
    ap.add_argument("--rows", type=int, default=131072, help="B*H*N of every shape")
    ap.add_argument("--iters", type=int, default=10)
    ap.add_argument("--workload", nargs="+", default=None, choices=sorted(fa_inputs.WORKLOADS),
                    help="time named workloads (their own shapes and inputs) instead of the N x d grid")
    ap.add_argument("--stepnorm", action="store_true",
                    help="also time fa_fwd_stepnorm (the per-step normalised update rule)")
    a = ap.parse_args()
    peak, src = _peak()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    if a.workload:
        for name in a.workload:
            w = fa_inputs.WORKLOADS[name]
            if w.dtype != "bf16":
                continue
            inp = fa_inputs.workload_inputs(w, with_grad=w.backward)
            t = {n: x.cuda() for n, x in inp.items()}
            o, lse = fa.fa_fwd(t["q"], t["k"], t["v"], w.scale)
            tf = _time(lambda: fa.fa_fwd(t["q"], t["k"], t["v"], w.scale, o, lse), flush, a.iters)
            line = {"workload": name, "fwd_ms": tf, "fwd_tflops": w.fwd_flops() / tf / 1e9,
                    "fwd_frac": w.fwd_flops() / tf / 1e9 / peak, "peak_tflops": peak, "peak_source": src}
            if w.backward:
                dq, dk, dv = (torch.empty_like(t["q"]) for _ in range(3))
                ws = torch.empty(fa.fa_bwd_workspace_size(w.B, w.H, w.N, w.d), dtype=torch.uint8, device="cuda")
                tb = _time(lambda: fa.fa_bwd(t["q"], t["k"], t["v"], o, t["do"], lse, w.scale, dq, dk, dv, ws),
                           flush, a.iters)
                line.update(bwd_ms=tb, bwd_tflops=w.bwd_flops() / tb / 1e9, bwd_frac=w.bwd_flops() / tb / 1e9 / peak)
            fa.fa_check_status()
            print(json.dumps(line), flush=True)
            del t, o, lse
            torch.cuda.empty_cache()
        return
    for d in a.d:
        for N in a.N:
            H = max(1, a.rows // N)
            inp = fa_inputs.make_inputs(1, H, N, d, "bf16", seed=N + d, with_grad=True)
            q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
            scale = 1 / math.sqrt(d)
            o, lse = fa.fa_fwd(q, k, v, scale)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            ws = torch.empty(fa.fa_bwd_workspace_size(1, H, N, d), dtype=torch.uint8, device="cuda")
            tf = _time(lambda: fa.fa_fwd(q, k, v, scale, o, lse), flush, a.iters)
            tb = _time(lambda: fa.fa_bwd(q, k, v, o, do, lse, scale, dq, dk, dv, ws), flush, a.iters)
            tsn = _time(lambda: fa.fa_fwd_stepnorm(q, k, v, scale, o, lse), flush, a.iters) if a.stepnorm else None
            fa.fa_check_status()
            ff = 4.0 * H * N * N * d
            line = {"B": 1, "H": H, "N": N, "d": d, "fwd_ms": tf, "fwd_tflops": ff / tf / 1e9,
                    "fwd_frac": ff / tf / 1e9 / peak, "bwd_ms": tb, "bwd_tflops": 2.5 * ff / tb / 1e9,
                    "bwd_frac": 2.5 * ff / tb / 1e9 / peak, "fwdbwd_tflops": 3.5 * ff / (tf + tb) / 1e9,
                    "fwdbwd_frac": 3.5 * ff / (tf + tb) / 1e9 / peak, "peak_tflops": peak, "peak_source": src}
            if tsn is not None:
                line.update(stepnorm_fwd_ms=tsn, stepnorm_fwd_tflops=ff / tsn / 1e9, stepnorm_slowdown=tsn / tf)
            print(json.dumps(line), flush=True)
            del q, k, v, do, o, lse, dq, dk, dv, ws
            torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
