"""Runs the forward (and optionally the backward) on one seeded shape a few times: a fixed, small
command for profilers.  Example:
    python -m exact_io_aware_17_gb300.run_case --B 1 --H 32 --N 8192 --d 128 --iters 3 --bwd
"""
import argparse
import math
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import exact_io_aware_17_gb300 as fa  # noqa: E402
import fa_inputs  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--H", type=int, default=32)
    ap.add_argument("--N", type=int, default=8192)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--bwd", action="store_true")
    a = ap.parse_args()
    inp = fa_inputs.make_inputs(a.B, a.H, a.N, a.d, "bf16", seed=5, with_grad=a.bwd)
    t = {n: x.cuda() for n, x in inp.items()}
    scale = 1 / math.sqrt(a.d)
    for _ in range(a.iters):
        o, lse = fa.fa_fwd(t["q"], t["k"], t["v"], scale)
        if a.bwd:
            fa.fa_bwd(t["q"], t["k"], t["v"], o, t["do"], lse, scale)
    torch.cuda.synchronize()
    fa.fa_check_status()
    print("ok")


if __name__ == "__main__":
    main()
