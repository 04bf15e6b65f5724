"""Measured throughput of the exponential unit (ex2.approx.f32) on this GPU: the ceiling of the softmax
exponentials, beside the tensor-core ceiling of the products.

    python -m exact_io_aware_17_gb300.mufu_peak

Compiles measure/mufu_peak.cu for sm_103a into a temporary directory, runs it and prints one JSON line
(ex2 per second over the whole GPU, ex2 per SM per clock).
"""
import os
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))


def main():
    src = os.path.join(HERE, "measure", "mufu_peak.cu")
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "mufu_peak")
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe, src], check=True)
        r = subprocess.run([exe], capture_output=True, text=True)
        sys.stdout.write(r.stdout)
        if r.returncode != 0:
            sys.stderr.write(r.stderr)
        return r.returncode


if __name__ == "__main__":
    sys.exit(main())
