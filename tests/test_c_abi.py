"""The C ABI used from a plain C program (tests/c/abi_smoke.c), with no Python in the call path."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_smoke.c")
LIBDIR = os.path.join(ROOT, "exact_io_aware_17_gb300")


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _build(tmp_path):
    cuda = _cuda_home()
    libdirs = [d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"),
                           os.path.join(cuda, "targets", "sbsa-linux", "lib"),
                           os.path.join(cuda, "targets", "x86_64-linux", "lib")) if os.path.isdir(d)]
    exe = str(tmp_path / "abi_smoke")
    cmd = ["gcc", "-std=c11", "-O1", f"-I{ROOT}/include", f"-I{cuda}/include", SRC, os.path.join(LIBDIR, "libfa.so"),
           *[f"-L{d}" for d in libdirs], "-lcudart", "-lm", f"-Wl,-rpath,{LIBDIR}",
           *[f"-Wl,-rpath,{d}" for d in libdirs], "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_program_compiles_against_the_header(tmp_path):
    if not os.path.exists(os.path.join(LIBDIR, "libfa.so")):
        pytest.skip("libfa.so not built")
    _build(tmp_path)


@pytest.mark.gpu
def test_c_program_runs_on_the_gpu(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "C ABI smoke: ok" in r.stdout
