"""Helpers of the GPU parity tests: run the CUDA path through the binding, compare with the oracle."""
import numpy as np
import pytest
import torch

# Tolerances of the attention paths (max-abs for O and LSE, relative Frobenius for the gradients).
TOL_F32 = 1e-4
TOL_O_BF16 = 2e-2
TOL_LSE_BF16 = 1e-3
TOL_GRAD_BF16 = 2e-2


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import exact_io_aware_17_gb300 as fa
    fa.load_library()
    return fa


def np64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def max_abs(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)))) if np.size(a) else 0.0


def rel_fro(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))
