"""Failure detection of the bounded device waits (GPU; no fault, trap or hang).

While the test switch fa_test_force_wait_timeout(1) is on, the forward and backward kernels withhold their Q
loads and their waits get a ~10 ms budget, so the MMA warp's first wait on Q runs out: the kernel must wind down
by itself (the other warps stop at their next wait, copies in flight land, tensor memory is freed) and
fa_check_status must report FA_ERR_TIMEOUT.  The CUDA context must stay usable: the next call with the
switch off computes correct results."""
import math

import pytest
import torch

import fa_inputs
import oracle
from parity_util import TOL_GRAD_BF16, TOL_LSE_BF16, TOL_O_BF16, max_abs, need_gpu, np64, rel_fro

pytestmark = pytest.mark.gpu


def test_forward_wait_that_runs_out_reports_timeout():
    fa = need_gpu()
    B, H, N, d = 1, 1, 200, 128
    scale = 1 / math.sqrt(d)
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", seed=77)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    fa.fa_check_status()                                  # start from a clear status word
    fa.fa_test_force_wait_timeout(True)
    try:
        fa.fa_fwd(q, k, v, scale)
    finally:
        fa.fa_test_force_wait_timeout(False)
    with pytest.raises(fa.FAError) as err:
        fa.fa_check_status()
    assert err.value.status == fa.FA_ERR_TIMEOUT
    fa.fa_check_status()                                  # reading the status cleared it
    o, lse = fa.fa_fwd(q, k, v, scale)
    torch.cuda.synchronize()
    fa.fa_check_status()
    ro, rl = oracle.forward(np64(inp["q"]), np64(inp["k"]), np64(inp["v"]), scale)
    assert max_abs(np64(o), ro) <= TOL_O_BF16
    assert max_abs(np64(lse), rl) <= TOL_LSE_BF16


def test_backward_wait_that_runs_out_reports_timeout():
    fa = need_gpu()
    B, H, N, d = 1, 2, 300, 64
    scale = 1 / math.sqrt(d)
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", seed=78, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.fa_fwd(q, k, v, scale)
    torch.cuda.synchronize()
    fa.fa_check_status()                                  # start from a clear status word
    fa.fa_test_force_wait_timeout(True)
    try:
        fa.fa_bwd(q, k, v, o, do, lse, scale)
    finally:
        fa.fa_test_force_wait_timeout(False)
    with pytest.raises(fa.FAError) as err:
        fa.fa_check_status()
    assert err.value.status == fa.FA_ERR_TIMEOUT
    fa.fa_check_status()
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do, lse, scale)
    torch.cuda.synchronize()
    fa.fa_check_status()
    rq, rk, rv = oracle.backward(*(np64(inp[n]) for n in ("q", "k", "v", "do")), scale)
    errs = rel_fro(np64(dq), rq), rel_fro(np64(dk), rk), rel_fro(np64(dv), rv)
    assert max(errs) <= TOL_GRAD_BF16, errs


def test_environment_cannot_switch_the_test_path_on(monkeypatch):
    """The old environment switch is gone: with it set, calls compute normally and report no timeout."""
    fa = need_gpu()
    monkeypatch.setenv("FA_TEST_STARVE_WAIT", "1")
    B, H, N, d = 1, 2, 300, 128
    scale = 1 / math.sqrt(d)
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", seed=79)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    fa.fa_check_status()
    o, lse = fa.fa_fwd(q, k, v, scale)
    torch.cuda.synchronize()
    fa.fa_check_status()
    ro, rl = oracle.forward(np64(inp["q"]), np64(inp["k"]), np64(inp["v"]), scale)
    assert max_abs(np64(o), ro) <= TOL_O_BF16
