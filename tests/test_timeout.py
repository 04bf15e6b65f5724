"""Failure detection of the bounded device waits (GPU; no fault, trap or hang).

With FA_TEST_STARVE_WAIT=1 in the environment the forward withholds its Q loads and its waits get a
~10 ms budget, so the MMA warp's first wait runs out: the kernel must wind down by itself (the other
warps stop at their next wait, tensor memory is freed) and fa_check_status must report FA_ERR_TIMEOUT.
The CUDA context must stay usable: the next call with the switch off computes correct results."""
import math

import pytest
import torch

import fa_inputs
import oracle
from parity_util import TOL_LSE_BF16, TOL_O_BF16, max_abs, need_gpu, np64

pytestmark = pytest.mark.gpu


def test_forward_wait_that_runs_out_reports_timeout(monkeypatch):
    fa = need_gpu()
    B, H, N, d = 1, 1, 200, 128
    scale = 1 / math.sqrt(d)
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", seed=77)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    fa.fa_check_status()                                  # start from a clear status word
    monkeypatch.setenv("FA_TEST_STARVE_WAIT", "1")
    fa.fa_fwd(q, k, v, scale)
    with pytest.raises(fa.FAError) as err:
        fa.fa_check_status()
    assert err.value.status == fa.FA_ERR_TIMEOUT
    monkeypatch.delenv("FA_TEST_STARVE_WAIT")
    fa.fa_check_status()                                  # reading the status cleared it
    o, lse = fa.fa_fwd(q, k, v, scale)
    torch.cuda.synchronize()
    fa.fa_check_status()
    ro, rl = oracle.forward(np64(inp["q"]), np64(inp["k"]), np64(inp["v"]), scale)
    assert max_abs(np64(o), ro) <= TOL_O_BF16
    assert max_abs(np64(lse), rl) <= TOL_LSE_BF16
