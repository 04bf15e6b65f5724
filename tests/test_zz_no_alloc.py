"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory (a plugin handed only
its input and output buffers, or code that must not call cudaMalloc because it can synchronise the
device).  It runs the same kernels as fa_bwd on a scratch array compiled into the library, so its
gradients must match fa_bwd's, call after call, while the array keeps each call's leftovers.

This file is collected last on purpose: the GPU test calls the entry point after every other test
has run, and also works alone in a fresh process."""
import ctypes
import math

import pytest
import torch

import fa_inputs
from parity_util import TOL_GRAD_BF16, need_gpu, np64, rel_fro


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    """Host-side check, no GPU needed: nothing is launched for a shape that does not fit."""
    import exact_io_aware_17_gb300 as fa
    lib = fa.load_library()
    B, H, N, d = 1, 16, 8192, 128
    assert fa.fa_bwd_workspace_size(B, H, N, d) > fa.NOALLOC_MAX_SCRATCH_BYTES
    fake = [ctypes.c_void_p(0x10000)] * 9
    st = lib.fa_bwd_noalloc(*fake, B, H, N, d, 1 / math.sqrt(d), None)
    assert st == fa.FA_ERR_INVALID_ARG
    assert "static scratch" in fa.fa_last_error_string()


def test_noalloc_checks_the_head_size_before_the_scratch_size():
    """Host-side check: an unsupported head size is reported as such, under this entry point's name, even
    for a shape whose scratch would not fit either; nothing is launched."""
    import exact_io_aware_17_gb300 as fa
    lib = fa.load_library()
    fake = [ctypes.c_void_p(0x10000)] * 9
    launches = fa.fa_kernel_launches()
    st = lib.fa_bwd_noalloc(*fake, 1, 16, 8192, 96, 0.1, None)
    assert st == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_last_error_string().startswith("fa_bwd_noalloc: d must be 64 or 128")
    st = lib.fa_bwd_noalloc(*fake, 1, 0, 8192, 128, 0.1, None)
    assert st == fa.FA_ERR_INVALID_ARG and fa.fa_last_error_string().startswith("fa_bwd_noalloc:")
    assert fa.fa_kernel_launches() == launches


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(2, 4, 1000, 128), (1, 3, 2049, 64)])
def test_noalloc_matches_fa_bwd_on_two_calls_in_a_row(shape):
    fa = need_gpu()
    B, H, N, d = shape
    assert fa.fa_bwd_workspace_size(B, H, N, d) <= fa.NOALLOC_MAX_SCRATCH_BYTES
    scale = 1 / math.sqrt(d)
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", seed=4242 + N, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.fa_fwd(q, k, v, scale)
    ref = fa.fa_bwd(q, k, v, o, do, lse, scale)
    outs = [tuple(torch.empty_like(q) for _ in range(3)) for _ in range(2)]
    # The set-up call: with CUDA's lazy module loading the library's kernels and the static array reach the
    # device at their first use, which is this call when the test runs alone in a fresh process.
    fa.fa_bwd_noalloc(q, k, v, o, do, lse, scale, *outs[0])
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    before = torch.cuda.memory_allocated()
    free_before = torch.cuda.mem_get_info()[0]
    for dq, dk, dv in outs:                         # two calls in a row on the shared static scratch
        fa.fa_bwd_noalloc(q, k, v, o, do, lse, scale, dq, dk, dv)
    torch.cuda.synchronize()
    # No torch allocation during the calls: the peak never rose above what was allocated before them
    # (the current figure may drop if the collector frees an unrelated tensor meanwhile) ...
    assert torch.cuda.max_memory_allocated() <= before
    # ... and no allocation inside the library either: the device's free memory did not shrink (the
    # static array is part of the library's device code, which the set-up call loaded).
    assert torch.cuda.mem_get_info()[0] >= free_before
    fa.fa_check_status()
    for got in outs:
        for g, r in zip(got, ref):
            assert rel_fro(np64(g), np64(r)) <= TOL_GRAD_BF16
