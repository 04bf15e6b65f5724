"""GPU backward parity: dQ, dK, dV of the CUDA path against the fp64 oracle (relative Frobenius error)."""
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from parity_util import TOL_GRAD_BF16, max_abs, need_gpu, np64, rel_fro

pytestmark = pytest.mark.gpu


def _gpu_fwd_bwd(fa, inp, scale):
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.fa_fwd(q, k, v, scale)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do, lse, scale)
    torch.cuda.synchronize()
    fa.fa_check_status()
    return o, lse, dq, dk, dv


def _check_full(fa, B, H, N, d, seed, q_gain=1.0):
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", seed, q_gain, with_grad=True)
    scale = 1 / math.sqrt(d)
    _, _, dq, dk, dv = _gpu_fwd_bwd(fa, inp, scale)
    rq, rk, rv = oracle.backward(*(np64(inp[n]) for n in ("q", "k", "v", "do")), scale)
    if N == 1:
        # One key: P = 1, so dS = 0 and the exact dQ and dK vanish; a relative error is undefined there.
        assert max_abs(np64(dq), 0.0) <= 1e-3 and max_abs(np64(dk), 0.0) <= 1e-3
        assert rel_fro(np64(dv), rv) <= TOL_GRAD_BF16
        return
    errs = rel_fro(np64(dq), rq), rel_fro(np64(dk), rk), rel_fro(np64(dv), rv)
    assert max(errs) <= TOL_GRAD_BF16, (B, H, N, d, errs)
    return errs


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 7, 64, 65, 128, 129, 200, 383, 512])
def test_bwd_ragged(N, d):
    fa = need_gpu()
    _check_full(fa, 1, 2, N, d, seed=800 + N + d)


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_several_heads(d):
    fa = need_gpu()
    _check_full(fa, 2, 3, 1000, d, seed=900 + d)


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_peaky_rows(d):
    fa = need_gpu()
    _check_full(fa, 1, 2, 777, d, seed=950 + d, q_gain=4.0)


def test_bwd_gradient_invariants_on_gpu_outputs():
    """sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i hold for exact gradients at any size."""
    fa = need_gpu()
    B, H, N, d = 1, 4, 3000, 128
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", 990, with_grad=True)
    _, _, dq, dk, dv = _gpu_fwd_bwd(fa, inp, 1 / math.sqrt(d))
    dk_sum = dk.double().sum(dim=2)
    dv_sum = dv.double().sum(dim=2)
    do_sum = inp["do"].double().sum(dim=2).cuda()
    scale_k = dk.double().abs().sum(dim=2)
    assert (dk_sum.abs() <= 2e-2 * scale_k + 1e-3).all()
    assert ((dv_sum - do_sum).abs() <= 2e-2 * dv.double().abs().sum(dim=2) + 1e-3).all()


def test_workload_b4_h16_n2048_d64_full():
    fa = need_gpu()
    w = fa_inputs.WORKLOADS["bf16-fwdbwd-B4-H16-N2048-d64"]
    inp = fa_inputs.workload_inputs(w)
    _, _, dq, dk, dv = _gpu_fwd_bwd(fa, inp, w.scale)
    rq, rk, rv = oracle.backward(*(np64(inp[n]) for n in ("q", "k", "v", "do")), w.scale)
    errs = rel_fro(np64(dq), rq), rel_fro(np64(dk), rk), rel_fro(np64(dv), rv)
    assert max(errs) <= TOL_GRAD_BF16, errs


def test_workload_b1_h16_n8192_d128_every_element():
    """The headline workload: dQ, dK and dV of all 16 heads against the full oracle, relative Frobenius
    error per tensor over the whole [B, H, N, d] array."""
    fa = need_gpu()
    w = fa_inputs.WORKLOADS["bf16-fwdbwd-B1-H16-N8192-d128"]
    inp = fa_inputs.workload_inputs(w)
    _, _, dq, dk, dv = _gpu_fwd_bwd(fa, inp, w.scale)
    got = [np64(t) for t in (dq, dk, dv)]
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    del dq, dk, dv
    ref = [np.empty_like(g) for g in got]
    for h in range(w.H):        # one head at a time bounds the oracle's memory
        parts = oracle.backward(*(np64(inp[n][:, h:h + 1]) for n in ("q", "k", "v", "do")), w.scale)
        for r, p in zip(ref, parts):
            r[:, h:h + 1] = p
    errs = [rel_fro(g, r) for g, r in zip(got, ref)]
    assert max(errs) <= TOL_GRAD_BF16, errs


def _long_backward_check(fa, w, q_rows, k_rows, k_head):
    """Backward of workload w at full size: dQ at q_rows sampled query rows of every head; dK and dV at
    k_rows sampled key rows of head k_head (each needs every query row's softmax of that head); the exact
    invariants sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i on every head."""
    inp = fa_inputs.workload_inputs(w, with_grad=True)
    _, _, dq, dk, dv = _gpu_fwd_bwd(fa, inp, w.scale)
    qrows = fa_inputs.sample_rows(w.N, w.H, q_rows, seed_base=1000)
    krows = fa_inputs.sample_rows(w.N, w.H, k_rows, seed_base=2000)
    for h in range(w.H):
        sub = {n: np64(inp[n][:, h:h + 1]) for n in ("q", "k", "v", "do")}
        if h == k_head:
            rq, rk, rv = oracle.backward_rows(sub["q"], sub["k"], sub["v"], sub["do"], w.scale,
                                              [qrows[h].numpy()], [krows[h].numpy()])
            assert max(rel_fro(np64(dk[:, h:h + 1, krows[h]]), rk),
                       rel_fro(np64(dv[:, h:h + 1, krows[h]]), rv)) <= TOL_GRAD_BF16, h
        else:
            rq = _dq_rows(sub, w.scale, qrows[h].numpy())
        assert rel_fro(np64(dq[:, h:h + 1, qrows[h]]), rq) <= TOL_GRAD_BF16, h
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    dk_sum = dk.double().sum(dim=2)
    assert (dk_sum.abs() <= 2e-2 * dk.double().abs().sum(dim=2) + 1e-3).all()
    dv_err = dv.double().sum(dim=2) - inp["do"].double().sum(dim=2).cuda()
    assert (dv_err.abs() <= 2e-2 * dv.double().abs().sum(dim=2) + 1e-3).all()


def _dq_rows(sub, scale, rows):
    """The oracle's dQ at the given query rows of one head (no key rows asked: only those rows' softmax)."""
    rq, _, _ = oracle.backward_rows(sub["q"], sub["k"], sub["v"], sub["do"], scale, [rows],
                                    [np.zeros(0, dtype=np.int64)])
    return rq


def test_bwd_workload_shape_b1_h8_n32768_d128_q4():
    """Backward at the peaky long workload's shape and inputs (B=1 H=8 N=32768 d=128, Q x 4)."""
    fa = need_gpu()
    _long_backward_check(fa, fa_inputs.WORKLOADS["bf16-fwd-B1-H8-N32768-d128-q4"], 256, 64, k_head=5)


@pytest.mark.slow
def test_bwd_workload_shape_b1_h4_n131072_d128():
    """Backward at the longest workload's shape and inputs (B=1 H=4 N=131072 d=128).  The dK/dV rows of one
    head need that head's whole softmax (1.7e10 scores) in the oracle: about two minutes of CPU."""
    fa = need_gpu()
    _long_backward_check(fa, fa_inputs.WORKLOADS["bf16-fwd-B1-H4-N131072-d128"], 256, 32, k_head=2)


def test_bwd_workspace_contents_do_not_matter():
    fa = need_gpu()
    B, H, N, d = 1, 2, 300, 64
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", 991, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.fa_fwd(q, k, v)
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    ws.fill_(0x7f)
    g1 = fa.fa_bwd(q, k, v, o, do, lse, workspace=ws)
    ws.fill_(0xff)
    g2 = fa.fa_bwd(q, k, v, o, do, lse, workspace=ws)
    torch.cuda.synchronize()
    for a, b in zip(g1, g2):
        assert rel_fro(np64(a), np64(b)) <= 1e-2


@pytest.mark.parametrize("N,d,q_gain", [(32768, 128, 4.0), (32768, 64, 1.0), (8192, 64, 1.0)])
def test_bwd_long_sequences_sampled(N, d, q_gain):
    """Backward at long N (the peaky N=32K workload and d=64 up to 32K): a two-head launch, the oracle
    checks 128 query rows (dQ) and 128 key rows (dK, dV) of head 1, and the exact invariants hold for
    both heads at full size."""
    fa = need_gpu()
    B, H = 1, 2
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", 3000 + N + d, q_gain, with_grad=True)
    scale = 1 / math.sqrt(d)
    _, _, dq, dk, dv = _gpu_fwd_bwd(fa, inp, scale)
    qrows = fa_inputs.sample_rows(N, H, 128, seed_base=1000)
    krows = fa_inputs.sample_rows(N, H, 128, seed_base=2000)
    sub = {n: np64(inp[n][:, 1:2]) for n in ("q", "k", "v", "do")}
    rq, rk, rv = oracle.backward_rows(sub["q"], sub["k"], sub["v"], sub["do"], scale,
                                      [qrows[1].numpy()], [krows[1].numpy()])
    errs = (rel_fro(np64(dq[:, 1:2, qrows[1]]), rq), rel_fro(np64(dk[:, 1:2, krows[1]]), rk),
            rel_fro(np64(dv[:, 1:2, krows[1]]), rv))
    assert max(errs) <= TOL_GRAD_BF16, errs
    dk_sum = dk.double().sum(dim=2)
    assert (dk_sum.abs() <= 2e-2 * dk.double().abs().sum(dim=2) + 1e-3).all()
    dv_err = dv.double().sum(dim=2) - inp["do"].double().sum(dim=2).cuda()
    assert (dv_err.abs() <= 2e-2 * dv.double().abs().sum(dim=2) + 1e-3).all()


def test_bwd_more_heads_than_a_grid_dimension_holds():
    fa = need_gpu()
    B, H, N, d = 7, 10000, 5, 64
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", seed=4322, with_grad=True)
    _, _, dq, dk, dv = _gpu_fwd_bwd(fa, inp, 0.125)
    sel = [0, 4321, 69999]
    sub = [inp[n].reshape(B * H, 1, N, d)[sel].transpose(0, 1) for n in ("q", "k", "v", "do")]
    rq, rk, rv = oracle.backward(*(np64(t) for t in sub), 0.125)
    for g, r in ((dq, rq), (dk, rk), (dv, rv)):
        assert rel_fro(np64(g.reshape(B * H, N, d)[sel]), r[0]) <= TOL_GRAD_BF16


def test_bwd_allocates_nothing_with_caller_buffers():
    """With every output and the workspace owned by the caller, fa_bwd allocates no device memory at all;
    the workspace itself is O(B*H*N*d) (one fp32 score matrix at this shape would be 67 MB per head)."""
    fa = need_gpu()
    B, H, N, d = 1, 4, 4096, 128
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", seed=731, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.fa_fwd(q, k, v, 1 / math.sqrt(d))
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    assert ws.numel() < 2 * B * H * N * (d + 2) * 4 + 4096
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    before = torch.cuda.memory_allocated()
    fa.fa_bwd(q, k, v, o, do, lse, 1 / math.sqrt(d), dq, dk, dv, ws)
    torch.cuda.synchronize()
    fa.fa_check_status()
    assert torch.cuda.max_memory_allocated() == before


def test_kernel_launch_counter_per_call():
    """The library counts its own launches: fa_fwd enqueues one kernel, or two when the last partial wave
    of tile pairs runs as 2-CTA clusters; fa_bwd enqueues three (row terms, main, dQ conversion)."""
    fa = need_gpu()
    inp = fa_inputs.make_inputs(1, 4, 1024, 128, "bf16", seed=77, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    n0 = fa.fa_kernel_launches()
    o, lse = fa.fa_fwd(q, k, v, 0.088)
    n1 = fa.fa_kernel_launches()
    fa.fa_bwd(q, k, v, o, do, lse, 0.088)
    n2 = fa.fa_kernel_launches()
    torch.cuda.synchronize()
    fa.fa_check_status()
    assert n1 - n0 in (1, 2)
    assert n2 - n1 == 3


@pytest.mark.parametrize("H,N,d", [(16, 4096, 128), (16, 2048, 64)])
def test_bwd_dk_dv_bitwise_repeatable_dq_within_rounding(H, N, d):
    """dK and dV accumulate in tensor memory in a fixed order per CTA: the same bits on every call.  dQ is
    the sum of per-key-block reduce-adds whose order varies between calls, so only its rounding may differ
    (bounded here by 1 % of max |dQ|, about two bf16 ulps)."""
    fa = need_gpu()
    inp = fa_inputs.make_inputs(1, H, N, d, "bf16", seed=78, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(q, k, v, scale)
    r1 = fa.fa_bwd(q, k, v, o, do, lse, scale)
    r2 = fa.fa_bwd(q, k, v, o, do, lse, scale)
    torch.cuda.synchronize()
    fa.fa_check_status()
    dq1, dk1, dv1 = r1
    dq2, dk2, dv2 = r2
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert (dq1.float() - dq2.float()).abs().max().item() <= 1e-2 * dq1.float().abs().max().item()


def test_bwd_rejects_bad_caller_outputs_and_workspace():
    """Caller-given dq/dk/dv and workspace are checked before the library is called (a wrong dtype or shape
    would otherwise let the kernels write past the end of the buffer)."""
    fa = need_gpu()
    B, H, N, d = 1, 2, 256, 64
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", seed=79, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.fa_fwd(q, k, v)
    launches = fa.fa_kernel_launches()
    bad = [dict(dq=torch.empty(B, H, N, d, dtype=torch.float32, device="cuda")),
           dict(dk=torch.empty(B, H, N - 1, d, dtype=torch.bfloat16, device="cuda")),
           dict(dv=torch.empty(B, H, N, d, dtype=torch.bfloat16, device="cuda").transpose(2, 3).contiguous()
                .transpose(2, 3)),
           dict(workspace=torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8))]
    for kw in bad:
        with pytest.raises(ValueError):
            fa.fa_bwd(q, k, v, o, do, lse, **kw)
    for kw in bad[:3]:
        with pytest.raises(ValueError):
            fa.fa_bwd_noalloc(q, k, v, o, do, lse, **kw)
    torch.cuda.synchronize()
    assert fa.fa_kernel_launches() == launches    # nothing was launched


def test_main_kernel_timing_events_are_recorded_once():
    """fa_debug_time_bwd_main: the next backward records the two events around its main kernel only (a
    positive time below the whole call's), and the setting is used once."""
    fa = need_gpu()
    B, H, N, d = 1, 8, 4096, 128
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", seed=81, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.fa_fwd(q, k, v)
    stream = torch.cuda.current_stream()
    e0, e1, a, b = (torch.cuda.Event(enable_timing=True) for _ in range(4))
    for e in (e0, e1):
        e.record(stream)
    torch.cuda.synchronize()
    fa.fa_debug_time_bwd_main(e0, e1)
    a.record(stream)
    fa.fa_bwd(q, k, v, o, do, lse)
    b.record(stream)
    torch.cuda.synchronize()
    main_ms, call_ms = e0.elapsed_time(e1), a.elapsed_time(b)
    assert 0 < main_ms < call_ms
    fa.fa_bwd(q, k, v, o, do, lse)            # the setting was used once: these events stay as they were
    torch.cuda.synchronize()
    assert e0.elapsed_time(e1) == main_ms
    # A call that fails its checks takes the request too, so the next valid call records nothing.
    fa.fa_debug_time_bwd_main(e0, e1)
    lib = fa.load_library()
    null9 = [None] * 9
    assert lib.fa_bwd(*null9, B, H, N, d, 0.1, None, 0, None) == fa.FA_ERR_INVALID_ARG
    fa.fa_bwd(q, k, v, o, do, lse)
    torch.cuda.synchronize()
    assert e0.elapsed_time(e1) == main_ms
    fa.fa_check_status()


@pytest.mark.parametrize("d", [64, 128])
def test_timing_events_between_dependent_launches_change_nothing(d):
    """The main and dQ-conversion kernels start as programmatic dependents of the kernel before them; with
    the timing events recorded between the kernels the call must give the same gradients (dK, dV bitwise,
    dQ up to the order of its reduce-adds) as without."""
    fa = need_gpu()
    B, H, N = 2, 8, 2000      # ragged: the last key block of each head is partial
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", seed=82, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.fa_fwd(q, k, v)
    dq0, dk0, dv0 = fa.fa_bwd(q, k, v, o, do, lse)
    e0, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
    for e in (e0, e1):
        e.record(torch.cuda.current_stream())
    fa.fa_debug_time_bwd_main(e0, e1)
    dq1, dk1, dv1 = fa.fa_bwd(q, k, v, o, do, lse)
    torch.cuda.synchronize()
    fa.fa_check_status()
    assert torch.equal(dk0, dk1) and torch.equal(dv0, dv1)
    rel = ((dq0.float() - dq1.float()).norm() / dq0.float().norm()).item()
    assert rel < 1e-3


def test_forward_and_backward_replay_from_a_cuda_graph():
    """Both calls captured into one CUDA graph (their launches include programmatic dependents and the
    forward's 2-CTA cluster tail) replay to the results of the same calls made eagerly."""
    fa = need_gpu()
    B, H, N, d = 1, 20, 2048, 128       # 160 tile pairs: one full wave of 152 plus a split tail of 8
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", seed=83, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    scale = 1 / math.sqrt(d)
    o0, lse0 = fa.fa_fwd(q, k, v, scale)
    dq0, dk0, dv0 = fa.fa_bwd(q, k, v, o0, do, lse0, scale)
    o, lse = torch.empty_like(q), torch.empty(B, H, N, dtype=torch.float32, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=q.device)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                # warm-up off the default stream, as graph capture wants
        fa.fa_fwd(q, k, v, scale, o, lse)
        fa.fa_bwd(q, k, v, o, do, lse, scale, dq, dk, dv, ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for t in (o, lse, dq, dk, dv):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.fa_fwd(q, k, v, scale, o, lse)
        fa.fa_bwd(q, k, v, o, do, lse, scale, dq, dk, dv, ws)
    g.replay()
    torch.cuda.synchronize()
    fa.fa_check_status()
    assert torch.equal(o, o0) and torch.equal(lse, lse0)
    assert torch.equal(dk, dk0) and torch.equal(dv, dv0)
    assert rel_fro(np64(dq), np64(dq0)) < 1e-3
