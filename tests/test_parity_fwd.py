"""GPU forward parity: the CUDA path through the C ABI against the fp64 oracle on the same seeded inputs."""
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from parity_util import (TOL_F32, TOL_LSE_BF16, TOL_O_BF16, max_abs, need_gpu, np64)

pytestmark = pytest.mark.gpu


def _run_bf16(fa, inp, scale, entry="fa_fwd"):
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = getattr(fa, entry)(q, k, v, scale)
    torch.cuda.synchronize()
    fa.fa_check_status()
    return o, lse


def _check_full_bf16(fa, B, H, N, d, seed, q_gain=1.0, entry="fa_fwd"):
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", seed, q_gain)
    scale = 1 / math.sqrt(d)
    o, lse = _run_bf16(fa, inp, scale, entry)
    ro, rl = oracle.forward(np64(inp["q"]), np64(inp["k"]), np64(inp["v"]), scale)
    eo, el = max_abs(np64(o), ro), max_abs(np64(lse), rl)
    assert eo <= TOL_O_BF16, (B, H, N, d, eo)
    assert el <= TOL_LSE_BF16, (B, H, N, d, el)
    return eo, el


# --- fp32 path ------------------------------------------------------------------------------------

def test_fp32_workload_b1_h1_n64_d16():
    fa = need_gpu()
    w = fa_inputs.WORKLOADS["fp32-fwd-B1-H1-N64-d16"]
    inp = fa_inputs.workload_inputs(w)
    o, lse = fa.fa_fwd_f32(*(inp[n].cuda() for n in ("q", "k", "v")), w.scale)
    ro, rl = oracle.forward(*(np64(inp[n]) for n in ("q", "k", "v")), w.scale)
    assert max_abs(np64(o), ro) <= TOL_F32
    assert max_abs(np64(lse), rl) <= TOL_F32


@pytest.mark.parametrize("N", [1, 7, 33, 65, 129, 300])
@pytest.mark.parametrize("d", [4, 16, 64, 128])
def test_fp32_ragged_and_head_sizes(N, d):
    fa = need_gpu()
    inp = fa_inputs.make_inputs(2, 3, N, d, "f32", seed=100 + N + d)
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd_f32(*(inp[n].cuda() for n in ("q", "k", "v")), scale)
    ro, rl = oracle.forward(*(np64(inp[n]) for n in ("q", "k", "v")), scale)
    assert max_abs(np64(o), ro) <= TOL_F32
    assert max_abs(np64(lse), rl) <= TOL_F32


# --- bf16 tensor-core path: small shapes spanning several tiles and ragged tails ---------------------

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 7, 128, 129, 255, 256, 257, 300, 513, 1000])
def test_bf16_ragged(N, d):
    fa = need_gpu()
    _check_full_bf16(fa, 1, 3, N, d, seed=200 + N + d)


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_several_heads_and_batches(d):
    fa = need_gpu()
    _check_full_bf16(fa, 2, 5, 777, d, seed=300 + d)


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_peaky_rows_move_the_max_late(d):
    """Q scaled by 4: rows are peaky and the running max keeps growing across blocks (rescale path)."""
    fa = need_gpu()
    _check_full_bf16(fa, 1, 2, 1500, d, seed=400 + d, q_gain=4.0)


@pytest.mark.parametrize("H,N", [(1, 1024), (160, 384)])
@pytest.mark.parametrize("d", [64, 128])
def test_bf16_increasing_scores_force_every_rescale(d, H, N):
    """Keys ordered so every new block holds larger scores than all before it: every block rescales O,
    the last one included.  One head of 1024 keys runs as split 2-CTA clusters only; 160 heads of 384
    keys (a ragged last block) fill two full waves before the split tail."""
    fa = need_gpu()
    g = torch.Generator().manual_seed(7)
    q = torch.ones(1, H, N, d) / 4
    k = (torch.linspace(0, 800, N)[:, None] * torch.ones(d) / d * 4).expand(1, H, N, d)
    v = torch.randn(1, H, N, d, generator=g)
    inp = {n: t.to(torch.bfloat16).contiguous() for n, t in (("q", q), ("k", k), ("v", v))}
    scale = 1 / math.sqrt(d)
    o, lse = _run_bf16(fa, inp, scale)
    ro, rl = oracle.forward(np64(inp["q"]), np64(inp["k"]), np64(inp["v"]), scale)
    assert max_abs(np64(o), ro) <= TOL_O_BF16
    assert max_abs(np64(lse), rl) <= TOL_LSE_BF16


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_zero_queries_give_column_mean(d):
    fa = need_gpu()
    B, H, N = 1, 2, 700
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", seed=500 + d)
    inp["q"] = torch.zeros_like(inp["q"])
    o, lse = _run_bf16(fa, inp, 1 / math.sqrt(d))
    mean = np64(inp["v"]).mean(axis=2, keepdims=True)
    assert max_abs(np64(o), np.broadcast_to(mean, o.shape)) <= TOL_O_BF16
    assert max_abs(np64(lse), math.log(N)) <= TOL_LSE_BF16


def test_bf16_single_key_gives_value():
    fa = need_gpu()
    inp = fa_inputs.make_inputs(3, 2, 1, 128, "bf16", seed=600)
    o, lse = _run_bf16(fa, inp, 0.1)
    assert max_abs(np64(o), np64(inp["v"])) <= TOL_O_BF16
    qk = (np64(inp["q"]) * np64(inp["k"])).sum(-1) * 0.1
    assert max_abs(np64(lse), qk) <= TOL_LSE_BF16


def test_bf16_no_n_squared_allocation():
    fa = need_gpu()
    B, H, N, d = 1, 4, 4096, 128
    inp = fa_inputs.make_inputs(B, H, N, d, "bf16", seed=700)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device="cuda")
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    before = torch.cuda.memory_allocated()
    fa.fa_fwd(q, k, v, None, o, lse)
    torch.cuda.synchronize()
    assert torch.cuda.max_memory_allocated() - before < 1 << 20   # S alone would be B*H*N*N*4 = 268 MB


# --- the five workloads at full size (sampled rows where the oracle needs them) ----------------------

def _sampled(fa, w, rows_per_head):
    inp = fa_inputs.workload_inputs(w, with_grad=False)
    o, lse = _run_bf16(fa, inp, w.scale)
    rows = fa_inputs.sample_rows(w.N, w.H, rows_per_head)
    ro, rl = oracle.forward_rows(np64(inp["q"]), np64(inp["k"]), np64(inp["v"]), w.scale,
                                 [r.numpy() for r in rows])
    go = np.stack([np64(o[:, h, rows[h]]) for h in range(w.H)], axis=1)
    gl = np.stack([np64(lse[:, h, rows[h]]) for h in range(w.H)], axis=1)
    assert max_abs(go, ro) <= TOL_O_BF16
    assert max_abs(gl, rl) <= TOL_LSE_BF16
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    return o, lse


def test_workload_b4_h16_n2048_d64_full():
    fa = need_gpu()
    w = fa_inputs.WORKLOADS["bf16-fwdbwd-B4-H16-N2048-d64"]
    inp = fa_inputs.workload_inputs(w, with_grad=False)
    o, lse = _run_bf16(fa, inp, w.scale)
    ro, rl = oracle.forward(np64(inp["q"]), np64(inp["k"]), np64(inp["v"]), w.scale)
    assert max_abs(np64(o), ro) <= TOL_O_BF16
    assert max_abs(np64(lse), rl) <= TOL_LSE_BF16


@pytest.mark.parametrize("name", ["bf16-fwdbwd-B1-H16-N8192-d128", "bf16-fwd-B1-H8-N32768-d128-q4"])
def test_workload_every_element(name):
    """The headline workload (B=1 H=16 N=8192 d=128) and the peaky long one (B=1 H=8 N=32768 d=128, Q x 4):
    every element of O and LSE of every head against the oracle, which forms each row's full softmax
    (in blocks of whole rows, to bound its memory)."""
    fa = need_gpu()
    w = fa_inputs.WORKLOADS[name]
    inp = fa_inputs.workload_inputs(w, with_grad=False)
    o, lse = _run_bf16(fa, inp, w.scale)
    go, gl = np64(o), np64(lse)
    del o, lse
    for h in range(w.H):        # one head at a time keeps the oracle's memory at one head's arrays
        ro, rl = oracle.forward(*(np64(inp[n][:, h:h + 1]) for n in ("q", "k", "v")), w.scale)
        assert max_abs(go[:, h:h + 1], ro) <= TOL_O_BF16, (name, h)
        assert max_abs(gl[:, h:h + 1], rl) <= TOL_LSE_BF16, (name, h)


def test_workload_b1_h4_n131072_d128_sampled_rows():
    """The longest workload: the oracle checks a seeded sample of 256 query rows per head, each against
    all 131072 keys."""
    fa = need_gpu()
    _sampled(fa, fa_inputs.WORKLOADS["bf16-fwd-B1-H4-N131072-d128"], 256)


# --- the per-step normalised accumulator (fa_fwd_stepnorm): same results, different update rule --------

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 7, 129, 300, 1000])
def test_stepnorm_ragged(N, d):
    fa = need_gpu()
    _check_full_bf16(fa, 1, 3, N, d, seed=1200 + N + d, entry="fa_fwd_stepnorm")


@pytest.mark.parametrize("d", [64, 128])
def test_stepnorm_peaky_rows(d):
    fa = need_gpu()
    _check_full_bf16(fa, 1, 2, 1500, d, seed=1400 + d, q_gain=4.0, entry="fa_fwd_stepnorm")


def test_stepnorm_agrees_with_fa_fwd_at_the_headline_shape():
    """Both update rules on the B=1 H=16 N=8192 d=128 workload: sampled rows against the oracle, and the
    two GPU results within the bf16 output tolerance of each other everywhere."""
    fa = need_gpu()
    w = fa_inputs.WORKLOADS["bf16-fwdbwd-B1-H16-N8192-d128"]
    inp = fa_inputs.workload_inputs(w, with_grad=False)
    o1, l1 = _run_bf16(fa, inp, w.scale, "fa_fwd")
    o2, l2 = _run_bf16(fa, inp, w.scale, "fa_fwd_stepnorm")
    assert (o1.float() - o2.float()).abs().max().item() <= TOL_O_BF16
    assert (l1 - l2).abs().max().item() <= TOL_LSE_BF16
    rows = fa_inputs.sample_rows(w.N, w.H, 64)
    ro, rl = oracle.forward_rows(np64(inp["q"]), np64(inp["k"]), np64(inp["v"]), w.scale, [r.numpy() for r in rows])
    go = np.stack([np64(o2[:, h, rows[h]]) for h in range(w.H)], axis=1)
    gl = np.stack([np64(l2[:, h, rows[h]]) for h in range(w.H)], axis=1)
    assert max_abs(go, ro) <= TOL_O_BF16
    assert max_abs(gl, rl) <= TOL_LSE_BF16


@pytest.mark.parametrize("entry", ["fa_fwd", "fa_fwd_f32"])
def test_more_heads_than_a_grid_dimension_holds(entry):
    """B*H = 70,000 short heads: more than the 65,535 CUDA allows in a grid's y dimension."""
    fa = need_gpu()
    B, H, N, d = 7, 10000, 3, 64
    dtype = "bf16" if entry == "fa_fwd" else "f32"
    inp = fa_inputs.make_inputs(B, H, N, d, dtype, seed=4321)
    o, lse = getattr(fa, entry)(*(inp[n].cuda() for n in ("q", "k", "v")), 0.125)
    torch.cuda.synchronize()
    fa.fa_check_status()
    sel = [0, 1234, 69999]
    qf, kf, vf = (inp[n].reshape(B * H, 1, N, d)[sel].transpose(0, 1) for n in ("q", "k", "v"))
    ro, rl = oracle.forward(np64(qf), np64(kf), np64(vf), 0.125)
    tol_o, tol_l = (TOL_O_BF16, TOL_LSE_BF16) if entry == "fa_fwd" else (TOL_F32, TOL_F32)
    assert max_abs(np64(o.reshape(B * H, N, d)[sel]), ro[0]) <= tol_o
    assert max_abs(np64(lse.reshape(B * H, N)[sel]), rl[0]) <= tol_l


@pytest.mark.parametrize("H,N,d", [(16, 8192, 128), (32, 2048, 64), (3, 1000, 128)])
def test_forward_is_bitwise_repeatable(H, N, d):
    """No atomics and a fixed order of blocks per CTA (the split tail merges its two halves in a fixed
    order too): two calls on the same inputs give the same bits."""
    fa = need_gpu()
    inp = fa_inputs.make_inputs(1, H, N, d, "bf16", seed=77)
    scale = 1 / math.sqrt(d)
    o1, l1 = _run_bf16(fa, inp, scale)
    o2, l2 = _run_bf16(fa, inp, scale)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
