"""Pins for the fp64 oracle, against what the pages and the mathematics fix (CPU only).

Each check is chosen so that a plausible slip in the oracle (a dropped max subtraction, a wrong
scale, a transposed operand, a missing rescale factor, a sign error in the backward) fails at least
one of them.  None of the expected values comes from the CUDA path.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import sdpa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            vals[key] = [float(x) for x in val.split()]
    return vals


def _rand(shape, seed, gain=1.0):
    rng = np.random.default_rng(seed)
    return gain * rng.standard_normal(shape)


# --- closed forms and hand-worked values -------------------------------------------------------

def test_hand_worked_example():
    g = _read_golden("hand_example.txt")
    q = np.array(g["q"]).reshape(1, 1, 1, 1)
    k = np.array(g["k"]).reshape(1, 1, 2, 1)
    v = np.array(g["v"]).reshape(1, 1, 2, 1)
    o, lse = oracle.forward(q, k, v, 1.0)
    assert abs(o[0, 0, 0, 0] - g["o"][0]) < 1e-13
    assert abs(lse[0, 0, 0] - g["lse"][0]) < 1e-13
    p, _, _ = oracle.softmax_rows(oracle.scores(q[0, 0], k[0, 0], 1.0))
    np.testing.assert_allclose(p[0], g["p"], atol=1e-15)


def test_softmax_rows_sum_to_one():
    s = _rand((33, 71), 1, gain=7.0)
    p, m, l = oracle.softmax_rows(s)
    assert np.all(np.abs(p.sum(axis=1) - 1.0) <= 1e-12)
    assert np.all(p >= 0)
    np.testing.assert_array_equal(m, s.max(axis=1))
    # the max element of each row has weight exp(0) / l
    np.testing.assert_allclose(p[np.arange(33), s.argmax(axis=1)], 1.0 / l, rtol=1e-14)


def test_softmax_no_overflow_with_large_scores():
    s = np.array([[1000.0, 999.0, -1000.0]])
    p, _, _ = oracle.softmax_rows(s)
    e = math.exp(-1.0)
    np.testing.assert_allclose(p[0], [1 / (1 + e), e / (1 + e), 0.0], atol=1e-15)


def test_zero_queries_give_column_mean_and_log_n():
    B, H, N, d = 2, 3, 37, 8
    q = np.zeros((B, H, N, d))
    k, v = _rand((B, H, N, d), 2), _rand((B, H, N, d), 3)
    o, lse = oracle.forward(q, k, v, 0.25)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), atol=1e-13)
    np.testing.assert_allclose(lse, np.log(N), atol=1e-13)


def test_single_key_gives_value_and_dot_product():
    B, H, d = 2, 2, 5
    q, k, v = _rand((B, H, 1, d), 4), _rand((B, H, 1, d), 5), _rand((B, H, 1, d), 6)
    scale = 0.3
    o, lse = oracle.forward(q, k, v, scale)
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse, scale * (q * k).sum(-1), atol=1e-14)


def test_scores_are_scaled_q_kt():
    q, k = _rand((3, 4), 7), _rand((5, 4), 8)
    s = oracle.scores(q, k, 0.5)
    assert s.shape == (3, 5)
    for i in range(3):
        for j in range(5):
            assert abs(s[i, j] - 0.5 * sum(q[i, c] * k[j, c] for c in range(4))) < 1e-13


def test_brute_force_python_loops():
    """Triple loops straight from the definition, on a tiny head."""
    N, M, d = 4, 6, 3
    q, k, v = _rand((N, d), 9), _rand((M, d), 10), _rand((M, 2), 11)
    scale = 1 / math.sqrt(d)
    o, lse = oracle.forward(q[None, None], k[None, None], v[None, None], scale)
    for i in range(N):
        s = [scale * sum(q[i, c] * k[j, c] for c in range(d)) for j in range(M)]
        mx = max(s)
        w = [math.exp(x - mx) for x in s]
        tot = sum(w)
        for c in range(2):
            assert abs(o[0, 0, i, c] - sum(w[j] * v[j, c] for j in range(M)) / tot) < 1e-13
        assert abs(lse[0, 0, i] - (mx + math.log(tot))) < 1e-13


# --- invariants ----------------------------------------------------------------------------------

def test_row_shift_invariance():
    """Adding c_i to every score of row i leaves O unchanged and adds c_i to LSE
    (the exp-sum factorisation behind the rescale, [P3] 兩大核心魔法)."""
    s = _rand((9, 40), 12, gain=3.0)
    v = _rand((40, 6), 13)
    c = _rand((9, 1), 14, gain=50.0)
    o1, lse1 = oracle.forward_from_scores(s, v)
    o2, lse2 = oracle.forward_from_scores(s + c, v)
    np.testing.assert_allclose(o2, o1, atol=1e-12)
    np.testing.assert_allclose(lse2, lse1 + c[:, 0], atol=1e-11)


def test_key_value_permutation_invariance():
    B, H, N, d = 1, 2, 23, 6
    q, k, v, do = (_rand((B, H, N, d), s) for s in (15, 16, 17, 18))
    perm = np.random.default_rng(19).permutation(N)
    o1, lse1 = oracle.forward(q, k, v, 0.4)
    o2, lse2 = oracle.forward(q, k[:, :, perm], v[:, :, perm], 0.4)
    np.testing.assert_allclose(o2, o1, atol=1e-13)
    np.testing.assert_allclose(lse2, lse1, atol=1e-13)
    dq1, dk1, dv1 = oracle.backward(q, k, v, do, 0.4)
    dq2, dk2, dv2 = oracle.backward(q, k[:, :, perm], v[:, :, perm], do, 0.4)
    np.testing.assert_allclose(dq2, dq1, atol=1e-12)
    np.testing.assert_allclose(dk2, dk1[:, :, perm], atol=1e-12)
    np.testing.assert_allclose(dv2, dv1[:, :, perm], atol=1e-12)


def test_query_rows_are_independent():
    B, H, N, d = 1, 1, 19, 4
    q, k, v = (_rand((B, H, N, d), s) for s in (20, 21, 22))
    o, lse = oracle.forward(q, k, v, 0.7)
    o_top, lse_top = oracle.forward(q[:, :, :5], k, v, 0.7)
    np.testing.assert_allclose(o_top, o[:, :, :5], atol=1e-14)
    np.testing.assert_allclose(lse_top, lse[:, :, :5], atol=1e-14)


# --- the block-wise online recurrence against the two-pass definition ----------------------------

@pytest.mark.parametrize("N", [1, 7, 64, 65])
@pytest.mark.parametrize("block", [1, 7, 8, None])
@pytest.mark.parametrize("normalise", [False, True])
def test_online_recurrence_matches_two_pass(N, block, normalise):
    d = 5
    bk = N if block is None else block
    q, k, v = _rand((N, d), 23, gain=3.0), _rand((N, d), 24), _rand((N, d), 25)
    o_ref, lse_ref = oracle.forward(q[None, None], k[None, None], v[None, None], 0.45)
    o, lse, tiles = oracle.online_forward(q, k, v, 0.45, block_q=8, block_k=bk, normalise_each_step=normalise)
    np.testing.assert_allclose(o, o_ref[0, 0], atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, lse_ref[0, 0], atol=1e-12, rtol=0)
    assert tiles == math.ceil(N / 8) * math.ceil(N / bk)


def test_online_recurrence_needs_the_rescale():
    """A late, larger maximum must rescale the earlier sum: dropping exp(m_old - m_new) is detectable."""
    q = np.array([[1.0]])
    k = np.array([[0.0], [5.0]])
    v = np.array([[1.0], [-1.0]])
    o, lse, _ = oracle.online_forward(q, k, v, 1.0, block_q=1, block_k=1)
    e = math.exp(-5.0)
    assert abs(o[0, 0] - (e - 1) / (e + 1)) < 1e-15
    assert abs(lse[0] - (5.0 + math.log1p(e))) < 1e-15


def test_merchant_tiling_of_the_first_page():
    g = _read_golden("page_sizes.txt")
    n, pile = int(g["merchants"][0]), int(g["pile_size"][0])
    q, k, v = _rand((n, 4), 26), _rand((n, 4), 27), _rand((n, 4), 28)
    _, _, tiles = oracle.online_forward(q, k, v, 0.5, block_q=pile, block_k=pile)
    assert tiles == g["tile_pairs"][0]
    assert pile * pile == g["cells_per_tile"][0]
    assert tiles * pile * pile == g["table_cells"][0]
    assert oracle.scores(q, k, 0.5).size == g["table_cells"][0]


def test_printed_score_matrix_sizes():
    g = _read_golden("page_sizes.txt")
    n, eb = int(g["s_n"][0]), int(g["s_elem_bytes"][0])
    assert n * n * eb == g["s_bytes"][0]
    assert round(n * n * eb / 1e6) == g["s_mb_printed"][0]
    assert int(g["stars"][0]) ** 2 == g["star_pairs"][0]
    assert int(g["long_n"][0]) ** 2 > g["long_n_scores_lower_bound"][0]


# --- library-routine pins (torch fp64 CPU: independent code) -------------------------------------

def _torch_attention(q, k, v, scale):
    s = scale * q @ k.transpose(-1, -2)
    return torch.softmax(s, dim=-1) @ v, torch.logsumexp(s, dim=-1)


def test_forward_matches_torch_fp64():
    B, H, N, d = 2, 3, 45, 16
    q, k, v = (_rand((B, H, N, d), s) for s in (29, 30, 31))
    o, lse = oracle.forward(q, k, v, 0.25)
    to, tl = _torch_attention(*(torch.from_numpy(x) for x in (q, k, v)), 0.25)
    np.testing.assert_allclose(o, to.numpy(), atol=1e-12)
    np.testing.assert_allclose(lse, tl.numpy(), atol=1e-12)


def test_backward_matches_torch_autograd():
    B, H, N, d = 2, 2, 37, 8
    q, k, v, do = (_rand((B, H, N, d), s) for s in (32, 33, 34, 35))
    dq, dk, dv = oracle.backward(q, k, v, do, 0.3)
    tq, tk, tv = (torch.from_numpy(x).requires_grad_(True) for x in (q, k, v))
    to, _ = _torch_attention(tq, tk, tv, 0.3)
    gq, gk, gv = torch.autograd.grad(to, (tq, tk, tv), torch.from_numpy(do))
    np.testing.assert_allclose(dq, gq.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, gk.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, gv.numpy(), atol=1e-11)


def test_backward_matches_finite_differences():
    N, d = 6, 3
    q, k, v, do = (_rand((1, 1, N, d), s) for s in (36, 37, 38, 39))
    scale = 0.7
    dq, dk, dv = oracle.backward(q, k, v, do, scale)

    def loss(qq, kk, vv):
        o, _ = oracle.forward(qq, kk, vv, scale)
        return float((o * do).sum())

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            fp = loss(args["q"], args["k"], args["v"])
            args[name] = xm
            fm = loss(args["q"], args["k"], args["v"])
            num[idx] = (fp - fm) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


def test_gradient_invariants():
    """sum_j dS_ij = 0 for every row, so the key-rows of dK sum to zero, and sum_j dV_j = sum_i dO_i."""
    B, H, N, d = 1, 2, 29, 7
    q, k, v, do = (_rand((B, H, N, d), s) for s in (40, 41, 42, 43))
    _, dk, dv = oracle.backward(q, k, v, do, 0.5)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), atol=1e-12)


def test_row_term_equals_do_dot_o():
    """sum_k P_ik dP_ik = dO_i . O_i, the identity the GPU backward uses to form its row term."""
    N, d = 31, 6
    q, k, v, do = (_rand((N, d), s) for s in (44, 45, 46, 47))
    p, _, _ = oracle.softmax_rows(oracle.scores(q, k, 0.6))
    o = p @ v
    dp = do @ v.T
    np.testing.assert_allclose((p * dp).sum(axis=1), (do * o).sum(axis=1), atol=1e-13)


# --- sampled-row and row-blocked forms agree with the full form -----------------------------------

def test_rows_forms_match_full():
    B, H, N, d = 2, 2, 50, 8
    q, k, v, do = (_rand((B, H, N, d), s) for s in (48, 49, 50, 51))
    rows = [np.array([0, 7, 49]), np.array([3, 4, 20])]
    krows = [np.array([1, 2, 48]), np.array([0, 30, 31])]
    o, lse = oracle.forward(q, k, v, 0.35)
    orow, lrow = oracle.forward_rows(q, k, v, 0.35, rows)
    dq, dk, dv = oracle.backward(q, k, v, do, 0.35)
    sq, sk, sv = oracle.backward_rows(q, k, v, do, 0.35, rows, krows)
    for h in range(H):
        np.testing.assert_allclose(orow[:, h], o[:, h, rows[h]], atol=1e-14)
        np.testing.assert_allclose(lrow[:, h], lse[:, h, rows[h]], atol=1e-14)
        np.testing.assert_allclose(sq[:, h], dq[:, h, rows[h]], atol=1e-13)
        np.testing.assert_allclose(sk[:, h], dk[:, h, krows[h]], atol=1e-13)
        np.testing.assert_allclose(sv[:, h], dv[:, h, krows[h]], atol=1e-13)
    # Query rows only (the pass over every row for dK, dV skipped): the same dQ rows.
    none = [np.zeros(0, dtype=np.int64)] * H
    oq, ok_, ov = oracle.backward_rows(q, k, v, do, 0.35, rows, none)
    assert ok_.shape == (B, H, 0, d) and ov.shape == (B, H, 0, d)
    for h in range(H):
        np.testing.assert_allclose(oq[:, h], dq[:, h, rows[h]], atol=1e-13)


def test_row_blocking_does_not_change_results(monkeypatch):
    B, H, N, d = 1, 1, 70, 4
    q, k, v, do = (_rand((B, H, N, d), s) for s in (52, 53, 54, 55))
    o1, l1 = oracle.forward(q, k, v, 0.5)
    g1 = oracle.backward(q, k, v, do, 0.5)
    monkeypatch.setattr(sdpa, "_ROW_BLOCK_ELEMS", 3 * N)   # three rows at a time, ragged last block
    o2, l2 = oracle.forward(q, k, v, 0.5)
    g2 = oracle.backward(q, k, v, do, 0.5)
    np.testing.assert_allclose(o2, o1, atol=1e-14)
    np.testing.assert_allclose(l2, l1, atol=1e-14)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a, b, atol=1e-13)
