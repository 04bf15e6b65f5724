"""fp64 CPU oracle for exact scaled dot-product attention (test infrastructure only).

This module is the checker, not the product.  Only the tests, the smoke check and the bench's CPU
baseline leg may import it; the CUDA path never calls it and shares no code with it.

Sources (the three web pages this build follows):
  [P1] "算珠楼的掌簿人" (hespethorn.github.io/posts/fable-flashattention/): sections 技术解读,
       核心概念回顾 and 故事中的隐喻对照 (the tables), 为什么这个故事对应 FlashAttention？
  [P2] "账房先生的奔命：Flash Attention 与内存 I/O 革命" (carrie-l.github.io/AI/2026-06-11-knowledge-20):
       §五 为什么标准 Attention 会"奔命" (the standard three-step pseudo-code), §六 Tiling + Online Softmax
       (技巧一, 技巧二 and the per-tile update rule), §七 重计算.
  [P3] the FlashAttention fable on ckw19810413.github.io (blog/2026-10-11-flashattention-fable/):
       sections 概念揭曉 (the Attention(Q,K,V) formula), 為什麼過去的 Attention 會慢？ and
       FlashAttention 的兩大核心魔法 (the softmax with max subtraction and the rescale identity).

What is computed here is the plain definition, with S and P materialised (the "standard" method of
[P2] §五 and [P3] 為什麼過去的 Attention 會慢？), because the pages state that the tiled method reaches
exactly this result ([P1] 技术解读 / 故事中的隐喻对照, [P2] §八 v1, [P3] 兩大核心魔法).  Rows are
processed in blocks of whole rows only to bound memory: each row's softmax still sees every key.
The backward formulas are not on the pages; they are the textbook gradient of that definition.

All arithmetic is numpy float64; the matrix products call numpy's matmul (a library primitive).
Inputs are float arrays [B, H, N, d]; bf16 inputs are widened exactly by the caller.
"""
from __future__ import annotations

import numpy as np

# Rows of S materialised at once: bounds the oracle's memory at long N without changing any row.
_ROW_BLOCK_ELEMS = 1 << 25


def _row_block(n_keys: int) -> int:
    return max(1, min(4096, _ROW_BLOCK_ELEMS // max(1, n_keys)))


def scores(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """S = scale * Q K^T for one head ([P2] §五 first pseudo-code step; [P3] 概念揭曉 formula)."""
    return scale * (q @ k.T)


def softmax_rows(s: np.ndarray):
    """Two-pass softmax of each row with the row maximum subtracted ([P2] §六 技巧二 classic softmax;
    [P3] 兩大核心魔法: subtract the global max m = max(x), then divide by the sum).

    Returns (P, m, l) with m the row max and l = sum_j exp(s_j - m)."""
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=-1, keepdims=True)
    return e / l, m[..., 0], l[..., 0]


def forward_from_scores(s: np.ndarray, v: np.ndarray):
    """O = softmax(S) V and LSE = m + ln l for given scores of one head ([P2] §五 steps two and three).

    LSE is the single saved statistic: the pages keep the running max m and the running sum l
    ([P1] 故事中的隐喻对照 "两个数"; [P2] §六); one log-sum-exp carries both."""
    p, m, l = softmax_rows(s)
    return p @ v, m + np.log(l)


def _head_forward(q, k, v, scale, rows=None):
    qr = q if rows is None else q[rows]
    n = qr.shape[0]
    o = np.empty((n, v.shape[1]), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rb = _row_block(k.shape[0])
    for r0 in range(0, n, rb):
        s = scores(qr[r0:r0 + rb], k, scale)
        o[r0:r0 + rb], lse[r0:r0 + rb] = forward_from_scores(s, v)
    return o, lse


def forward(q, k, v, scale: float):
    """Exact attention forward for [B, H, N, d] inputs: returns O [B,H,N,d] and LSE [B,H,N] (float64).

    O = softmax(scale * Q K^T) V ([P3] 概念揭曉; [P2] §五)."""
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    B, H, N, d = q.shape
    o = np.empty((B, H, N, v.shape[-1]), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = _head_forward(q[b, h], k[b, h], v[b, h], scale)
    return o, lse


def forward_rows(q, k, v, scale: float, rows):
    """Forward for selected query rows only: ``rows[h]`` indexes the rows of head h (all b).

    Each selected row still attends to every key, so it is the full definition for that row.
    Returns O [B,H,R,d] and LSE [B,H,R]."""
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    B, H, N, d = q.shape
    R = len(rows[0])
    o = np.empty((B, H, R, v.shape[-1]), dtype=np.float64)
    lse = np.empty((B, H, R), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = _head_forward(q[b, h], k[b, h], v[b, h], scale, np.asarray(rows[h]))
    return o, lse


def _head_backward(q, k, v, do, scale):
    """Textbook gradient of O = softmax(scale Q K^T) V for one head, contracted with dO.

    dV = P^T dO;  dP = dO V^T;  dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik);  dQ = scale dS K;  dK = scale dS^T Q.
    The row term sum_k P_ik dP_ik is formed directly from P and dP.  P is recomputed from Q and K here,
    the recomputation of [P2] §七."""
    N = q.shape[0]
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    rb = _row_block(k.shape[0])
    for r0 in range(0, N, rb):
        sl = slice(r0, r0 + rb)
        p, _, _ = softmax_rows(scores(q[sl], k, scale))
        dv += p.T @ do[sl]
        dp = do[sl] @ v.T
        row = (p * dp).sum(axis=-1, keepdims=True)
        ds = p * (dp - row)
        dq[sl] = scale * (ds @ k)
        dk += scale * (ds.T @ q[sl])
    return dq, dk, dv


def backward(q, k, v, do, scale: float):
    """dQ, dK, dV [B,H,N,d] (float64) of exact attention for upstream gradient dO."""
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    B, H = q.shape[:2]
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = _head_backward(q[b, h], k[b, h], v[b, h], do[b, h], scale)
    return dq, dk, dv


def backward_rows(q, k, v, do, scale: float, q_rows, k_rows):
    """Gradients at selected rows: dQ at query rows ``q_rows[h]``, dK and dV at key rows ``k_rows[h]``.

    dQ_i needs row i of P and dP.  dK_j and dV_j need column j of P and dS, hence every row's softmax
    statistics (m_i, l_i) and row term, which are formed from the full rows first (a pass over every row
    that is skipped when no key rows are asked for).
    Returns dq [B,H,Rq,d], dk [B,H,Rk,d], dv [B,H,Rk,d]."""
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    B, H, N, d = q.shape
    Rq, Rk = len(q_rows[0]), len(k_rows[0])
    dq = np.empty((B, H, Rq, d))
    dk = np.empty((B, H, Rk, d))
    dv = np.empty((B, H, Rk, v.shape[-1]))
    for b in range(B):
        for h in range(H):
            qh, kh, vh, doh = q[b, h], k[b, h], v[b, h], do[b, h]
            qi, kj = np.asarray(q_rows[h]), np.asarray(k_rows[h])
            rb = _row_block(N)
            dk_acc = np.zeros((Rk, d))
            dv_acc = np.zeros((Rk, vh.shape[1]))
            for r0 in range(0, N if Rk else 0, rb):
                sl = slice(r0, r0 + rb)
                p, _, _ = softmax_rows(scores(qh[sl], kh, scale))
                dp = doh[sl] @ vh.T
                row = (p * dp).sum(axis=-1, keepdims=True)
                ds = p * (dp - row)
                dv_acc += p[:, kj].T @ doh[sl]
                dk_acc += scale * (ds[:, kj].T @ qh[sl])
            dk[b, h], dv[b, h] = dk_acc, dv_acc
            p, _, _ = softmax_rows(scores(qh[qi], kh, scale))
            dp = doh[qi] @ vh.T
            ds = p * (dp - (p * dp).sum(axis=-1, keepdims=True))
            dq[b, h] = scale * (ds @ kh)
    return dq, dk, dv


def online_forward(q, k, v, scale: float, block_q: int, block_k: int, normalise_each_step: bool = False):
    """Block-wise online-softmax attention for one head ([N, d] arrays), in the pages' order.

    Q is cut into blocks Q_i and K, V into blocks K_j, V_j ([P2] §六 技巧一).  For each Q_i the state
    is the running max m, the running exp-sum l and the output accumulator ([P2] §六 技巧二;
    [P3] 兩大核心魔法).  For each new block j:
        S_ij  = scale * Q_i K_j^T
        m_new = max(m_old, rowmax(S_ij))
        l_new = exp(m_old - m_new) * l_old + rowsum(exp(S_ij - m_new))
    and the accumulator takes one of two forms:
      * unnormalised ([P3] 兩大核心魔法: the previously accumulated unnormalised output is multiplied by
        exp(m_old - m_new)):  A_new = exp(m_old - m_new) * A_old + exp(S_ij - m_new) V_j, and O = A / l
        after the last block;
      * normalised each step ([P2] §六 update rule, printed as a simplified form):
        O_new = exp(m_old - m_new) * O_old * l_old / l_new + exp(S_ij - m_new) V_j / l_new.
    The initial state is m = -inf, l = 0, accumulator 0; exp(m_old - m_new) is taken as 0 while m_old
    is still -inf.  Returns (O, LSE, tiles) where tiles counts the (Q_i, K_j) pairs visited.
    Pure Python loops over blocks: for small inputs only."""
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    N, Nk = q.shape[0], k.shape[0]
    o = np.empty((N, v.shape[1]))
    lse = np.empty((N,))
    tiles = 0
    for i0 in range(0, N, block_q):
        qi = q[i0:i0 + block_q]
        r = qi.shape[0]
        m = np.full((r,), -np.inf)
        l = np.zeros((r,))
        acc = np.zeros((r, v.shape[1]))
        for j0 in range(0, Nk, block_k):
            tiles += 1
            s = scale * (qi @ k[j0:j0 + block_k].T)
            m_new = np.maximum(m, s.max(axis=1))
            alpha = np.where(np.isneginf(m), 0.0, np.exp(m - m_new))
            e = np.exp(s - m_new[:, None])
            l_new = alpha * l + e.sum(axis=1)
            pv = e @ v[j0:j0 + block_k]
            if normalise_each_step:
                acc = (alpha * l / l_new)[:, None] * acc + pv / l_new[:, None]
            else:
                acc = alpha[:, None] * acc + pv
            m, l = m_new, l_new
        o[i0:i0 + r] = acc if normalise_each_step else acc / l[:, None]
        lse[i0:i0 + r] = m + np.log(l)
    return o, lse, tiles
