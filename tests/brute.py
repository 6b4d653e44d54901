"""Independent numpy fp64 formulations used to pin the oracle.

Each function computes the same quantity as the oracle by a different route
that the pages or plain algebra fix, so that a slip in the oracle's loops (a
dropped term, an inclusive instead of exclusive prefix, a wrong scale, a
transposed operand) shows up as a mismatch:

* ``explicit_matrix``: O = U * (A V) with one explicit n x n mixing matrix A
  (the GAU form O = (U * A V) W_o of "FLASH: Possibly the Most Interesting
  Efficient Transformer Design Recently", section "Strong Combination", eq. mix,
  with A assembled from the "Mixed Chunk" terms: a block-diagonal masked relu^2
  part and a low-rank part restricted to earlier chunks or to all chunks).
* ``full_relu2_attention``: the FLASH-Quad attention of section "Weak
  Attention" (appendix scale relu(x/n)^2) -- what the core reduces to when the
  chunk spans the whole sequence.
* ``linear_attention_q_ktv`` / ``linear_attention_qkt_v``: the two association
  orders of plain linear attention (same page, "Existing Methods"), which the
  non-causal global term equals ("Mixed Chunk": equivalent to linear attention
  with the full matrices).
* ``rnn_global_term``: the token-by-token recurrence S_t = S_{t-1} + k_t^T v_t
  of causal linear attention ("大模型训练之加速篇 -attention优化", section 1.4,
  first way), read at the start of each chunk.
"""
from __future__ import annotations

import numpy as np


def affine(Z, gamma, beta, k):
    return Z * gamma[k][None, None, :] + beta[k][None, None, :]


def explicit_matrix(Z, V, U, gamma, beta, C, causal, quad_scale=None, lin_norm=0):
    """O = U * (A V), A assembled entry by entry.  ``quad_scale`` (default
    1/C^2) multiplies relu(q . k)^2; ``lin_norm`` picks the divisor of the
    low-rank part per query row: 0 n, 1 the number of keys the row's global
    sum covers (its count of True entries in the low-rank mask), 2 the row's
    position counted from 1."""
    Z, V, U, gamma, beta = (np.asarray(a, dtype=np.float64) for a in (Z, V, U, gamma, beta))
    B, n, s = Z.shape
    T = [affine(Z, gamma, beta, k) for k in range(4)]
    chunk = np.arange(n) // C
    pos = np.arange(n)
    same = chunk[:, None] == chunk[None, :]
    if causal:
        quad_mask = same & (pos[None, :] <= pos[:, None])
        lin_mask = chunk[None, :] < chunk[:, None]
    else:
        quad_mask = same
        lin_mask = np.ones((n, n), dtype=bool)
    if lin_norm == 0:
        div = np.full(n, float(n))
    elif lin_norm == 1:
        div = lin_mask.sum(axis=1).astype(np.float64)  # keys each row's sum covers
    elif lin_norm == 2:
        div = pos + 1.0
    else:
        raise ValueError(lin_norm)
    inv = np.where(div > 0, 1.0 / np.maximum(div, 1.0), 0.0)
    out = np.empty_like(U)
    for b in range(B):
        raw = T[0][b] @ T[1][b].T
        if quad_scale is None:
            quad = np.maximum(raw / C, 0.0) ** 2
        else:
            quad = quad_scale * np.maximum(raw, 0.0) ** 2
        A = np.where(quad_mask, quad, 0.0)
        A = A + np.where(lin_mask, (T[2][b] @ T[3][b].T) * inv[:, None], 0.0)
        out[b] = U[b] * (A @ V[b])
    return out


def full_relu2_attention(Q, K, V, causal):
    """relu(Q K^T / n)^2 V over the whole length n, optionally lower-triangular."""
    n = Q.shape[0]
    A = np.maximum(Q @ K.T / n, 0.0) ** 2
    if causal:
        A = np.tril(A)
    return A @ V


def linear_attention_q_ktv(Q, K, V):
    return Q @ (K.T @ V) / Q.shape[0]


def linear_attention_qkt_v(Q, K, V):
    return (Q @ K.T) @ V / Q.shape[0]


def rnn_global_term(Q, K, V, C):
    """Causal chunk-level global term through the token recurrence."""
    n, s = Q.shape
    e = V.shape[1]
    S = np.zeros((s, e))
    out = np.zeros((n, e))
    for t in range(n):
        if t % C == 0:
            chunk_state = S.copy()  # state after the tokens of all earlier chunks
        out[t] = Q[t] @ chunk_state / n
        S = S + np.outer(K[t], V[t])
    return out
