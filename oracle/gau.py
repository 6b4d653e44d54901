"""fp64 CPU oracle of the GAU projections around the attention core.

TEST INFRASTRUCTURE ONLY (as the rest of ``oracle/``).

"FLASH: Possibly the Most Interesting Efficient Transformer Design Recently":
  section "Initial Power": U = phi(X W_u), V = phi(X W_v), with phi = Swish
  (SiLU: x * sigmoid(x)) for both in this model;
  section "Weak Attention", eq. relu-att: Z = phi(X W_z), W_z in R^{d x s};
  section "Strong Combination", eq. mix: the layer output is
  (U * A V) W_o, W_o in R^{e x d}.
No biases appear in these equations, and none are used.

Weights are passed transposed, one row per output feature: Wt = [W_u | W_v |
W_z]^T of shape [2e + s, d] and Wo_t = W_o^T of shape [d, e].
"""
from __future__ import annotations

import numpy as np


def silu(x: np.ndarray) -> np.ndarray:
    """x * sigmoid(x) = x / (1 + exp(-x))."""
    return x / (1.0 + np.exp(-x))


def gau_project(X, Wt, e: int, s: int):
    """(U, V, Z) = phi(X W_u), phi(X W_v), phi(X W_z) for X [M, d], Wt [2e+s, d]."""
    X = np.asarray(X, dtype=np.float64)
    Wt = np.asarray(Wt, dtype=np.float64)
    H = silu(X @ Wt.T)
    return H[:, :e], H[:, e:2 * e], H[:, 2 * e:2 * e + s]


def gau_output(Y, Wo_t):
    """Y W_o for Y [M, e], Wo_t = W_o^T [d, e]."""
    return np.asarray(Y, dtype=np.float64) @ np.asarray(Wo_t, dtype=np.float64).T
