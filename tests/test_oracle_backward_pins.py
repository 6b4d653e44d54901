"""Pins of the backward oracle (oracle/backward.py).

The pages define only the forward pass; the backward is its gradient.  The
backward oracle differentiates an fp64 torch restatement of the forward with
autograd.  These checks tie it to the independent C oracle (mca_oracle.c): its
forward agrees with the C forward, and every gradient entry agrees with a
central finite difference of the C forward.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import backward as obwd
from tests.test_oracle_pins import close, rand_inputs

VARIANTS = [(None, 0), (None, 1), (None, 2), (0.3, 3), (0.05, 0)]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("qs,ln", VARIANTS)
def test_torch_forward_matches_the_c_oracle(causal, qs, ln):
    args = rand_inputs(2, 12, 3, 4, seed=7 + ln)
    want = oracle.forward(*args, C=4, causal=causal, quad_scale=qs, lin_norm=ln)
    got = obwd.forward_torch(*(torch.as_tensor(a) for a in args), 4, causal, qs, ln).numpy()
    assert close(got, want)


def _fd_grad(args, idx, dO, C, causal, qs, ln, h=1e-6):
    """Central differences of sum(O * dO) w.r.t. argument `idx`, by the C oracle."""
    base = [np.array(a, dtype=np.float64) for a in args]
    x = base[idx]
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        mi = it.multi_index
        old = x[mi]
        x[mi] = old + h
        fp = np.sum(oracle.forward(*base, C=C, causal=causal, quad_scale=qs, lin_norm=ln) * dO)
        x[mi] = old - h
        fm = np.sum(oracle.forward(*base, C=C, causal=causal, quad_scale=qs, lin_norm=ln) * dO)
        x[mi] = old
        g[mi] = (fp - fm) / (2 * h)
    return g


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("qs,ln", VARIANTS)
def test_gradients_match_finite_differences_of_the_c_oracle(causal, qs, ln):
    B, n, C, s, e = 1, 6, 3, 2, 3
    args = rand_inputs(B, n, s, e, seed=30 + ln + (1 if causal else 0), beta_scale=0.5)
    dO = np.random.default_rng(ln + 5).standard_normal((B, n, e))
    grads = obwd.backward(*args, dO, C, causal, qs, ln)
    for idx, g in enumerate(grads):
        fd = _fd_grad(args, idx, dO, C, causal, qs, ln)
        # relu^2 is C^1, so central differences are accurate to O(h^2)
        assert np.max(np.abs(g - fd)) <= 1e-6 * max(1.0, np.max(np.abs(fd))), idx


def test_gate_gradient_is_the_ungated_output():
    """dU = dO * (quad + glob) = dO * O / U."""
    args = rand_inputs(1, 8, 3, 2, seed=3)
    O = oracle.forward(*args, C=4, causal=True)
    dO = np.ones_like(O)
    _, _, dU, _, _ = obwd.backward(*args, dO, 4, True)
    assert close(dU * args[2], O)


def test_no_global_term_has_no_lin_gradients():
    """Without the global term, lin_q and lin_k get no gradient."""
    args = rand_inputs(1, 8, 3, 2, seed=4)
    dO = np.random.default_rng(1).standard_normal((1, 8, 2))
    _, _, _, dg, db = obwd.backward(*args, dO, 4, True, lin_norm=3)
    assert np.all(dg[2:] == 0) and np.all(db[2:] == 0)
    assert np.max(np.abs(dg[:2])) > 0
