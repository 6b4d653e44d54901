"""Pins of the GAU projection oracle (oracle/gau.py) against closed forms,
brute-force loops and the page's layer equation."""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
from oracle import gau
from tests import brute


def test_silu_closed_form_values():
    # sigmoid(0) = 1/2, sigmoid(1) = e/(1+e), sigmoid(-1) = 1/(1+e)
    x = np.array([0.0, 1.0, -1.0, 40.0, -40.0, 2.0])
    want = np.array([0.0, math.e / (1 + math.e), -1.0 / (1 + math.e), 40.0, -40.0 * math.exp(-40.0) /
                     (1 + math.exp(-40.0)), 2.0 * math.exp(2.0) / (1 + math.exp(2.0))])
    np.testing.assert_allclose(gau.silu(x), want, rtol=1e-14, atol=1e-300)


def test_projection_matches_brute_force_loops():
    rng = np.random.default_rng(0)
    M, d, e, s = 5, 7, 3, 2
    X = rng.standard_normal((M, d))
    Wt = rng.standard_normal((2 * e + s, d))
    U, V, Z = gau.gau_project(X, Wt, e, s)
    for m in range(M):
        for j in range(2 * e + s):
            h = 0.0
            for k in range(d):
                h += X[m, k] * Wt[j, k]
            val = h * (1.0 / (1.0 + math.exp(-h)))
            got = U[m, j] if j < e else (V[m, j - e] if j < 2 * e else Z[m, j - 2 * e])
            assert abs(got - val) <= 1e-12 * max(1.0, abs(val))


def test_identity_weights_give_silu_of_the_input():
    rng = np.random.default_rng(1)
    d = e = 4
    s = 2
    X = rng.standard_normal((6, d))
    Wt = np.concatenate([np.eye(d), 2 * np.eye(d), np.eye(d)[:s]])
    U, V, Z = gau.gau_project(X, Wt, e, s)
    np.testing.assert_allclose(U, gau.silu(X), rtol=1e-15)
    np.testing.assert_allclose(V, gau.silu(2 * X), rtol=1e-15)
    np.testing.assert_allclose(Z, gau.silu(X[:, :s]), rtol=1e-15)


def test_output_projection_matches_loops():
    rng = np.random.default_rng(2)
    Y = rng.standard_normal((3, 5))
    Wo_t = rng.standard_normal((4, 5))
    got = gau.gau_output(Y, Wo_t)
    for m in range(3):
        for j in range(4):
            assert abs(got[m, j] - sum(Y[m, k] * Wo_t[j, k] for k in range(5))) <= 1e-12


@pytest.mark.parametrize("causal", [True, False])
def test_gau_layer_is_the_mix_equation(causal):
    """Projections -> core -> output projection equals (U * A V) W_o with the
    explicit mixing matrix A ("Strong Combination", eq. mix)."""
    rng = np.random.default_rng(3)
    n, d, e, s, C = 8, 6, 4, 3, 4
    X = rng.standard_normal((n, d))
    Wt = 0.5 * rng.standard_normal((2 * e + s, d))
    Wo_t = rng.standard_normal((d, e))
    gamma = 1 + 0.2 * rng.standard_normal((4, s))
    beta = 0.2 * rng.standard_normal((4, s))
    U, V, Z = gau.gau_project(X, Wt, e, s)
    core = oracle.forward(Z[None], V[None], U[None], gamma, beta, C, causal)[0]
    got = gau.gau_output(core, Wo_t)
    want = brute.explicit_matrix(Z[None], V[None], U[None], gamma, beta, C, causal)[0] @ Wo_t.T
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
