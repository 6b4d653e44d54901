"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: every check is a hand-worked
example, an independent formulation (``tests/brute.py``), an identity or an
invariant.  ``test_pins_catch_planted_mistakes`` plants plausible mistakes in a
copy of the oracle source and checks that the pins fail for each of them.
"""
from __future__ import annotations

import json
import os
import re
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from tests import brute

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def rand_inputs(B, n, s, e, seed, beta_scale=0.3):
    rng = np.random.default_rng(seed)
    Z = rng.standard_normal((B, n, s))
    V = rng.standard_normal((B, n, e))
    U = rng.standard_normal((B, n, e))
    gamma = 1.0 + 0.3 * rng.standard_normal((4, s))
    beta = beta_scale * rng.standard_normal((4, s))
    return Z, V, U, gamma, beta


def close(a, b, rtol=1e-12):
    scale = max(np.max(np.abs(b)), 1e-300)
    return np.max(np.abs(a - b)) / scale <= rtol


# --------------------------------------------------------------------------
# hand-worked examples (tests/golden/hand_examples.json)
# --------------------------------------------------------------------------
with open(os.path.join(HERE, "golden", "hand_examples.json")) as f:
    GOLDEN = json.load(f)["cases"]


@pytest.mark.parametrize("case", GOLDEN, ids=[c["name"] for c in GOLDEN])
@pytest.mark.parametrize("causal", [True, False])
def test_hand_examples(case, causal):
    args = [np.array(case[k], dtype=np.float64) for k in ("Z", "V", "U", "gamma", "beta")]
    got = oracle.forward(*args, C=case["C"], causal=causal)
    want = np.array(case["O_causal" if causal else "O_noncausal"])
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# the whole op against one explicit n x n mixing matrix
# --------------------------------------------------------------------------
@pytest.mark.parametrize("B,n,C,s,e", [(1, 8, 4, 3, 5), (2, 12, 3, 4, 2), (1, 16, 16, 5, 7),
                                       (2, 20, 5, 6, 3), (1, 9, 1, 2, 4)])
@pytest.mark.parametrize("causal", [True, False])
def test_explicit_matrix(B, n, C, s, e, causal):
    args = rand_inputs(B, n, s, e, seed=n * 31 + C)
    got = oracle.forward(*args, C=C, causal=causal)
    want = brute.explicit_matrix(*args, C=C, causal=causal)
    assert close(got, want)


# --------------------------------------------------------------------------
# C = n: the core is full relu^2 attention (FLASH-Quad) plus, non-causal,
# full linear attention; causal with one chunk has no global term at all
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [True, False])
def test_single_chunk_is_full_relu2_attention(causal):
    n, s, e = 24, 6, 5
    Z, V, U, gamma, beta = rand_inputs(1, n, s, e, seed=7)
    U = np.ones_like(U)
    got = oracle.forward(Z, V, U, gamma, beta, C=n, causal=causal)[0]
    T = [brute.affine(Z, gamma, beta, k)[0] for k in range(4)]
    want = brute.full_relu2_attention(T[0], T[1], V[0], causal)
    if not causal:
        want = want + brute.linear_attention_q_ktv(T[2], T[3], V[0])
    assert close(got, want)


# --------------------------------------------------------------------------
# global term alone (quad switched off by gamma_0 = beta_0 = 0, so relu(0) = 0)
# --------------------------------------------------------------------------
def _global_only(B, n, s, e, seed):
    Z, V, U, gamma, beta = rand_inputs(B, n, s, e, seed)
    gamma[0] = 0.0
    beta[0] = 0.0
    U = np.ones_like(U)
    return Z, V, U, gamma, beta


def test_noncausal_global_is_linear_attention_both_orders():
    n, C, s, e = 24, 6, 4, 7
    Z, V, U, gamma, beta = _global_only(2, n, s, e, seed=11)
    got = oracle.forward(Z, V, U, gamma, beta, C=C, causal=False)
    for b in range(2):
        Q = brute.affine(Z, gamma, beta, 2)[b]
        K = brute.affine(Z, gamma, beta, 3)[b]
        assert close(got[b], brute.linear_attention_q_ktv(Q, K, V[b]))
        assert close(got[b], brute.linear_attention_qkt_v(Q, K, V[b]))


def test_causal_global_is_token_recurrence_read_at_chunk_starts():
    n, C, s, e = 32, 8, 5, 3
    Z, V, U, gamma, beta = _global_only(2, n, s, e, seed=12)
    got = oracle.forward(Z, V, U, gamma, beta, C=C, causal=True)
    for b in range(2):
        Q = brute.affine(Z, gamma, beta, 2)[b]
        K = brute.affine(Z, gamma, beta, 3)[b]
        assert close(got[b], brute.rnn_global_term(Q, K, V[b], C))


def test_causal_first_chunk_has_no_global_term():
    n, C, s, e = 16, 4, 3, 4
    Z, V, U, gamma, beta = _global_only(1, n, s, e, seed=13)
    got = oracle.forward(Z, V, U, gamma, beta, C=C, causal=True)
    assert np.all(got[0, :C] == 0.0)
    assert np.max(np.abs(got[0, C:])) > 0.0


# --------------------------------------------------------------------------
# invariants and special cases
# --------------------------------------------------------------------------
def test_causality_future_tokens_do_not_matter():
    B, n, C, s, e = 1, 24, 6, 4, 5
    Z, V, U, gamma, beta = rand_inputs(B, n, s, e, seed=14)
    base = oracle.forward(Z, V, U, gamma, beta, C=C, causal=True)
    for p in (1, 5, 6, 13, 23):  # inside a chunk and at chunk starts
        Z2, V2, U2 = Z.copy(), V.copy(), U.copy()
        Z2[:, p:] += 1.7
        V2[:, p:] -= 2.3
        U2[:, p:] *= -1.0
        pert = oracle.forward(Z2, V2, U2, gamma, beta, C=C, causal=True)
        assert np.array_equal(pert[:, :p], base[:, :p])
        assert not np.allclose(pert[:, p:], base[:, p:])


def test_gate_of_ones_gives_attention_alone_and_gate_is_elementwise():
    B, n, C, s, e = 1, 12, 4, 3, 4
    Z, V, U, gamma, beta = rand_inputs(B, n, s, e, seed=15)
    att = oracle.forward(Z, V, np.ones_like(U), gamma, beta, C=C, causal=True)
    got = oracle.forward(Z, V, U, gamma, beta, C=C, causal=True)
    assert close(got, U * att)


def test_zero_affine_maps_give_zero():
    Z, V, U, gamma, beta = rand_inputs(1, 12, 3, 4, seed=16)
    got = oracle.forward(Z, V, U, np.zeros_like(gamma), np.zeros_like(beta), C=4, causal=False)
    assert np.all(got == 0.0)


def test_linear_in_v():
    Z, V, U, gamma, beta = rand_inputs(2, 12, 3, 4, seed=17)
    a = oracle.forward(Z, V, U, gamma, beta, C=3, causal=True)
    b = oracle.forward(Z, 2.5 * V, U, gamma, beta, C=3, causal=True)
    assert close(b, 2.5 * a)


def test_z_scaling_degrees_quad_four_global_two():
    """With beta = 0: scaling Z by alpha scales relu(q.k/C)^2 by alpha^4 and
    the global term q.(k^T v)/n by alpha^2 (alpha > 0)."""
    B, n, C, s, e = 1, 16, 4, 3, 5
    Z, V, U, gamma, beta = rand_inputs(B, n, s, e, seed=18)
    beta = np.zeros_like(beta)
    g_quad = gamma.copy(); g_quad[2] = 0.0          # global off
    g_lin = gamma.copy(); g_lin[0] = 0.0            # quad off
    alpha = 1.7
    for causal in (True, False):
        q1 = oracle.forward(Z, V, U, g_quad, beta, C=C, causal=causal)
        q2 = oracle.forward(alpha * Z, V, U, g_quad, beta, C=C, causal=causal)
        assert close(q2, alpha ** 4 * q1, rtol=1e-11)
        l1 = oracle.forward(Z, V, U, g_lin, beta, C=C, causal=causal)
        l2 = oracle.forward(alpha * Z, V, U, g_lin, beta, C=C, causal=causal)
        assert close(l2, alpha ** 2 * l1, rtol=1e-11)
        # and the two parts add up to the whole
        whole = oracle.forward(Z, V, U, gamma, beta, C=C, causal=causal)
        assert close(whole, q1 + l1)


def test_noncausal_chunk_permutation_permutes_output():
    B, n, C, s, e = 1, 20, 4, 3, 4
    Z, V, U, gamma, beta = rand_inputs(B, n, s, e, seed=19)
    base = oracle.forward(Z, V, U, gamma, beta, C=C, causal=False)
    perm = np.array([3, 0, 4, 1, 2])
    idx = (perm[:, None] * C + np.arange(C)[None, :]).reshape(-1)
    got = oracle.forward(Z[:, idx], V[:, idx], U[:, idx], gamma, beta, C=C, causal=False)
    assert close(got, base[:, idx])


def test_batch_elements_are_independent():
    Z, V, U, gamma, beta = rand_inputs(3, 12, 3, 4, seed=20)
    whole = oracle.forward(Z, V, U, gamma, beta, C=4, causal=True)
    for b in range(3):
        one = oracle.forward(Z[b:b + 1], V[b:b + 1], U[b:b + 1], gamma, beta, C=4, causal=True)
        assert np.array_equal(one[0], whole[b])


def test_rows_entry_matches_the_explicit_matrix():
    B, n, C, s, e = 2, 24, 6, 4, 3
    args = rand_inputs(B, n, s, e, seed=21)
    ids = np.array([0, 5, 6, 23, 24, 29, 30, 47])
    for causal in (True, False):
        want = brute.explicit_matrix(*args, C=C, causal=causal).reshape(B * n, e)[ids]
        got = oracle.rows(*args, C=C, causal=causal, row_ids=ids)
        assert close(got, want)


def test_rejects_bad_arguments():
    Z, V, U, gamma, beta = rand_inputs(1, 12, 3, 4, seed=22)
    with pytest.raises(ValueError):
        oracle.forward(Z, V, U, gamma, beta, C=5, causal=True)   # C does not divide n
    with pytest.raises(ValueError):
        oracle.forward(Z, V, U, gamma, beta, C=24, causal=True)  # C > n
    with pytest.raises(ValueError):
        oracle.rows(Z, V, U, gamma, beta, C=4, causal=True, row_ids=[12])  # out of range


# --------------------------------------------------------------------------
# the pins are sharp: plausible mistakes planted in a copy of the oracle fail
# --------------------------------------------------------------------------
MUTATIONS = {
    "inclusive_prefix": ("int hend = causal ? g : G;", "int hend = causal ? g + 1 : G;"),
    "no_chunk_scale": ("relu(dot(q0, k1, s) / (double)C)", "relu(dot(q0, k1, s))"),
    "sqrt_style_scale": ("double w = r * r;", "double w = r;"),
    "mask_diagonal": ("int jmax = causal ? i : C - 1;", "int jmax = causal ? i - 1 : C - 1;"),
    "global_normaliser_C": ("double qa = q2[a] / (double)n;", "double qa = q2[a] / (double)C;"),
    "wrong_affine_row": ("affine_row(Z, gamma, beta, s, row, 2, q2);",
                         "affine_row(Z, gamma, beta, s, row, 3, q2);"),
    "drop_gate": ("for (int c = 0; c < e; ++c) out[c] *= u[c];", ""),
    "drop_beta": ("out[c] = z[c] * gamma[k * s + c] + beta[k * s + c];",
                  "out[c] = z[c] * gamma[k * s + c];"),
}


def _pin_suite_fails(lib_path):
    """Run a compact set of pins against a compiled oracle variant; return
    True when at least one pin fails."""
    import ctypes
    lib = ctypes.CDLL(lib_path)
    d = ctypes.POINTER(ctypes.c_double)
    i = ctypes.c_int
    lib.mca_oracle_forward.argtypes = [d, d, d, d, d, d, i, i, i, i, i, i, i]
    lib.mca_oracle_forward.restype = i

    def fwd(Z, V, U, gamma, beta, C, causal):
        Z, V, U, gamma, beta = (np.ascontiguousarray(a, dtype=np.float64) for a in (Z, V, U, gamma, beta))
        B, n, s = Z.shape
        e = V.shape[2]
        O = np.zeros((B, n, e))
        p = lambda a: a.ctypes.data_as(d)
        lib.mca_oracle_forward(p(Z), p(V), p(U), p(gamma), p(beta), p(O), B, n, s, e, C, int(causal), 1)
        return O

    for case in GOLDEN:
        args = [np.array(case[k], dtype=np.float64) for k in ("Z", "V", "U", "gamma", "beta")]
        for causal in (True, False):
            want = np.array(case["O_causal" if causal else "O_noncausal"])
            if not np.allclose(fwd(*args, case["C"], causal), want, rtol=0, atol=1e-12):
                return True
    for causal in (True, False):
        args = rand_inputs(2, 12, 3, 5, seed=99)
        if not close(fwd(*args, 4, causal), brute.explicit_matrix(*args, C=4, causal=causal)):
            return True
    return False


def test_pins_catch_planted_mistakes(tmp_path):
    src = open(os.path.join(ROOT, "oracle", "mca_oracle.c")).read()
    # the unmodified source passes the compact suite
    variants = {"unmodified": src}
    for name, (old, new) in MUTATIONS.items():
        assert src.count(old) >= 1, f"mutation anchor for {name} not found"
        variants[name] = src.replace(old, new)
    for name, text in variants.items():
        c = tmp_path / f"{name}.c"
        so = tmp_path / f"{name}.so"
        c.write_text(text)
        subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(c)],
                       check=True)
        failed = _pin_suite_fails(str(so))
        if name == "unmodified":
            assert not failed, "the pins must pass on the real oracle"
        else:
            assert failed, f"planted mistake '{name}' was not caught by the pins"
