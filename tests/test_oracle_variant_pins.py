"""Pins of the oracle's scale and normalisation variants.

"FLASH: Possibly the Most Interesting Efficient Transformer Design Recently",
section "Mixed Chunk", writes the intra-chunk term as 1/(cs) relu^2(Q K^T) V and
divides the decoder's global term by the number of tokens in the earlier chunks;
section "Extended Thoughts" says the decoder's running sum of the first t items
should be divided by t.  The oracle offers these as ``quad_scale`` and
``lin_norm``.  Each check below pins them to something other than the oracle:
hand-worked values (tests/golden/hand_variants.json), the explicit n x n matrix
of tests/brute.py, the token recurrence, or identities between the variants.
"""
from __future__ import annotations

import json
import os

import numpy as np
import pytest

import oracle
from tests import brute
from tests.test_oracle_pins import close, rand_inputs

HERE = os.path.dirname(os.path.abspath(__file__))
with open(os.path.join(HERE, "golden", "hand_variants.json")) as f:
    GOLDEN = json.load(f)["cases"]

N, SUMMED, POSITION = oracle.LIN_NORM_N, oracle.LIN_NORM_SUMMED, oracle.LIN_NORM_POSITION


@pytest.mark.parametrize("case", GOLDEN, ids=[c["name"] for c in GOLDEN])
@pytest.mark.parametrize("causal", [True, False])
def test_hand_examples(case, causal):
    args = [np.array(case[k], dtype=np.float64) for k in ("Z", "V", "U", "gamma", "beta")]
    got = oracle.forward(*args, C=case["C"], causal=causal, quad_scale=case["quad_scale"],
                         lin_norm=case["lin_norm"])
    want = np.array(case["O_causal" if causal else "O_noncausal"])
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("B,n,C,s,e", [(1, 8, 4, 3, 5), (2, 12, 3, 4, 2), (1, 16, 16, 5, 7),
                                       (2, 20, 5, 6, 3), (1, 9, 1, 2, 4)])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("variant", [("cs", N), (None, SUMMED), (None, POSITION),
                                     ("cs", SUMMED), (0.37, POSITION)])
def test_explicit_matrix(B, n, C, s, e, causal, variant):
    qs, ln = variant
    quad_scale = 1.0 / (C * s) if qs == "cs" else qs
    args = rand_inputs(B, n, s, e, seed=31 * n + C + 7 * ln)
    got = oracle.forward(*args, C=C, causal=causal, quad_scale=quad_scale, lin_norm=ln)
    want = brute.explicit_matrix(*args, C=C, causal=causal, quad_scale=quad_scale, lin_norm=ln)
    assert close(got, want)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("ln", [N, SUMMED, POSITION])
def test_rows_entry_matches_the_explicit_matrix(causal, ln):
    B, n, C, s, e = 2, 12, 4, 3, 5
    args = rand_inputs(B, n, s, e, seed=5 + ln)
    ids = np.array([0, 3, 5, 11, 12, 17, 23])
    got = oracle.rows(*args, C=C, causal=causal, row_ids=ids, quad_scale=0.2, lin_norm=ln)
    want = brute.explicit_matrix(*args, C=C, causal=causal, quad_scale=0.2,
                                 lin_norm=ln).reshape(B * n, e)[ids]
    assert close(got, want)


@pytest.mark.parametrize("causal", [True, False])
def test_default_arguments_reduce_to_the_plain_definition(causal):
    """quad_scale = 1/C^2 with divisor n is the definition the plain entry
    point computes: relu(x/C)^2 = relu(x)^2 / C^2."""
    args = rand_inputs(2, 24, 4, 6, seed=3)
    plain = oracle.forward(*args, C=6, causal=causal)
    variant = oracle.forward(*args, C=6, causal=causal, quad_scale=1.0 / 36.0, lin_norm=N)
    assert close(variant, plain, rtol=1e-13)


def test_summed_divisor_is_n_without_a_mask():
    """Bidirectional: every token's global sum covers all n tokens."""
    args = rand_inputs(2, 20, 3, 4, seed=8)
    a = oracle.forward(*args, C=5, causal=False, lin_norm=SUMMED)
    b = oracle.forward(*args, C=5, causal=False, lin_norm=N)
    assert close(a, b, rtol=1e-14)


def test_quad_scale_is_linear_in_the_intra_chunk_term():
    """With lin_q = 0 only the intra-chunk term remains, and it scales with
    quad_scale."""
    Z, V, U, gamma, beta = rand_inputs(1, 16, 4, 3, seed=4)
    gamma[2] = 0.0
    beta[2] = 0.0
    a = oracle.forward(Z, V, U, gamma, beta, C=4, causal=True, quad_scale=0.1)
    b = oracle.forward(Z, V, U, gamma, beta, C=4, causal=True, quad_scale=0.7)
    assert close(7.0 * a, b)
    assert np.max(np.abs(a)) > 0


@pytest.mark.parametrize("ln", [SUMMED, POSITION])
def test_causal_global_term_is_the_normalised_token_recurrence(ln):
    """Causal global term of token t = T2[t] . S / d with S the token
    recurrence S_u = S_{u-1} + T3[u]^T V[u] read at the start of t's chunk, and
    d its token count g*C (SUMMED) or t+1 (POSITION).  Isolated with U = 1 and
    quad_q = 0 (no intra-chunk term)."""
    B, n, C, s, e = 1, 12, 3, 4, 2
    Z, V, U, gamma, beta = rand_inputs(B, n, s, e, seed=11)
    U = np.ones_like(U)
    gamma[0] = 0.0
    beta[0] = 0.0
    got = oracle.forward(Z, V, U, gamma, beta, C=C, causal=True, lin_norm=ln)[0]
    T2 = Z[0] * gamma[2] + beta[2]
    T3 = Z[0] * gamma[3] + beta[3]
    S = np.zeros((s, e))
    want = np.zeros((n, e))
    chunk_start_state = np.zeros((s, e))
    for t in range(n):
        if t % C == 0:
            chunk_start_state = S.copy()
        g = t // C
        d = (g * C) if ln == SUMMED else (t + 1)
        want[t] = 0.0 if g == 0 else T2[t] @ chunk_start_state / d
        S = S + np.outer(T3[t], V[0, t])
    assert close(got, want)


def test_chunk_zero_of_the_summed_divisor_has_no_global_term():
    Z, V, U, gamma, beta = rand_inputs(1, 8, 3, 2, seed=2)
    gamma[0] = 0.0
    beta[0] = 0.0  # no intra-chunk term
    O = oracle.forward(Z, V, U, gamma, beta, C=4, causal=True, lin_norm=SUMMED)
    assert np.all(O[0, :4] == 0.0)
    assert np.max(np.abs(O[0, 4:])) > 0


def test_bad_variant_arguments_are_rejected():
    args = rand_inputs(1, 4, 2, 2, seed=1)
    for kw in ({"quad_scale": -1.0}, {"quad_scale": float("nan")}, {"quad_scale": float("inf")},
               {"lin_norm": 4}, {"lin_norm": -1}):
        with pytest.raises(ValueError):
            oracle.forward(*args, C=2, causal=True, **kw)


# --------------------------------------------------------------------------
# the pins above catch plausible mistakes in the variant code
# --------------------------------------------------------------------------
MUTATIONS = {
    "summed_counts_its_own_chunk": (
        "return g > 0 ? 1.0 / ((double)g * (double)C) : 0.0;",
        "return g > 0 ? 1.0 / ((double)(g + 1) * (double)C) : 0.0;"),
    "position_counted_from_zero": (
        "if (lin_norm == 2) return 1.0 / ((double)g * (double)C + (double)i + 1.0);",
        "if (lin_norm == 2) return 1.0 / ((double)g * (double)C + (double)i + 2.0);"),
    "relu_not_squared": ("double w = quad_scale * r * r;", "double w = quad_scale * r;"),
    "summed_bidirectional_divides_by_C": (
        "    if (!causal) return 1.0 / (double)n;", "    if (!causal) return 1.0 / (double)C;"),
    "variant_ignores_lin_norm": (
        "  double f = lin_factor(lin_norm, causal, n, C, g, i);",
        "  double f = 1.0 / (double)n;"),
}


def _variant_suite_fails(lib_path: str) -> bool:
    import ctypes
    lib = ctypes.CDLL(lib_path)
    d = ctypes.POINTER(ctypes.c_double)
    i = ctypes.c_int
    lib.mca_oracle_forward_ex.argtypes = [d, d, d, d, d, d, i, i, i, i, i, i, ctypes.c_double, i, i]
    lib.mca_oracle_forward_ex.restype = i

    def fwd(Z, V, U, gamma, beta, C, causal, qs, ln):
        Z, V, U, gamma, beta = (np.ascontiguousarray(a, dtype=np.float64) for a in (Z, V, U, gamma, beta))
        B, n, s = Z.shape
        e = V.shape[2]
        O = np.zeros((B, n, e))
        p = lambda a: a.ctypes.data_as(d)
        lib.mca_oracle_forward_ex(p(Z), p(V), p(U), p(gamma), p(beta), p(O), B, n, s, e, C,
                                  int(causal), qs, ln, 1)
        return O

    for case in GOLDEN:
        args = [np.array(case[k], dtype=np.float64) for k in ("Z", "V", "U", "gamma", "beta")]
        for causal in (True, False):
            want = np.array(case["O_causal" if causal else "O_noncausal"])
            got = fwd(*args, case["C"], causal, case["quad_scale"], case["lin_norm"])
            if not np.allclose(got, want, rtol=0, atol=1e-12):
                return True
    for causal in (True, False):
        for ln in (N, SUMMED, POSITION):
            args = rand_inputs(2, 12, 3, 5, seed=90 + ln)
            want = brute.explicit_matrix(*args, C=4, causal=causal, quad_scale=0.3, lin_norm=ln)
            if not close(fwd(*args, 4, causal, 0.3, ln), want):
                return True
    return False


def test_pins_catch_planted_mistakes_in_the_variants(tmp_path):
    import subprocess
    src = open(os.path.join(HERE, "..", "oracle", "mca_oracle.c")).read()
    variants = {"unmodified": src}
    for name, (old, new) in MUTATIONS.items():
        assert src.count(old) == 1, f"mutation anchor for {name} not found once"
        variants[name] = src.replace(old, new)
    for name, text in variants.items():
        c = tmp_path / f"{name}.c"
        so = tmp_path / f"{name}.so"
        c.write_text(text)
        subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(c), "-lm"],
                       check=True)
        failed = _variant_suite_fails(str(so))
        if name == "unmodified":
            assert not failed, "the pins must pass on the real oracle"
        else:
            assert failed, f"planted mistake '{name}' was not caught by the pins"


# --------------------------------------------------------------------------
# no global term: with C = n, the quadratic-only model (FLASH-Quad)
# --------------------------------------------------------------------------
NONE = oracle.LIN_NORM_NONE


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("n,s,e", [(16, 4, 3), (24, 5, 6)])
def test_no_global_term_with_one_chunk_is_flash_quad(causal, n, s, e):
    """"Weak Attention": O = U * relu(Q K^T / n)^2 V with Q, K affine maps of Z,
    masked for a decoder -- brute force over the whole n x n matrix, with
    lin_q and lin_k left non-zero (they must not contribute)."""
    Z, V, U, gamma, beta = rand_inputs(2, n, s, e, seed=n + s)
    got = oracle.forward(Z, V, U, gamma, beta, C=n, causal=causal, lin_norm=NONE)
    for b in range(2):
        T0 = Z[b] * gamma[0] + beta[0]
        T1 = Z[b] * gamma[1] + beta[1]
        want = U[b] * brute.full_relu2_attention(T0, T1, V[b], causal)
        assert close(got[b], want)


@pytest.mark.parametrize("causal", [True, False])
def test_no_global_term_equals_zero_lin_maps(causal):
    """Dropping the global term equals zeroing lin_q's affine map (T2 = 0)."""
    Z, V, U, gamma, beta = rand_inputs(1, 20, 3, 4, seed=6)
    a = oracle.forward(Z, V, U, gamma, beta, C=5, causal=causal, lin_norm=NONE)
    g2, b2 = gamma.copy(), beta.copy()
    g2[2] = 0.0
    b2[2] = 0.0
    b = oracle.forward(Z, V, U, g2, b2, C=5, causal=causal)
    assert close(a, b, rtol=1e-14)
    assert np.max(np.abs(a - oracle.forward(Z, V, U, gamma, beta, C=5, causal=causal))) > 0
