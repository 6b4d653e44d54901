"""GPU parity of the tensor-core backward pass (bf16, s = 128, C % 128 == 0,
e % 256 == 0) against the fp64 backward oracle (oracle/backward.py), at the
bf16 bar of the forward pass (normwise 2e-2 per gradient).  The shapes cover
both N tiles of the score-gradient product (C % 256 == 0 and C = 128 mod 256),
several e tiles, more than one batch, single- and multi-chunk sequences, the
FLASH-Quad shape (one chunk per sequence) and every scale / divisor variant.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mca_inputs

from tests.test_gpu_backward import check, run_backward
from tests.test_gpu_parity import fm

pytestmark = pytest.mark.gpu

BF = torch.bfloat16
VARIANTS = [(None, 0), (None, 1), (None, 2), (0.1, 3), ("cs", 0), ("cs", 1)]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("variant", VARIANTS, ids=[f"{q}-{l}" for q, l in VARIANTS])
def test_tc_backward_variants(causal, variant):
    check(2, 512, 128, 128, 512, causal, BF, variant, seed=21)


@pytest.mark.parametrize("B,n,C,e,causal", [
    (1, 256, 256, 256, True),      # one chunk: no prefix, global term from nothing
    (1, 1024, 256, 768, True),
    (1, 1024, 256, 768, False),
    (3, 384, 128, 256, True),      # odd batch count, three chunks
    (1, 768, 384, 256, False),     # C = 384: N tile 128 for the score gradients
    (1, 1024, 1024, 512, True),    # FLASH-Quad: C = n
])
def test_tc_backward_shapes(B, n, C, e, causal):
    check(B, n, C, 128, e, causal, BF, (None, 0), seed=5 + n + e)


def test_tc_backward_flash_quad_no_global():
    check(2, 512, 512, 128, 256, True, BF, (None, 3), seed=8)


def test_tc_backward_is_deterministic():
    B, n, C, s, e = 1, 512, 256, 128, 256
    Z, V, U, gamma, beta = mca_inputs.make_inputs(B, n, s, e, 6, BF)
    dO = torch.randn(B, n, e, generator=torch.Generator().manual_seed(2)).to(BF)
    a = run_backward(Z, V, U, gamma, beta, dO, C, True, None, 0)
    b = run_backward(Z, V, U, gamma, beta, dO, C, True, None, 0)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("variant", [(None, 0), (None, 2), (None, 3)], ids=["n", "position", "none"])
def test_tc_backward_saved_matches_recompute(causal, variant):
    # the forward pass's intermediates kept in the workspace: the same bits as
    # the backward pass that recomputes them
    m = fm()
    dev = torch.device("cuda:0")
    B, n, C, s, e = 2, 1024, 256, 128, 512
    qs, ln = variant
    Z, V, U, gamma, beta = (t.to(dev) for t in mca_inputs.make_inputs(B, n, s, e, 12, BF))
    dO = torch.randn(B, n, e, generator=torch.Generator().manual_seed(13)).to(BF).to(dev)
    nb = m.flash_mca_backward_workspace_bytes(B, n, s, e, C, causal, m.FMCA_BF16)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    O = torch.empty_like(U)
    m.flash_mca_forward_ex(Z, V, U, gamma, beta, O, C, causal, ws, qs, ln, m.FMCA_PATH_AUTO)

    def grads(saved):
        out = (torch.empty_like(Z), torch.empty_like(V), torch.empty_like(U),
               torch.empty(4, s, device=dev), torch.empty(4, s, device=dev))
        m.flash_mca_backward(Z, V, U, gamma, beta, dO, *out, C, causal, ws, qs, ln, saved=saved)
        return out
    kept = grads(True)          # right after the forward pass: its intermediates
    torch.cuda.synchronize()
    full = grads(False)         # recomputes them (into the same workspace)
    torch.cuda.synchronize()
    for a, b in zip(kept, full):
        assert torch.equal(a, b)
    st, where = m.flash_mca_device_status()
    assert st == m.FMCA_OK, f"device status {st} at {where}"
