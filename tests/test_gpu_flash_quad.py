"""GPU parity of longer chunks on the tensor-core path and of the
quadratic-only model FLASH-Quad ("FLASH: Possibly the Most Interesting
Efficient Transformer Design Recently", section "Weak Attention": relu(q.k/n)^2
attention over the whole sequence, masked for a decoder) -- the core with one
chunk spanning the sequence (C = n) and no global term (FMCA_LIN_NORM_NONE).
Against the oracle, same bars as tests/test_gpu_parity.py.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mca_inputs
import oracle

from tests.test_gpu_parity import TOL, fm, rel_err
from tests.test_gpu_variants import run_ex

pytestmark = pytest.mark.gpu
NONE = 3


@pytest.mark.parametrize("B,n,C,s,e,causal", [
    (1, 1024, 512, 128, 256, True),    # 4 row tiles per chunk
    (1, 1024, 512, 128, 256, False),
    (1, 2048, 1024, 128, 256, True),   # 8 row tiles, 16 key stages
    (2, 1152, 384, 128, 512, True),    # C = 384: three row tiles
])
def test_longer_chunks_on_the_tensor_core_path(B, n, C, s, e, causal):
    m = fm()
    assert m.flash_mca_auto_path(B, n, s, e, C, causal, m.FMCA_BF16) == m.FMCA_PATH_TCGEN05
    Z, V, U, gamma, beta = mca_inputs.make_inputs(B, n, s, e, 60 + n + C, torch.bfloat16)
    got = run_ex(Z, V, U, gamma, beta, C, causal, None, 0, m.FMCA_PATH_TCGEN05)
    ref = oracle.forward(Z, V, U, gamma, beta, C, causal)
    err = rel_err(got, ref)
    assert err <= TOL[torch.bfloat16], f"normwise error {err:.3e}"


@pytest.mark.parametrize("B,n,s,e,causal", [
    (2, 512, 128, 256, True),
    (2, 512, 128, 256, False),
    (1, 1024, 128, 512, True),
    (1, 2048, 128, 256, True),
    (1, 1280, 128, 256, False),
    (2, 256, 128, 384, True),     # e % 256 == 128 (C = n = 256: the fused kernel)
    (2, 256, 128, 384, False),
    (2, 256, 128, 320, True),     # a 64-column last e tile
])
def test_flash_quad_tensor_core(B, n, s, e, causal):
    m = fm()
    Z, V, U, gamma, beta = mca_inputs.make_inputs(B, n, s, e, 80 + n, torch.bfloat16)
    got = run_ex(Z, V, U, gamma, beta, n, causal, None, NONE, m.FMCA_PATH_TCGEN05)
    ref = oracle.forward(Z, V, U, gamma, beta, n, causal, lin_norm=NONE)
    err = rel_err(got, ref)
    assert err <= TOL[torch.bfloat16], f"normwise error {err:.3e}"


@pytest.mark.parametrize("B,n,C,s,e,causal,dtype", [
    (1, 128, 128, 32, 64, True, torch.float32),    # FLASH-Quad, fp32
    (2, 96, 96, 20, 40, False, torch.float32),
    (1, 256, 64, 32, 64, True, torch.float32),     # chunked, quad term only
])
def test_no_global_term_simt(B, n, C, s, e, causal, dtype):
    m = fm()
    Z, V, U, gamma, beta = mca_inputs.make_inputs(B, n, s, e, 5 + n, dtype)
    got = run_ex(Z, V, U, gamma, beta, C, causal, None, NONE, m.FMCA_PATH_SIMT)
    ref = oracle.forward(Z, V, U, gamma, beta, C, causal, lin_norm=NONE)
    assert rel_err(got, ref) <= TOL[dtype]


def test_flash_quad_base_workload_whole_output():
    """B = 8, n = 1024 (the pages' base-scale sequence length), s = 128,
    e = 1536, causal, compared over the whole output."""
    m = fm()
    w = mca_inputs.WORKLOADS["flash_quad_base"]
    Z, V, U, gamma, beta = mca_inputs.workload_inputs(w, mca_inputs.WORKLOAD_ORDER.index(w.name) + 1)
    got = run_ex(Z, V, U, gamma, beta, w.C, w.causal, None, NONE, m.FMCA_PATH_AUTO)
    ref = oracle.forward(Z, V, U, gamma, beta, w.C, w.causal, lin_norm=NONE)
    err = rel_err(got, ref)
    print(f"parity flash_quad_base: normwise error {err:.3e}")
    assert err <= TOL[torch.bfloat16], f"normwise error {err:.3e}"
