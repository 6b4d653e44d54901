"""Full-size parity of the backward pass: the bench workloads' shapes (the
launch configuration ``bench.py --backward`` times), every gradient against
the fp64 backward oracle (oracle/backward.py, autograd of the forward
definition; vectorised over chunks, so the full shapes take seconds on the
host), normwise at the bf16 bar 2e-2.  The inputs and dO come from the same
seeded generator the bench uses.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mca_inputs
from oracle import backward as obwd

from tests.test_gpu_backward import NAMES, run_backward
from tests.test_gpu_parity import TOL, rel_err

pytestmark = pytest.mark.gpu

LIN_NORM = {"n": 0, "summed": 1, "position": 2, "none": 3}


@pytest.mark.parametrize("name", ["long_causal", "gau_base_causal", "bidir_mlm",
                                  "flash_quad_base"])
def test_backward_full_size(name):
    w = mca_inputs.WORKLOADS[name]
    seed = mca_inputs.WORKLOAD_ORDER.index(name) + 1
    Z, V, U, gamma, beta = mca_inputs.workload_inputs(w, seed)
    dO = torch.randn(w.B, w.n, w.e, generator=torch.Generator().manual_seed(seed + 100)).to(
        Z.dtype)
    ln = LIN_NORM[w.lin_norm]
    got = run_backward(Z, V, U, gamma, beta, dO, w.C, w.causal, None, ln)
    ref = obwd.backward(Z, V, U, gamma, beta, dO, w.C, w.causal, None, ln)
    for gname, a, b in zip(NAMES, got, ref):
        assert np.all(np.isfinite(a)), gname
        err = rel_err(a, b)
        assert err <= TOL[torch.bfloat16], f"{name} {gname}: normwise error {err:.3e}"
