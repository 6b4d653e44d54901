"""GPU parity of the backward pass (flash_mca_backward) against the fp64
backward oracle (oracle/backward.py: autograd of the forward definition,
pinned by finite differences of the C oracle).  Every gradient -- dZ, dV, dU,
dgamma, dbeta -- is compared normwise (max |got - ref| / max |ref|) at the
forward pass's bars: 1e-5 for fp32 I/O, 2e-2 for bf16 I/O.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mca_inputs
from oracle import backward as obwd

from tests.test_gpu_parity import TOL, fm, rel_err

pytestmark = pytest.mark.gpu

VARIANTS = [(None, 0), (None, 1), (None, 2), (0.1, 3), ("cs", 0)]
NAMES = ("dZ", "dV", "dU", "dgamma", "dbeta")


def run_backward(Z, V, U, gamma, beta, dO, C, causal, quad_scale, lin_norm):
    m = fm()
    dev = torch.device("cuda:0")
    out = m.backward(Z.to(dev), V.to(dev), U.to(dev), gamma.to(dev), beta.to(dev), dO.to(dev), C,
                     causal, quad_scale, lin_norm)
    torch.cuda.synchronize()
    st, where = m.flash_mca_device_status()
    assert st == m.FMCA_OK, f"device status {st} at {where}"
    return [t.float().cpu().numpy() for t in out]


def check(B, n, C, s, e, causal, dtype, variant, seed):
    qs, ln = variant
    quad_scale = 1.0 / (C * s) if qs == "cs" else qs
    Z, V, U, gamma, beta = mca_inputs.make_inputs(B, n, s, e, seed, dtype)
    g = torch.Generator().manual_seed(seed + 1)
    dO = torch.randn(B, n, e, generator=g).to(dtype)
    got = run_backward(Z, V, U, gamma, beta, dO, C, causal, quad_scale, ln)
    ref = obwd.backward(Z, V, U, gamma, beta, dO, C, causal, quad_scale, ln)
    for name, a, b in zip(NAMES, got, ref):
        assert np.all(np.isfinite(a)), name
        if np.max(np.abs(b)) == 0:
            assert np.max(np.abs(a)) == 0, name
            continue
        err = rel_err(a, b)
        assert err <= TOL[dtype], f"{name}: normwise error {err:.3e}"


@pytest.mark.parametrize("variant", VARIANTS, ids=[f"{q}-{l}" for q, l in VARIANTS])
@pytest.mark.parametrize("B,n,C,s,e,causal", [
    (1, 64, 16, 8, 24, True),
    (1, 64, 16, 8, 24, False),
    (1, 96, 32, 20, 40, True),      # ragged tiles
    (2, 128, 64, 32, 72, True),
    (2, 128, 64, 32, 72, False),
])
def test_backward_fp32(B, n, C, s, e, causal, variant):
    check(B, n, C, s, e, causal, torch.float32, variant, seed=11 + n + s)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("variant", [(None, 0), (None, 3)], ids=["default", "no-global"])
def test_backward_bf16(causal, variant):
    # a tensor-core shape: the bf16 tensor-core backward
    check(1, 512, 256, 128, 256, causal, torch.bfloat16, variant, seed=3)


@pytest.mark.parametrize("causal", [True, False])
def test_backward_bf16_cuda_cores(causal):
    # s = 64: not a tensor-core shape, so bf16 I/O through the CUDA-core backward
    check(2, 256, 64, 64, 96, causal, torch.bfloat16, (None, 0), seed=4)


def test_backward_is_deterministic():
    B, n, C, s, e = 1, 128, 64, 32, 64
    Z, V, U, gamma, beta = mca_inputs.make_inputs(B, n, s, e, 4, torch.float32)
    dO = torch.randn(B, n, e, generator=torch.Generator().manual_seed(9))
    a = run_backward(Z, V, U, gamma, beta, dO, C, True, None, 0)
    b = run_backward(Z, V, U, gamma, beta, dO, C, True, None, 0)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
