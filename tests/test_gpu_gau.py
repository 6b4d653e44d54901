"""GPU parity of the GAU projections (flash_mca_gau_project / _output, on
the tensor cores) against the fp64 oracle (oracle/gau.py) on the same bf16
inputs: normwise 2e-2 (bf16 outputs)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import gau

from tests.test_gpu_parity import fm, rel_err

pytestmark = pytest.mark.gpu


def rand_bf16(shape, scale, seed):
    g = torch.Generator().manual_seed(seed)
    return (scale * torch.randn(*shape, generator=g)).to(torch.bfloat16)


@pytest.mark.parametrize("M,d,e,s", [
    (256, 768, 1536, 128),     # GAU base dims
    (300, 768, 1536, 128),     # ragged rows
    (130, 72, 64, 64),         # K not a multiple of 64, small N
    (1, 64, 128, 64),          # one row
    (1000, 1024, 2048, 128),   # e = 2d with d = 1024
])
def test_projection(M, d, e, s):
    m = fm()
    X = rand_bf16((M, d), 1.0, 1 + M)
    Wt = rand_bf16((2 * e + s, d), d ** -0.5, 2 + d)
    U, V, Z = m.gau_project(X.cuda(), Wt.cuda(), e, s)
    torch.cuda.synchronize()
    rU, rV, rZ = gau.gau_project(X.double().numpy(), Wt.double().numpy(), e, s)
    for name, got, ref in (("U", U, rU), ("V", V, rV), ("Z", Z, rZ)):
        err = rel_err(got.float().cpu().numpy(), ref)
        assert err <= 2e-2, f"{name}: normwise error {err:.3e}"


@pytest.mark.parametrize("M,e,d", [(256, 1536, 768), (77, 136, 64), (2048, 2048, 1024)])
def test_output_projection(M, e, d):
    m = fm()
    Y = rand_bf16((M, e), 1.0, 5 + M)
    Wo_t = rand_bf16((d, e), e ** -0.5, 6 + e)
    Out = m.gau_output(Y.cuda(), Wo_t.cuda())
    torch.cuda.synchronize()
    ref = gau.gau_output(Y.double().numpy(), Wo_t.double().numpy())
    assert rel_err(Out.float().cpu().numpy(), ref) <= 2e-2


def test_gau_layer_on_the_gpu():
    """Projections -> core (tensor-core path) -> output projection, against
    the oracle's composition."""
    import oracle
    m = fm()
    n, d, e, s, C = 512, 256, 512, 128, 256
    X = rand_bf16((n, d), 1.0, 9)
    Wt = rand_bf16((2 * e + s, d), d ** -0.5, 10)
    Wo_t = rand_bf16((d, e), e ** -0.5, 11)
    gamma = (1 + 0.1 * torch.randn(4, s, generator=torch.Generator().manual_seed(12))).float()
    beta = (0.1 * torch.randn(4, s, generator=torch.Generator().manual_seed(13))).float()
    U, V, Z = m.gau_project(X.cuda(), Wt.cuda(), e, s)
    O = m.forward(Z[None], V[None], U[None], gamma.cuda(), beta.cuda(), C, True)
    Out = m.gau_output(O[0], Wo_t.cuda())
    torch.cuda.synchronize()
    rU, rV, rZ = gau.gau_project(X.double().numpy(), Wt.double().numpy(), e, s)
    rO = oracle.forward(rZ[None], rV[None], rU[None], gamma.double().numpy(),
                        beta.double().numpy(), C, True)[0]
    ref = gau.gau_output(rO, Wo_t.double().numpy())
    assert rel_err(Out.float().cpu().numpy(), ref) <= 2e-2
