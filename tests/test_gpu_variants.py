"""GPU parity of the scale and normalisation variants (flash_mca_forward_ex)
against the oracle's variant form, on both kernel paths.

Variants ("FLASH: Possibly the Most Interesting Efficient Transformer Design
Recently", sections "Mixed Chunk" and "Extended Thoughts"): intra-chunk weights
quad_scale * relu(q . k)^2 with the page's quad_scale = 1/(C s), and the
global-term divisor n, the number of tokens the sum covers, or the token's
position.  Same error metric and bars as tests/test_gpu_parity.py.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mca_inputs
import oracle

from tests.test_gpu_parity import TOL, fm, rel_err

pytestmark = pytest.mark.gpu

N, SUMMED, POSITION = 0, 1, 2
VARIANTS = [("cs", N), (None, SUMMED), (None, POSITION), ("cs", SUMMED), (0.05, POSITION)]


def run_ex(Z, V, U, gamma, beta, C, causal, quad_scale, lin_norm, path):
    m = fm()
    dev = torch.device("cuda:0")
    O = m.forward(Z.to(dev), V.to(dev), U.to(dev), gamma.to(dev), beta.to(dev), C, causal,
                  path=path, quad_scale=quad_scale, lin_norm=lin_norm)
    torch.cuda.synchronize()
    st, where = m.flash_mca_device_status()
    assert st == m.FMCA_OK, f"device status {st} at {where}"
    return O.float().cpu().numpy()


def check(B, n, C, s, e, causal, dtype, variant, path, seed):
    qs, ln = variant
    quad_scale = 1.0 / (C * s) if qs == "cs" else qs
    Z, V, U, gamma, beta = mca_inputs.make_inputs(B, n, s, e, seed, dtype)
    got = run_ex(Z, V, U, gamma, beta, C, causal, quad_scale, ln, path)
    ref = oracle.forward(Z, V, U, gamma, beta, C, causal, quad_scale=quad_scale, lin_norm=ln)
    assert np.all(np.isfinite(got))
    err = rel_err(got, ref)
    assert err <= TOL[dtype], f"normwise error {err:.3e}"


@pytest.mark.parametrize("variant", VARIANTS, ids=[f"{q}-{l}" for q, l in VARIANTS])
@pytest.mark.parametrize("B,n,C,s,e,causal", [
    (1, 512, 256, 128, 512, True),
    (1, 512, 256, 128, 512, False),
    (2, 640, 128, 128, 256, True),   # five chunks of 128
    (1, 512, 256, 128, 640, True),   # e % 256 == 128: a half-wide last walker slice
    (1, 512, 256, 128, 448, False),  # e % 128 == 64: a 64-column last e tile
])
def test_tensor_core_path(B, n, C, s, e, causal, variant):
    m = fm()
    check(B, n, C, s, e, causal, torch.bfloat16, variant, m.FMCA_PATH_TCGEN05, seed=7 + n)


@pytest.mark.parametrize("variant", [(None, N)] + VARIANTS,
                         ids=["default"] + [f"{q}-{l}" for q, l in VARIANTS])
@pytest.mark.parametrize("B,n,C,s,e,causal", [
    (1, 8192, 128, 128, 256, True),    # 64 chunks: the segmented chunk scan
    (2, 8960, 128, 128, 256, True),    # 70 chunks: segments of 18, 18, 18, 16
    (1, 8960, 128, 128, 256, False),
])
def test_tensor_core_path_long_chunk_axis(B, n, C, s, e, causal, variant):
    m = fm()
    check(B, n, C, s, e, causal, torch.bfloat16, variant, m.FMCA_PATH_TCGEN05, seed=5 + n)


@pytest.mark.parametrize("variant", VARIANTS, ids=[f"{q}-{l}" for q, l in VARIANTS])
@pytest.mark.parametrize("B,n,C,s,e,causal,dtype", [
    (1, 96, 32, 48, 80, True, torch.float32),     # ragged tiles
    (2, 96, 32, 48, 80, False, torch.float32),
    (1, 256, 64, 64, 128, True, torch.bfloat16),
])
def test_simt_path(B, n, C, s, e, causal, dtype, variant):
    m = fm()
    check(B, n, C, s, e, causal, dtype, variant, m.FMCA_PATH_SIMT, seed=3 + n + e)


@pytest.mark.parametrize("ln", [SUMMED, POSITION])
def test_paths_agree(ln):
    """Both kernel paths on one bf16 shape the tensor-core path covers."""
    m = fm()
    B, n, C, s, e = 1, 512, 128, 128, 256
    Z, V, U, gamma, beta = mca_inputs.make_inputs(B, n, s, e, 21, torch.bfloat16)
    a = run_ex(Z, V, U, gamma, beta, C, True, 1.0 / (C * s), ln, m.FMCA_PATH_TCGEN05)
    b = run_ex(Z, V, U, gamma, beta, C, True, 1.0 / (C * s), ln, m.FMCA_PATH_SIMT)
    assert rel_err(a, b) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("ln", [SUMMED, POSITION])
def test_long_causal_whole_output(ln):
    """The full long causal shape (B=2, n=8192, C=256, s=128, e=1536) with the
    page's 1/(cs) scale, compared over the whole output."""
    w = mca_inputs.WORKLOADS["long_causal"]
    m = fm()
    Z, V, U, gamma, beta = mca_inputs.workload_inputs(w, 77)
    qs = 1.0 / (w.C * w.s)
    got = run_ex(Z, V, U, gamma, beta, w.C, w.causal, qs, ln, m.FMCA_PATH_AUTO)
    ref = oracle.forward(Z, V, U, gamma, beta, w.C, w.causal, quad_scale=qs, lin_norm=ln)
    err = rel_err(got, ref)
    print(f"parity long_causal lin_norm={ln}: normwise error {err:.3e}")
    assert err <= TOL[torch.bfloat16], f"normwise error {err:.3e}"
