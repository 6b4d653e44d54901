"""GPU parity of the decode step (flash_mca_decode_step): decoding a sequence
token by token must give, row by row, the causal forward pass over the whole
sequence -- the oracle's, at the same bars as the forward pass (2e-2 bf16,
1e-5 fp32, normwise).  "FLASH: Possibly the Most Interesting Efficient
Transformer Design Recently", section "Mixed Chunk" (the decoder form), and the
recurrent form of linear attention ("大模型训练之加速篇 -attention优化", §1.4).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mca_inputs
import oracle

from tests.test_gpu_parity import TOL, fm, rel_err

pytestmark = pytest.mark.gpu


def decode_sequence(Z, V, U, gamma, beta, C, quad_scale=None, lin_norm=0, state=None):
    """Decode all n positions of Z/V/U [B, n, ·] on the GPU; returns O [B, n, e]."""
    m = fm()
    dev = torch.device("cuda:0")
    B, n, s = Z.shape
    e = V.shape[2]
    dt = m.FMCA_BF16 if Z.dtype == torch.bfloat16 else m.FMCA_F32
    Zd, Vd, Ud = (x.to(dev) for x in (Z, V, U))
    gd, bd = gamma.to(dev), beta.to(dev)
    if state is None:
        state = torch.empty(m.flash_mca_decode_state_bytes(B, s, e, C, dt), dtype=torch.uint8,
                            device=dev)
    m.flash_mca_decode_reset(state, B, s, e, C, dt)
    O = torch.empty((B, n, e), dtype=Z.dtype, device=dev)
    o = torch.empty((B, e), dtype=Z.dtype, device=dev)
    for t in range(n):
        # per-token rows as fresh (aligned) copies, as a caller's would be
        m.flash_mca_decode_step(Zd[:, t].clone(), Vd[:, t].clone(), Ud[:, t].clone(), gd, bd,
                                o, C, t, state, n_norm=n,
                                quad_scale=quad_scale, lin_norm=lin_norm)
        O[:, t] = o
    torch.cuda.synchronize()
    st, where = m.flash_mca_device_status()
    assert st == m.FMCA_OK, f"device status {st} at {where}"
    return O.float().cpu().numpy()


VARIANTS = [(None, 0), (None, 1), (None, 2), ("cs", 0), ("cs", 1)]


@pytest.mark.parametrize("variant", VARIANTS, ids=[f"{q}-{l}" for q, l in VARIANTS])
@pytest.mark.parametrize("B,n,C,s,e,dtype", [
    # s or e not a multiple of 8: a column a lane
    (1, 100, 25, 20, 130, torch.float32),     # ragged everything
    (140, 64, 32, 16, 204, torch.float32),    # wide blocks (two 32-column groups per lane)
    (280, 64, 32, 16, 204, torch.float32),    # wider blocks (four groups), ragged e
    # s and e multiples of 8: 16-byte rows, a key weight a thread, blocks of
    # 256, 128 or 64 columns
    (2, 192, 64, 32, 80, torch.float32),      # 64 columns, few blocks; ragged e
    (2, 512, 128, 128, 256, torch.bfloat16),  # 64 columns, few blocks
    (280, 64, 32, 16, 200, torch.float32),    # 256 columns; ragged e: 25 of 32 lanes
    (160, 128, 64, 32, 512, torch.bfloat16),  # 256 columns, two blocks, two chunks
    (40, 64, 32, 16, 512, torch.bfloat16),    # 128 columns, two rows a warp
    (20, 96, 32, 16, 456, torch.float32),     # 64 columns, four rows a warp; ragged e
])
def test_decode_equals_the_causal_forward(B, n, C, s, e, dtype, variant):
    qs, ln = variant
    quad_scale = 1.0 / (C * s) if qs == "cs" else qs
    Z, V, U, gamma, beta = mca_inputs.make_inputs(B, n, s, e, 40 + n + s, dtype)
    got = decode_sequence(Z, V, U, gamma, beta, C, quad_scale, ln)
    ref = oracle.forward(Z, V, U, gamma, beta, C, True, quad_scale=quad_scale, lin_norm=ln)
    assert np.all(np.isfinite(got))
    err = rel_err(got, ref)
    assert err <= TOL[dtype], f"normwise error {err:.3e}"
    # early rows carry the divisor's extremes (chunk 0, first tokens): check
    # them on their own scale too
    err0 = rel_err(got[:, : 2 * C], ref[:, : 2 * C])
    assert err0 <= TOL[dtype], f"normwise error over the first two chunks {err0:.3e}"


def test_decode_matches_the_tensor_core_forward():
    """The decode state reproduces what the chunked tensor-core forward pass
    computes for the same bf16 sequence."""
    m = fm()
    B, n, C, s, e = 1, 768, 256, 128, 256
    Z, V, U, gamma, beta = mca_inputs.make_inputs(B, n, s, e, 9, torch.bfloat16)
    got = decode_sequence(Z, V, U, gamma, beta, C)
    dev = torch.device("cuda:0")
    fwd = m.forward(Z.to(dev), V.to(dev), U.to(dev), gamma.to(dev), beta.to(dev), C, True,
                    path=m.FMCA_PATH_TCGEN05).float().cpu().numpy()
    assert rel_err(got, fwd) <= TOL[torch.bfloat16]


def test_reset_restarts_the_sequence():
    m = fm()
    B, n, C, s, e = 2, 96, 32, 16, 64
    Z, V, U, gamma, beta = mca_inputs.make_inputs(B, n, s, e, 2, torch.float32)
    state = torch.empty(m.flash_mca_decode_state_bytes(B, s, e, C, m.FMCA_F32), dtype=torch.uint8,
                        device="cuda:0")
    a = decode_sequence(Z, V, U, gamma, beta, C, state=state)
    b = decode_sequence(Z, V, U, gamma, beta, C, state=state)
    assert np.array_equal(a, b)
