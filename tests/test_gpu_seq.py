"""The forward pass on pieces of longer causal sequences (flash_mca_forward_seq):
the cumsum form of the global term ("Mixed Chunk") carried from one call to
the next through an fp32 state.  Running the pieces of a sequence in order,
each with the state the previous one left, gives the whole sequence's output:
checked over the whole output against the fp64 oracle on the whole sequence,
for both output kernels (chunks of 256 and of 128) and every divisor."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mca_inputs
import oracle

from tests.test_gpu_parity import TOL, fm, rel_err

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


def run_pieces(Z, V, U, gamma, beta, C, cuts, lin_norm, quad_scale, in_place=False):
    m = fm()
    dev = torch.device("cuda:0")
    B, n, s = Z.shape
    e = V.shape[2]
    gd, bd = gamma.to(dev), beta.to(dev)
    state = torch.zeros((B, s, e), dtype=torch.float32, device=dev)
    outs = []
    bounds = [0] + list(cuts) + [n]
    for k in range(len(bounds) - 1):
        a, b = bounds[k], bounds[k + 1]
        Zp, Vp, Up = (t[:, a:b].contiguous().to(dev) for t in (Z, V, U))
        Op = torch.empty((B, b - a, e), dtype=BF, device=dev)
        ws = torch.empty(m.flash_mca_workspace_bytes(B, b - a, s, e, C, True, m.FMCA_BF16),
                         dtype=torch.uint8, device=dev)
        if in_place:
            state_in, state_out = (state if k > 0 else None), state
        else:
            state_in = state if k > 0 else None
            state_out = torch.empty_like(state)
        m.flash_mca_forward_seq(Zp, Vp, Up, gd, bd, Op, C, ws, state_in=state_in,
                                state_out=state_out, token_offset=a, n_norm=n,
                                quad_scale=quad_scale, lin_norm=lin_norm)
        state = state_out
        outs.append(Op)
    torch.cuda.synchronize()
    assert m.flash_mca_device_status() == (m.FMCA_OK, 0)
    return torch.cat(outs, dim=1), state


@pytest.mark.parametrize("C,ln,qs", [
    (256, 0, None),      # the default divisor 1/n with n the whole length
    (256, 1, "cs"),      # tokens summed, the page's 1/(C s) scale
    (256, 2, None),      # by position
    (128, 0, None),      # chunks of 128: the fused output kernel and the carry launch
])
def test_pieces_give_the_whole_sequence(C, ln, qs):
    B, n, s, e = 2, 4096, 128, 512
    Z, V, U, gamma, beta = mca_inputs.make_inputs(B, n, s, e, 200 + C + ln, BF)
    quad_scale = 1.0 / (C * s) if qs == "cs" else None
    got, _ = run_pieces(Z, V, U, gamma, beta, C, [1536, 2560], ln, quad_scale)
    ref = oracle.forward(Z, V, U, gamma, beta, C, True, quad_scale=quad_scale, lin_norm=ln)
    err = rel_err(got.float().cpu().numpy(), ref)
    print(f"parity pieces C{C} lin_norm={ln}: normwise error {err:.3e}")
    assert err <= TOL[BF], f"normwise error {err:.3e}"


def test_state_in_place_and_state_out_is_the_chunk_state_sum():
    """state_out after the last piece is the sum over every chunk of T3^T V
    (T3 = Z gamma_3 + beta_3), whatever the cuts; the state may be updated in
    place."""
    B, n, s, e, C = 2, 2048, 128, 512, 256
    Z, V, U, gamma, beta = mca_inputs.make_inputs(B, n, s, e, 211, BF)
    got, state = run_pieces(Z, V, U, gamma, beta, C, [256, 1024], 0, None, in_place=True)
    whole, _ = run_pieces(Z, V, U, gamma, beta, C, [], 0, None)
    assert rel_err(got.float().cpu().numpy(), whole.float().cpu().numpy()) <= TOL[BF]
    z = Z.double().numpy()
    T3 = z * gamma[3].double().numpy() + beta[3].double().numpy()
    ref = np.einsum("bts,bte->bse", T3, V.double().numpy())
    err = rel_err(state.cpu().numpy(), ref)
    print(f"parity state_out: normwise error {err:.3e}")
    assert err <= TOL[BF], f"normwise error {err:.3e}"


def test_pieces_reject_what_they_do_not_cover():
    m = fm()
    dev = torch.device("cuda:0")
    B, n, s, e, C = 1, 512, 128, 256, 256
    Z, V, U, gamma, beta = (t.to(dev) for t in mca_inputs.make_inputs(B, n, s, e, 5, BF))
    O = torch.empty_like(U)
    ws = torch.empty(m.flash_mca_workspace_bytes(B, n, s, e, C, True, m.FMCA_BF16),
                     dtype=torch.uint8, device=dev)
    opts = m.flash_mca_default_options(C)
    state = torch.zeros((B, s, e), dtype=torch.float32, device=dev)

    def call(causal, offset, ln=0, st=state):
        opts.lin_norm = ln
        seq = m.FmcaSeq(st.data_ptr(), st.data_ptr(), offset, 0)
        return m.lib.flash_mca_forward_seq(Z.data_ptr(), V.data_ptr(), U.data_ptr(),
                                           gamma.data_ptr(), beta.data_ptr(), O.data_ptr(), B,
                                           n, s, e, C, causal, m.FMCA_BF16, ws.data_ptr(),
                                           ws.numel(), m.ctypes.byref(opts),
                                           m.ctypes.byref(seq), None)
    assert call(0, 0) == m.FMCA_ERR_UNSUPPORTED       # bidirectional
    assert call(1, 128) == m.FMCA_ERR_INVALID_ARG     # not a chunk boundary
    assert call(1, -256) == m.FMCA_ERR_INVALID_ARG
    assert call(1, 0, ln=3) == m.FMCA_ERR_UNSUPPORTED  # no global term
    torch.cuda.synchronize()
    assert m.flash_mca_device_status() == (m.FMCA_OK, 0)
