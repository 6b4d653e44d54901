"""flash_mca_forward_noalloc: the forward pass for callers that cannot allocate
device memory (a component running inside a framework that owns all device
memory, or code that must not risk an out-of-memory failure), with its scratch
in a fixed array inside the library.

The GPU test calls the new entry point through the C ABI twice in a row, on
different inputs, then once more with another layout of the scratch (another
batch size, e and mode, so the states and prefix sit at other offsets over
what the earlier calls left), and compares each result with the regular entry
point (flash_mca_forward with a caller workspace) under the bf16 parity bar
used by every other test.  This file sorts last so that a run stopping at its first
failure has already run every other test; it also passes on its own in a fresh
process.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import mca_inputs


def fm():
    import flash_mixed_chunk_gb300 as m
    return m


def test_noalloc_rejects_problems_larger_than_its_scratch():
    """Host-side checks only: no GPU needed, nothing is queued."""
    m = fm()
    P = 0x7F0000000000
    # the very long causal workload: its bf16 states and prefix (2 x 67 MB)
    # exceed the fixed scratch
    B, n, C, s, e = 1, 32768, 256, 128, 2048
    G = n // C
    assert 2 * 2 * B * G * s * e > m.FMCA_NOALLOC_SCRATCH_BYTES
    st = m.lib.flash_mca_forward_noalloc(P, P + (1 << 30), P + (2 << 30), P + (3 << 30),
                                         P + (3 << 30) + 4096, P + (4 << 30), B, n, s, e, C, 1,
                                         m.FMCA_BF16, None)
    assert st == m.FMCA_ERR_WORKSPACE
    # shapes outside the tensor-core path, and bad arguments
    assert m.lib.flash_mca_forward_noalloc(P, P, P, P, P, P, 1, 256, 32, 64, 64, 1,
                                           m.FMCA_F32, None) == m.FMCA_ERR_UNSUPPORTED
    assert m.lib.flash_mca_forward_noalloc(P, P, P, P, P, P, 1, 250, 128, 256, 128, 1,
                                           m.FMCA_BF16, None) == m.FMCA_ERR_SHAPE
    assert m.lib.flash_mca_forward_noalloc(0, P, P, P, P, P, 1, 256, 128, 256, 128, 1,
                                           m.FMCA_BF16, None) == m.FMCA_ERR_INVALID_ARG


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_point_on_two_calls():
    m = fm()
    dev = torch.device("cuda:0")
    C, s = 256, 128
    stream = torch.cuda.current_stream(dev)
    # two calls in a row on different inputs, then a third whose states and
    # prefix lie elsewhere in the scratch
    for seed, B, n, e, causal in ((71, 2, 1024, 512, True), (72, 2, 1024, 512, True),
                                  (73, 3, 2048, 768, False)):
        assert m.flash_mca_workspace_bytes(B, n, s, e, C, causal, m.FMCA_BF16) <= \
            m.FMCA_NOALLOC_SCRATCH_BYTES
        Z, V, U, gamma, beta = (t.to(dev) for t in
                                mca_inputs.make_inputs(B, n, s, e, seed, torch.bfloat16))
        O_ref = torch.empty((B, n, e), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(m.flash_mca_workspace_bytes(B, n, s, e, C, causal, m.FMCA_BF16),
                         dtype=torch.uint8, device=dev)
        m.flash_mca_forward(Z, V, U, gamma, beta, O_ref, C, causal, ws, stream)
        O = torch.full((B, n, e), float("nan"), dtype=torch.bfloat16, device=dev)
        st = m.lib.flash_mca_forward_noalloc(
            Z.data_ptr(), V.data_ptr(), U.data_ptr(), gamma.data_ptr(), beta.data_ptr(),
            O.data_ptr(), B, n, s, e, C, int(causal), m.FMCA_BF16,
            ctypes.c_void_p(stream.cuda_stream))
        assert st == m.FMCA_OK, m.flash_mca_status_string(st)
        torch.cuda.synchronize(dev)
        assert m.flash_mca_device_status() == (m.FMCA_OK, 0)
        a = O.float().cpu().numpy()
        b = O_ref.float().cpu().numpy()
        assert np.all(np.isfinite(a))
        err = float(np.max(np.abs(a - b)) / np.max(np.abs(b)))
        assert err <= 2e-2, f"call with seed {seed}: normwise difference {err:.3e}"
