"""GPU parity: the CUDA path (called through the C ABI) against the fp64 CPU
oracle on the same seeded inputs.

Error metric (normwise): max |O_gpu - O_ref| / max |O_ref| over the compared
elements.  Bars: 2e-2 for bf16 I/O, 1e-5 for fp32 I/O.  Small cases are
compared element by element over the whole output; the full-size workloads
are compared over the whole output too.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mca_inputs
import oracle

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 2e-2, torch.float32: 1e-5}


def fm():
    import flash_mixed_chunk_gb300 as m
    return m


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def run_gpu(Z, V, U, gamma, beta, C, causal, path=0):
    m = fm()
    dev = torch.device("cuda:0")
    Zd, Vd, Ud = Z.to(dev), V.to(dev), U.to(dev)
    gd, bd = gamma.to(dev), beta.to(dev)
    O = m.forward(Zd, Vd, Ud, gd, bd, C, causal, path=path)
    torch.cuda.synchronize()
    st, where = m.flash_mca_device_status()
    assert st == m.FMCA_OK, f"device status {st} at {where}"
    return O


def check_full(B, n, C, s, e, causal, dtype, seed, path=0, tol=None):
    Z, V, U, gamma, beta = mca_inputs.make_inputs(B, n, s, e, seed, dtype)
    O = run_gpu(Z, V, U, gamma, beta, C, causal, path).float().cpu().numpy()
    ref = oracle.forward(Z, V, U, gamma, beta, C, causal)
    err = rel_err(O, ref)
    assert np.all(np.isfinite(O))
    assert err <= (tol if tol is not None else TOL[dtype]), f"normwise error {err:.3e}"
    return err


def report(case, err):
    """One line per case with its normwise error (visible under pytest -s)."""
    print(f"parity {case}: normwise error {err:.3e}")


# ---------------------------------------------------------------- small, whole output
def test_tiny_causal_f32_workload():
    w = mca_inputs.WORKLOADS["tiny_causal_f32"]
    report("tiny_causal_f32", check_full(w.B, w.n, w.C, w.s, w.e, w.causal, torch.float32,
                                         seed=1))


@pytest.mark.parametrize("B,n,C,s,e,causal", [
    (1, 512, 256, 128, 512, True),      # 2 chunks, 2 row tiles, 2 e tiles
    (1, 512, 256, 128, 512, False),
    (2, 384, 128, 128, 256, True),      # C = 128: one row tile per chunk
    (2, 384, 128, 128, 768, False),
    (1, 256, 256, 128, 256, True),      # one chunk: no global term
    (1, 256, 256, 128, 256, False),     # one chunk: global term = full linear attention
    (3, 1024, 256, 128, 1024, True),    # 4 chunks, 4 e tiles
])
def test_tensor_core_path_small(B, n, C, s, e, causal):
    m = fm()
    assert m.flash_mca_auto_path(B, n, s, e, C, causal, m.FMCA_BF16) == m.FMCA_PATH_TCGEN05
    check_full(B, n, C, s, e, causal, torch.bfloat16, seed=100 + n + e,
               path=m.FMCA_PATH_TCGEN05)


@pytest.mark.parametrize("B,n,C,s,e,causal,dtype", [
    (1, 96, 32, 48, 80, True, torch.float32),      # ragged: nothing a multiple of 64
    (2, 96, 32, 48, 80, False, torch.float32),
    (1, 100, 25, 20, 33, True, torch.float32),
    (1, 64, 64, 256, 70, True, torch.float32),     # s at its maximum, one chunk
    (2, 12, 1, 3, 5, True, torch.float32),         # C = 1: every chunk one token
    (1, 96, 32, 48, 80, True, torch.bfloat16),
    (1, 512, 256, 64, 256, True, torch.bfloat16),  # bf16 shape outside the tensor-core path
])
def test_simt_path_small(B, n, C, s, e, causal, dtype):
    m = fm()
    check_full(B, n, C, s, e, causal, dtype, seed=7 + n + s + e, path=m.FMCA_PATH_SIMT)


def test_tensor_core_matches_simt_path():
    """The two kernel families agree on the same bf16 inputs (both also match
    the oracle)."""
    m = fm()
    Z, V, U, gamma, beta = mca_inputs.make_inputs(2, 1024, 128, 512, 31, torch.bfloat16)
    a = run_gpu(Z, V, U, gamma, beta, 256, True, m.FMCA_PATH_TCGEN05).float().cpu().numpy()
    b = run_gpu(Z, V, U, gamma, beta, 256, True, m.FMCA_PATH_SIMT).float().cpu().numpy()
    assert rel_err(a, b) <= 2e-2


def test_deterministic_bits():
    m = fm()
    Z, V, U, gamma, beta = mca_inputs.make_inputs(1, 1024, 128, 512, 5, torch.bfloat16)
    a = run_gpu(Z, V, U, gamma, beta, 256, True, m.FMCA_PATH_TCGEN05)
    b = run_gpu(Z, V, U, gamma, beta, 256, True, m.FMCA_PATH_TCGEN05)
    assert torch.equal(a, b)


def test_causality_on_gpu():
    """Outputs before position p do not change when tokens from p on change."""
    m = fm()
    Z, V, U, gamma, beta = mca_inputs.make_inputs(1, 1024, 128, 256, 9, torch.bfloat16)
    base = run_gpu(Z, V, U, gamma, beta, 256, True, m.FMCA_PATH_TCGEN05)
    p = 300  # inside chunk 1, second row tile
    Z2, V2, U2 = Z.clone(), V.clone(), U.clone()
    Z2[:, p:] = Z2[:, p:].flip(1)
    V2[:, p:] = -V2[:, p:]
    pert = run_gpu(Z2, V2, U2, gamma, beta, 256, True, m.FMCA_PATH_TCGEN05)
    assert torch.equal(pert[:, :p], base[:, :p])
    assert not torch.equal(pert[:, p:], base[:, p:])


@pytest.mark.parametrize("B,causal", [(2, True), (5, False), (1, True)])
def test_host_buffer_entry_matches_device_entry(B, causal):
    m = fm()
    n, C, s, e = 512, 256, 128, 512
    Z, V, U, gamma, beta = mca_inputs.make_inputs(B, n, s, e, 3, torch.bfloat16)
    dev = run_gpu(Z, V, U, gamma, beta, C, causal).cpu()
    pins = [t.pin_memory() for t in (Z, V, U, gamma, beta)]
    Oh = torch.empty((B, n, e), dtype=torch.bfloat16).pin_memory()
    arena = torch.empty(m.flash_mca_host_arena_bytes(B, n, s, e, C, causal, m.FMCA_BF16),
                        dtype=torch.uint8, device="cuda:0")
    m.flash_mca_forward_host(*pins, Oh, C, causal, arena)
    assert torch.equal(Oh, dev)


@pytest.mark.parametrize("B,n,causal", [(2, 8192, True), (5, 4096, False), (1, 32768, True)])
def test_host_buffer_pipeline_whole_output(B, n, causal):
    """Problems of 96 MB and more go through the host-buffer entry point in
    pieces (copies overlapping the passes): of whole sequences (B = 5,
    bidirectional), or, for fewer than four causal sequences, of every
    sequence's tokens with the chunk-state sum carried between them (B = 2
    and B = 1).  The whole output against the oracle (each piece is a batch
    of its own, so the bits may differ from one call on the whole batch; the
    bar is the same)."""
    m = fm()
    C, s, e = 256, 128, 1536
    Z, V, U, gamma, beta = mca_inputs.make_inputs(B, n, s, e, 61 + B, torch.bfloat16)
    pins = [t.pin_memory() for t in (Z, V, U, gamma, beta)]
    Oh = torch.empty((B, n, e), dtype=torch.bfloat16).pin_memory()
    arena = torch.empty(m.flash_mca_host_arena_bytes(B, n, s, e, C, causal, m.FMCA_BF16),
                        dtype=torch.uint8, device="cuda:0")
    m.flash_mca_forward_host(*pins, Oh, C, causal, arena)
    assert m.flash_mca_device_status() == (m.FMCA_OK, 0)
    ref = oracle.forward(Z, V, U, gamma, beta, C, causal)
    err = rel_err(Oh.float().numpy(), ref)
    report(f"host_pipeline_B{B}_n{n}_{'causal' if causal else 'bidir'}", err)
    assert err <= TOL[torch.bfloat16], f"normwise error {err:.3e}"


def test_timeout_path_records_status_and_context_survives():
    m = fm()
    assert m.flash_mca_device_status() == (m.FMCA_OK, 0)
    m.flash_mca_selftest_timeout(2000)  # 2 ms limit on a wait nothing satisfies
    st, where = m.flash_mca_device_status()
    assert st == m.FMCA_ERR_TIMEOUT and where == 900
    assert m.flash_mca_device_status() == (m.FMCA_OK, 0)  # read clears it
    # the context is still usable
    check_full(1, 256, 128, 128, 256, True, torch.bfloat16, seed=44)


# ---------------------------------------------------------------- full-size workloads
# Every workload at full size, compared over the whole output.  Each test
# prints its normwise error ("parity <case>: <err>") so that the margin under
# the bar is on record; run pytest with -s to see the lines.
@pytest.mark.parametrize("name", ["gau_base_causal", "bidir_mlm", "long_causal",
                                  "very_long_causal"])
def test_full_size_workload_whole_output(name):
    w = mca_inputs.WORKLOADS[name]
    seed = mca_inputs.WORKLOAD_ORDER.index(name) + 1
    Z, V, U, gamma, beta = mca_inputs.workload_inputs(w, seed)
    m = fm()
    assert m.flash_mca_auto_path(w.B, w.n, w.s, w.e, w.C, w.causal, m.FMCA_BF16) == \
        m.FMCA_PATH_TCGEN05
    O = run_gpu(Z, V, U, gamma, beta, w.C, w.causal)
    assert torch.isfinite(O.float()).all()
    got = O.float().cpu().numpy()
    del O
    ref = oracle.forward(Z, V, U, gamma, beta, w.C, w.causal)
    err = rel_err(got, ref)
    report(name, err)
    assert err <= TOL[torch.bfloat16], f"{name}: normwise error {err:.3e}"


@pytest.mark.parametrize("B,n,C,e,causal", [
    # 512 output tiles and 128 walker units of 2 chunks: every CTA of the
    # output kernel takes several tiles and its rings wrap
    (4, 4096, 128, 512, True),
    (4, 4096, 128, 512, False),
    # 160 walker units (one segment per sequence and e slice): more than the
    # SMs, so walkers take a second unit; 1280 row-pair tiles
    (16, 1024, 256, 2560, True),
    (16, 1024, 256, 2560, False),
    # e % 256 == 128: the walkers' last e slice is 128 columns wide
    (4, 2048, 256, 640, True),
    (4, 2048, 256, 640, False),
    (4, 2048, 128, 384, True),
    # e % 128 == 64: the last e tile is 64 columns, the last slice 64 of 256
    (4, 2048, 256, 576, True),
    (4, 2048, 256, 576, False),
    (4, 2048, 128, 320, True),
])
def test_more_units_than_sms_whole_output(B, n, C, e, causal):
    """Shapes that are not benchmark workloads, with more work units than SMs."""
    m = fm()
    s = 128
    assert m.flash_mca_auto_path(B, n, s, e, C, causal, m.FMCA_BF16) == m.FMCA_PATH_TCGEN05
    err = check_full(B, n, C, s, e, causal, torch.bfloat16, seed=n + e + causal,
                     path=m.FMCA_PATH_TCGEN05)
    report(f"B{B}_n{n}_C{C}_e{e}_{'causal' if causal else 'bidir'}", err)
