"""The forward pass captured in a CUDA graph: the library's calls are
asynchronous, allocation-free and queued on the caller's stream (the
tensor-core path's kernels chained by programmatic dependent launch), so a
stream capture of one call replays to the same bits as the eager call, on
both paths, and replays again after the inputs change in place."""
from __future__ import annotations

import pytest
import torch

import mca_inputs

from tests.test_gpu_parity import fm

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,n,C,s,e,causal,dtype", [
    (2, 1024, 256, 128, 512, True, torch.bfloat16),    # tensor-core path
    (1, 512, 128, 128, 256, False, torch.bfloat16),    # tensor-core path, bidirectional
    (1, 256, 64, 32, 64, True, torch.float32),         # CUDA-core path (launch-bound shape)
])
def test_forward_graph_replay(B, n, C, s, e, causal, dtype):
    m = fm()
    dev = torch.device("cuda:0")
    Z, V, U, gamma, beta = (t.to(dev) for t in mca_inputs.make_inputs(B, n, s, e, 7, dtype))
    code = m.FMCA_BF16 if dtype == torch.bfloat16 else m.FMCA_F32
    ws = torch.empty(m.flash_mca_workspace_bytes(B, n, s, e, C, causal, code), dtype=torch.uint8,
                     device=dev)
    O_eager = torch.empty(B, n, e, dtype=dtype, device=dev)
    O_graph = torch.empty_like(O_eager)
    stream = torch.cuda.current_stream(dev)
    m.flash_mca_forward(Z, V, U, gamma, beta, O_eager, C, causal, ws, stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        m.flash_mca_forward(Z, V, U, gamma, beta, O_graph, C, causal, ws,
                            torch.cuda.current_stream(dev))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(O_graph, O_eager)
    # new inputs in the captured buffers: the replay computes from them
    Z2, V2, U2, _, _ = (t.to(dev) for t in mca_inputs.make_inputs(B, n, s, e, 8, dtype))
    Z.copy_(Z2)
    V.copy_(V2)
    U.copy_(U2)
    m.flash_mca_forward(Z, V, U, gamma, beta, O_eager, C, causal, ws, stream)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(O_graph, O_eager)
    st, where = m.flash_mca_device_status()
    assert st == m.FMCA_OK, f"device status {st} at {where}"


@pytest.mark.parametrize("causal", [True, False])
def test_backward_graph_replay(causal):
    # the tensor-core backward (its launches chained by programmatic dependent
    # launch) and the CUDA-core one, captured and replayed
    m = fm()
    dev = torch.device("cuda:0")
    for (B, n, C, s, e, dtype) in ((2, 1024, 256, 128, 512, torch.bfloat16),
                                   (1, 256, 64, 32, 64, torch.float32)):
        Z, V, U, gamma, beta = (t.to(dev) for t in mca_inputs.make_inputs(B, n, s, e, 9, dtype))
        dO = torch.randn(B, n, e, generator=torch.Generator().manual_seed(4)).to(dtype).to(dev)
        code = m.FMCA_BF16 if dtype == torch.bfloat16 else m.FMCA_F32
        ws = torch.empty(m.flash_mca_backward_workspace_bytes(B, n, s, e, C, causal, code),
                         dtype=torch.uint8, device=dev)

        def outs():
            return (torch.empty_like(Z), torch.empty_like(V), torch.empty_like(U),
                    torch.empty(4, s, device=dev), torch.empty(4, s, device=dev))
        eager, graphed = outs(), outs()
        m.flash_mca_backward(Z, V, U, gamma, beta, dO, *eager, C, causal, ws)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            m.flash_mca_backward(Z, V, U, gamma, beta, dO, *graphed, C, causal, ws,
                                 stream=torch.cuda.current_stream(dev))
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(graphed, eager):
            assert torch.equal(a, b)
        st, where = m.flash_mca_device_status()
        assert st == m.FMCA_OK, f"device status {st} at {where}"
