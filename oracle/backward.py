"""fp64 CPU oracle of the BACKWARD pass of the mixed-chunk attention core.

TEST INFRASTRUCTURE ONLY (as the rest of ``oracle/``): only the test suite and
the benchmark's CPU legs may import it; the CUDA library never does, and the
two share no code.

The pages ("FLASH: Possibly the Most Interesting Efficient Transformer Design
Recently", section "Mixed Chunk") define the forward pass only.  Its gradient
is fixed by calculus: this module restates the forward definition with plain
fp64 torch operations, step by step in the pages' order, and lets
``torch.autograd`` differentiate it.  There is no blocking or reordering
beyond the definition:

  (1) T_k = Z * gamma[k] + beta[k], k = 0 quad_q, 1 quad_k, 2 lin_q, 3 lin_k
      ("Weak Attention", eq. relu-att; "Mixed Chunk", four affine maps);
  (2) chunks of C tokens ("Mixed Chunk", first paragraph);
  (3) quad_g = (quad_scale * relu(T0_g T1_g^T)^2, strict upper triangle masked
      in causal mode) V_g; quad_scale = 1/C^2 by default, i.e. relu(x/C)^2
      ("Mixed Chunk", eq. for V-hat^quad_g);
  (4) state_h = T3_h^T V_h; the global term of token t in chunk g is
      T2_t . (sum over h < g, or over all h) state_h / d(t), with d(t) = n,
      the tokens the sum covers, or t+1 (lin_norm 0, 1, 2), or no global term
      (lin_norm 3) ("Mixed Chunk", the non-causal and decoder equations;
      "Extended Thoughts", the divisor remark);
  (5) O = U * (quad + glob) ("Mixed Chunk", eq. for O_g).

``backward`` returns dZ, dV, dU, dgamma, dbeta for a given dO: the gradients
of sum(O * dO).  Pinned in tests/test_oracle_backward_pins.py by central
finite differences of the C oracle (mca_oracle.c, which shares nothing with
this file) and by its forward agreeing with the C oracle.
"""
from __future__ import annotations

import numpy as np
import torch


def _t64(x) -> torch.Tensor:
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64).clone()
    return torch.as_tensor(np.asarray(x, dtype=np.float64)).clone()


def forward_torch(Z, V, U, gamma, beta, C: int, causal: bool, quad_scale=None,
                  lin_norm: int = 0) -> torch.Tensor:
    """The forward definition in fp64 torch operations (differentiable)."""
    B, n, s = Z.shape
    e = V.shape[2]
    G = n // C
    qs = 1.0 / (C * C) if quad_scale is None else float(quad_scale)
    T = [Z * gamma[k] + beta[k] for k in range(4)]                        # (1)
    Tc = [t.reshape(B, G, C, s) for t in T]                               # (2)
    Vc = V.reshape(B, G, C, e)
    scores = torch.einsum("bgis,bgjs->bgij", Tc[0], Tc[1])                # (3)
    w = qs * torch.relu(scores) ** 2
    if causal:
        w = w * torch.tril(torch.ones(C, C, dtype=w.dtype))
    quad = torch.einsum("bgij,bgje->bgie", w, Vc)
    states = torch.einsum("bgcs,bgce->bgse", Tc[3], Vc)                   # (4)
    if causal:
        before = torch.cumsum(states, dim=1) - states                      # h < g
    else:
        before = states.sum(dim=1, keepdim=True).expand(B, G, s, e)        # all h
    pos = torch.arange(n, dtype=torch.float64).reshape(G, C)
    g_idx = torch.arange(G, dtype=torch.float64).reshape(G, 1).expand(G, C)
    if lin_norm == 0:
        inv = torch.full((G, C), 1.0 / n, dtype=torch.float64)
    elif lin_norm == 1:
        if causal:
            cnt = g_idx * C
            inv = torch.where(cnt > 0, 1.0 / torch.clamp(cnt, min=1.0), torch.zeros_like(cnt))
        else:
            inv = torch.full((G, C), 1.0 / n, dtype=torch.float64)
    elif lin_norm == 2:
        inv = 1.0 / (pos + 1.0)
    elif lin_norm == 3:
        inv = torch.zeros((G, C), dtype=torch.float64)
    else:
        raise ValueError(lin_norm)
    glob = torch.einsum("bgis,bgse->bgie", Tc[2], before) * inv[None, :, :, None]
    O = U * (quad + glob).reshape(B, n, e)                                 # (5)
    return O


def backward(Z, V, U, gamma, beta, dO, C: int, causal: bool, quad_scale=None,
             lin_norm: int = 0):
    """(dZ, dV, dU, dgamma, dbeta) as numpy fp64 arrays."""
    Zt, Vt, Ut, gt, bt = (_t64(x).requires_grad_(True) for x in (Z, V, U, gamma, beta))
    O = forward_torch(Zt, Vt, Ut, gt, bt, C, causal, quad_scale, lin_norm)
    grads = torch.autograd.grad(O, (Zt, Vt, Ut, gt, bt), grad_outputs=_t64(dO))
    return tuple(g.numpy() for g in grads)
