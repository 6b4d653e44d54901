"""Seeded synthetic inputs for the mixed-chunk attention forward core.

This module is shared by the tests, the benchmark and the smoke check.  It holds
none of the method's arithmetic: it only names the workloads and draws their
inputs.  Both the CUDA path and the CPU oracle receive exactly the tensors made
here (after the cast to the run dtype), so neither side generates its own data.

Recipe (the same for every workload):
  * a CPU ``torch.Generator`` seeded with ``seed`` draws, in this order and in
    fp32: Z ~ N(0,1) [B,n,s], V ~ N(0,1) [B,n,e], U ~ N(0,1) [B,n,e],
    gamma ~ N(0,1) [4,s], beta ~ N(0,1) [4,s];
  * Z, V and U go through SiLU (the GAU applies Swish/SiLU to its U, V and Z
    projections before the attention core: "FLASH: Possibly the Most
    Interesting Efficient Transformer Design Recently", sections "Initial
    Power" and "Weak Attention");
  * gamma = 1 + 0.1 * draw, beta = 0.1 * draw (rows: quad_q, quad_k, lin_q,
    lin_k), kept in fp32;
  * Z, V, U are then rounded to the run dtype (round-to-nearest-even for bf16).
"""
from __future__ import annotations

from dataclasses import dataclass, asdict

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    n: int
    C: int
    s: int
    e: int
    causal: bool
    dtype: str  # "f32" or "bf16"
    lin_norm: str = "n"  # global-term divisor: "n", "summed", "position" or "none"

    @property
    def G(self) -> int:
        return self.n // self.C

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def as_dict(self) -> dict:
        d = asdict(self)
        d["G"] = self.G
        return d


# The five workloads: a tiny fp32 case, the GAU-base language-model shape, a
# bidirectional (MLM-style) shape, a long causal shape and a very long causal
# shape (e = 2d with d = 768 or 1024, s = 128, chunk 256 as the paper uses).
WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_causal_f32", B=1, n=256, C=64, s=32, e=64, causal=True, dtype="f32"),
        Workload("gau_base_causal", B=8, n=1024, C=256, s=128, e=1536, causal=True, dtype="bf16"),
        Workload("bidir_mlm", B=4, n=4096, C=256, s=128, e=1536, causal=False, dtype="bf16"),
        Workload("long_causal", B=2, n=8192, C=256, s=128, e=1536, causal=True, dtype="bf16"),
        Workload("very_long_causal", B=1, n=32768, C=256, s=128, e=2048, causal=True, dtype="bf16"),
        # the quadratic-only model (FLASH-Quad) at the pages' base scale, sequence
        # length 1024: one chunk spanning the sequence, no global term
        Workload("flash_quad_base", B=8, n=1024, C=1024, s=128, e=1536, causal=True,
                 dtype="bf16", lin_norm="none"),
    ]
}
WORKLOAD_ORDER = list(WORKLOADS)


def make_inputs(B: int, n: int, s: int, e: int, seed: int, dtype: torch.dtype = torch.bfloat16):
    """Return (Z, V, U, gamma, beta) as CPU tensors; Z/V/U in ``dtype``,
    gamma/beta fp32 [4, s]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    Z = torch.randn((B, n, s), generator=g, dtype=torch.float32)
    V = torch.randn((B, n, e), generator=g, dtype=torch.float32)
    U = torch.randn((B, n, e), generator=g, dtype=torch.float32)
    gr = torch.randn((4, s), generator=g, dtype=torch.float32)
    br = torch.randn((4, s), generator=g, dtype=torch.float32)
    silu = torch.nn.functional.silu
    Z, V, U = silu(Z).to(dtype), silu(V).to(dtype), silu(U).to(dtype)
    gamma = (1.0 + 0.1 * gr).contiguous()
    beta = (0.1 * br).contiguous()
    return Z.contiguous(), V.contiguous(), U.contiguous(), gamma, beta


def workload_inputs(w: Workload, seed: int):
    return make_inputs(w.B, w.n, w.s, w.e, seed, w.torch_dtype)
