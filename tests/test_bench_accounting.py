"""The benchmark's accounting, pinned to hand-computed figures (CPU only):
the algorithmic FLOPs and compulsory bytes of a forward pass, the decode
step's byte model, and how the rotating buffer sets relate to L2."""
from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import mca_inputs  # noqa: E402

W = mca_inputs.WORKLOADS


def test_long_causal_flops_and_bytes():
    w = W["long_causal"]
    # per chunk: 2 P (s + e) over the P = C (C + 1) / 2 unmasked pairs, plus
    # 4 C s e for the chunk state and the global term; 64 chunks
    P = 256 * 257 // 2
    per_chunk = 2 * P * (128 + 1536) + 4 * 256 * 128 * 1536
    assert bench.algorithmic_flops(w) == pytest.approx(per_chunk * 64)
    assert bench.algorithmic_flops(w) == pytest.approx(19.89e9, rel=1e-3)
    # Z, V, U read once and O written once, bf16: (s + 3 e) * 2 bytes a token
    assert bench.algorithmic_bytes(w) == 2 * 8192 * (128 + 3 * 1536) * 2
    assert bench.algorithmic_bytes(w) / (2 * 8192) == 9472


def test_flops_variants():
    w = W["bidir_mlm"]           # bidirectional: all C^2 pairs
    per_chunk = 2 * 256 * 256 * (128 + 1536) + 4 * 256 * 128 * 1536
    assert bench.algorithmic_flops(w) == pytest.approx(per_chunk * 4 * 16)
    q = W["flash_quad_base"]     # no global term (lin_norm 3): the quad part only
    P = 1024 * 1025 // 2
    assert bench.algorithmic_flops(q, 3) == pytest.approx(2 * P * (128 + 1536) * 8)


def test_decode_bytes_model():
    s, e, C = 128, 1536, 256
    # index 0: the bf16 state copy, no cached rows, the token's z, v, u and o
    assert bench.decode_bytes_per_token(s, e, C, 0) == 2 * s * e + 2 * (s + 3 * e)
    # index 10: ten cached Z and V rows more
    assert bench.decode_bytes_per_token(s, e, C, 10) == \
        2 * s * e + 2 * 10 * (s + e) + 2 * (s + 3 * e)
    # the chunk's last token also folds: the cache once, the fp32 sum read and
    # written, the bf16 copy written
    last = bench.decode_bytes_per_token(s, e, C, C - 1)
    assert last == 2 * s * e + 2 * (C - 1) * (s + e) + 2 * (s + 3 * e) + \
        2 * C * (s + e) + 10 * s * e


def test_l2_note():
    assert bench.l2_note(W["long_causal"]).startswith("inputs larger than L2")
    assert "together larger than L2" in bench.l2_note(W["gau_base_causal"])
    assert "L2-resident" in bench.l2_note(W["tiny_causal_f32"])
