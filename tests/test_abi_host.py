"""Host-side tests of the C ABI: the library loads, exports every entry point
the header declares, sizes its workspace as documented and rejects bad
arguments before queuing any work.  No call here reaches the GPU: every call
with device pointers carries one argument the host checks refuse."""
from __future__ import annotations

import os
import re

import pytest

import flash_mixed_chunk_gb300 as fm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flash_mca.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(flash_mca_\w+)\s*\(", text)))


def test_header_declares_the_documented_entry_points():
    names = declared_functions()
    for must in ("flash_mca_forward", "flash_mca_workspace_bytes", "flash_mca_status_string",
                 "flash_mca_forward_host", "flash_mca_host_arena_bytes"):
        assert must in names


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    for name in names:
        assert hasattr(fm.lib, name), f"{name} declared in the header but not exported"
    assert sorted(fm.EXPORTED_SYMBOLS) == names, "binding and header disagree"


def test_library_is_in_tree_and_not_the_oracle():
    assert os.path.dirname(fm.library_path) == os.path.join(ROOT, "flash_mixed_chunk_gb300")
    # the product binding never imports the oracle
    src = open(os.path.join(ROOT, "flash_mixed_chunk_gb300", "__init__.py")).read()
    assert "oracle" not in src.replace("no CPU fallback", "")


def test_status_strings():
    for code in range(8):
        sname = fm.flash_mca_status_string(code)
        assert sname.startswith("FMCA_")
    assert "unknown" in fm.flash_mca_status_string(99)
    assert fm.flash_mca_version() == "0.1.0"


def walk_segments(B, n, e, C):
    """Segments of the chunk axis the tensor-core path's chunk walkers use:
    about 144 (sequence, 256 e columns, segment) units, every segment
    non-empty (the last slice of e may be narrower)."""
    G = n // C
    slices = B * (-(-e // 256))
    S = max(1, min(G, 144 // slices)) if slices else 1
    L = -(-G // S)
    return -(-G // L)


@pytest.mark.parametrize("B,n,s,e,C,causal", [(2, 8192, 128, 1536, 256, 1),
                                              (4, 4096, 128, 1536, 256, 0),
                                              (1, 256, 32, 64, 64, 1),
                                              (3, 96, 48, 80, 32, 0)])
def test_workspace_bytes_formula(B, n, s, e, C, causal):
    """Enough for either path: fp32 states and prefix (SIMT) or, on the tensor
    cores, the bf16 local sums of each chunk's segment (causal), the segment
    totals/carries, the work counters and the bf16 rows T0, T1, T2; no
    per-chunk states and no [B*n][C] buffer of relu^2 weights."""
    a = lambda x: (x + 255) // 256 * 256
    G = n // C
    Gp = G if causal else 1
    simt = a(4 * B * G * s * e) + a(4 * B * Gp * s * e)
    tc = (a(2 * B * G * s * e) * causal + a(2 * B * walk_segments(B, n, e, C) * s * e) + 256
          + a(3 * 2 * B * n * s))  # + the bf16 rows T0, T1, T2
    for dt in (fm.FMCA_F32, fm.FMCA_BF16):
        assert fm.flash_mca_workspace_bytes(B, n, s, e, C, causal, dt) == max(simt, tc)


def test_workspace_bytes_zero_for_rejected_shapes():
    assert fm.flash_mca_workspace_bytes(1, 100, 32, 64, 30, 1, fm.FMCA_F32) == 0   # C !| n
    assert fm.flash_mca_workspace_bytes(1, 64, 32, 64, 128, 1, fm.FMCA_F32) == 0   # C > n
    assert fm.flash_mca_workspace_bytes(0, 64, 32, 64, 64, 1, fm.FMCA_F32) == 0
    assert fm.flash_mca_workspace_bytes(1, 64, 512, 64, 64, 1, fm.FMCA_F32) == 0   # s > 256
    assert fm.flash_mca_workspace_bytes(1, 64, 32, 64, 64, 1, 7) == 0              # bad dtype


def test_auto_path_choice():
    bf, f32 = fm.FMCA_BF16, fm.FMCA_F32
    assert fm.flash_mca_auto_path(2, 8192, 128, 1536, 256, 1, bf) == fm.FMCA_PATH_TCGEN05
    assert fm.flash_mca_auto_path(1, 32768, 128, 2048, 256, 1, bf) == fm.FMCA_PATH_TCGEN05
    assert fm.flash_mca_auto_path(1, 256, 128, 256, 128, 0, bf) == fm.FMCA_PATH_TCGEN05
    assert fm.flash_mca_auto_path(2, 8192, 128, 1536, 256, 1, f32) == fm.FMCA_PATH_SIMT
    assert fm.flash_mca_auto_path(1, 256, 32, 64, 64, 1, f32) == fm.FMCA_PATH_SIMT
    assert fm.flash_mca_auto_path(1, 512, 64, 256, 256, 1, bf) == fm.FMCA_PATH_SIMT   # s != 128
    assert fm.flash_mca_auto_path(1, 512, 128, 200, 256, 1, bf) == fm.FMCA_PATH_SIMT  # e % 64
    # e a multiple of 64 but not of 256: the forward pass's own forms take it
    assert fm.flash_mca_auto_path(1, 512, 128, 640, 256, 1, bf) == fm.FMCA_PATH_TCGEN05
    assert fm.flash_mca_auto_path(1, 512, 128, 320, 256, 1, bf) == fm.FMCA_PATH_TCGEN05
    assert fm.flash_mca_auto_path(1, 512, 128, 256, 64, 1, bf) == fm.FMCA_PATH_SIMT   # C = 64
    assert fm.flash_mca_auto_path(1, 500, 128, 256, 64, 1, bf) == -1


def test_launch_counts():
    bf = fm.FMCA_BF16
    # chunks of 256: the segment walkers (local sums, totals, T rows), then
    # the row-pair kernel, which forms the segment carries (or, bidirectional,
    # the total) itself
    assert fm.flash_mca_launch_count(2, 8192, 128, 1536, 256, 1, bf) == 2
    assert fm.flash_mca_launch_count(4, 4096, 128, 1536, 256, 0, bf) == 2
    # chunks of 128, bidirectional: walkers, the total, the fused chunk kernel
    assert fm.flash_mca_launch_count(4, 4096, 128, 1536, 128, 0, bf) == 3
    # one segment per sequence (B * e / 256 >= 144 units): no carries
    assert fm.flash_mca_launch_count(16, 1024, 128, 2560, 256, 1, bf) == 2
    # without a global term: the T0 / T1 rows and the fused chunk kernel
    assert fm.flash_mca_launch_count(8, 1024, 128, 1536, 1024, 1, bf,
                                     lin_norm=fm.FMCA_LIN_NORM_NONE) == 2
    assert fm.flash_mca_launch_count(8, 1024, 128, 1536, 1024, 1, bf, fm.FMCA_PATH_SIMT,
                                     lin_norm=fm.FMCA_LIN_NORM_NONE) == 3
    assert fm.flash_mca_launch_count(2, 8192, 128, 1536, 256, 1, bf,
                                     lin_norm=fm.FMCA_LIN_NORM_POSITION) == 2
    assert fm.flash_mca_launch_count(2, 8192, 128, 1536, 256, 1, bf, fm.FMCA_PATH_SIMT) == 3
    assert fm.flash_mca_launch_count(1, 512, 64, 256, 256, 1, bf, fm.FMCA_PATH_TCGEN05) == 0
    # e % 256 != 0: every form but the stored-weights one (no global term,
    # chunks over 256 tokens), which goes to the CUDA cores
    assert fm.flash_mca_launch_count(2, 2048, 128, 640, 256, 1, bf) == 2
    assert fm.flash_mca_launch_count(2, 2048, 128, 640, 512, 1, bf, fm.FMCA_PATH_TCGEN05,
                                     lin_norm=fm.FMCA_LIN_NORM_NONE) == 0
    assert fm.flash_mca_launch_count(2, 2048, 128, 640, 512, 1, bf,
                                     lin_norm=fm.FMCA_LIN_NORM_NONE) == 3
    assert fm.flash_mca_launch_count(2, 2048, 128, 768, 512, 1, bf,
                                     lin_norm=fm.FMCA_LIN_NORM_NONE) == 2
    assert fm.flash_mca_launch_count(1, 500, 128, 256, 64, 1, bf) == 0


# A fake device address: aligned, never dereferenced (each call below fails a
# host check first).
P = 0x7F0000000000
BIG = 1 << 40


def fwd(**kw):
    args = dict(Z=P, V=P + 0x10000000, U=P + 0x20000000, g=P + 0x30000000, b=P + 0x30001000,
                O=P + 0x40000000, B=1, n=256, s=32, e=64, C=64, causal=1, dt=fm.FMCA_F32,
                ws=P + 0x50000000, wsb=BIG, path=fm.FMCA_PATH_AUTO)
    args.update(kw)
    return fm.lib.flash_mca_forward_path(args["Z"], args["V"], args["U"], args["g"], args["b"],
                                         args["O"], args["B"], args["n"], args["s"], args["e"],
                                         args["C"], args["causal"], args["dt"], args["ws"],
                                         args["wsb"], args["path"], None)


def test_validation_codes():
    assert fwd(C=60) == fm.FMCA_ERR_SHAPE
    assert fwd(C=512) == fm.FMCA_ERR_SHAPE
    assert fwd(B=0) == fm.FMCA_ERR_INVALID_ARG
    assert fwd(e=-1) == fm.FMCA_ERR_INVALID_ARG
    assert fwd(dt=5) == fm.FMCA_ERR_INVALID_ARG
    assert fwd(path=9) == fm.FMCA_ERR_INVALID_ARG
    assert fwd(Z=0) == fm.FMCA_ERR_INVALID_ARG
    assert fwd(O=0) == fm.FMCA_ERR_INVALID_ARG
    assert fwd(g=0) == fm.FMCA_ERR_INVALID_ARG
    assert fwd(s=300) == fm.FMCA_ERR_UNSUPPORTED
    assert fwd(V=P + 0x10000008) == fm.FMCA_ERR_ALIGN
    assert fwd(O=P + 0x40000004) == fm.FMCA_ERR_ALIGN
    assert fwd(ws=0) == fm.FMCA_ERR_WORKSPACE
    assert fwd(ws=P + 0x50000010) == fm.FMCA_ERR_ALIGN
    assert fwd(wsb=100) == fm.FMCA_ERR_WORKSPACE
    # O overlapping an input or the workspace
    assert fwd(O=P + 0x10000000) == fm.FMCA_ERR_INVALID_ARG
    assert fwd(O=P + 0x50000000) == fm.FMCA_ERR_INVALID_ARG
    # explicit tensor-core path on a shape it does not cover: no fallback
    assert fwd(path=fm.FMCA_PATH_TCGEN05) == fm.FMCA_ERR_UNSUPPORTED
    assert fwd(dt=fm.FMCA_BF16, s=64, e=256, n=512, C=256,
               path=fm.FMCA_PATH_TCGEN05) == fm.FMCA_ERR_UNSUPPORTED


def test_host_entry_validation():
    f = fm.lib.flash_mca_forward_host
    good = dict(B=1, n=256, s=32, e=64, C=64, causal=1, dt=fm.FMCA_F32)
    need = fm.flash_mca_host_arena_bytes(1, 256, 32, 64, 64, 1, fm.FMCA_F32)
    assert need > fm.flash_mca_workspace_bytes(1, 256, 32, 64, 64, 1, fm.FMCA_F32)
    h = P  # host pointers are never touched either
    assert f(h, h, h, h, h, h, 1, 256, 32, 64, 60, 1, fm.FMCA_F32, P, need, None) == fm.FMCA_ERR_SHAPE
    assert f(0, h, h, h, h, h, 1, 256, 32, 64, 64, 1, fm.FMCA_F32, P, need, None) == fm.FMCA_ERR_INVALID_ARG
    assert f(h, h, h, h, h, h, 1, 256, 32, 64, 64, 1, fm.FMCA_F32, 0, need, None) == fm.FMCA_ERR_WORKSPACE
    assert f(h, h, h, h, h, h, 1, 256, 32, 64, 64, 1, fm.FMCA_F32, P, need - 1, None) == fm.FMCA_ERR_WORKSPACE
    assert f(h, h, h, h, h, h, 1, 256, 32, 64, 64, 1, fm.FMCA_F32, P + 16, need, None) == fm.FMCA_ERR_ALIGN


def test_selftest_rejects_bad_limits():
    assert fm.lib.flash_mca_selftest_timeout(0, None) == fm.FMCA_ERR_INVALID_ARG
    assert fm.lib.flash_mca_selftest_timeout(20_000_000, None) == fm.FMCA_ERR_INVALID_ARG


def test_python_binding_rejects_bad_tensors():
    import torch
    Z = torch.zeros(1, 256, 32)
    V = torch.zeros(1, 256, 64)
    with pytest.raises(ValueError):
        fm.flash_mca_forward(Z, V, V, torch.zeros(4, 32), torch.zeros(4, 32), V, 64, True, Z)
    with pytest.raises(ValueError):
        fm.forward(Z[0], V, V, torch.zeros(4, 32), torch.zeros(4, 32), 64, True)


def fwd_ex(opts, **kw):
    args = dict(Z=P, V=P + 0x10000000, U=P + 0x20000000, g=P + 0x30000000, b=P + 0x30001000,
                O=P + 0x40000000, B=1, n=256, s=32, e=64, C=64, causal=1, dt=fm.FMCA_F32,
                ws=P + 0x50000000, wsb=BIG, path=fm.FMCA_PATH_AUTO)
    args.update(kw)
    return fm.lib.flash_mca_forward_ex(args["Z"], args["V"], args["U"], args["g"], args["b"],
                                       args["O"], args["B"], args["n"], args["s"], args["e"],
                                       args["C"], args["causal"], args["dt"], args["ws"],
                                       args["wsb"], args["path"], opts, None)


def test_default_options():
    import ctypes
    o = fm.FmcaOptions()
    assert fm.lib.flash_mca_default_options(256, ctypes.byref(o)) == fm.FMCA_OK
    assert o.quad_scale == 1.0 / 65536.0 and o.lin_norm == fm.FMCA_LIN_NORM_N
    assert fm.lib.flash_mca_default_options(0, ctypes.byref(o)) == fm.FMCA_ERR_INVALID_ARG
    assert fm.lib.flash_mca_default_options(64, None) == fm.FMCA_ERR_INVALID_ARG


def test_options_validation_codes():
    import ctypes
    for q, ln in ((-1.0, 0), (float("nan"), 0), (float("inf"), 0), (0.5, 4), (0.5, -1)):
        o = fm.FmcaOptions(q, ln)
        assert fwd_ex(ctypes.byref(o)) == fm.FMCA_ERR_INVALID_ARG, (q, ln)
    # valid options still go through the other host checks first
    o = fm.FmcaOptions(0.25, fm.FMCA_LIN_NORM_POSITION)
    assert fwd_ex(ctypes.byref(o), C=60) == fm.FMCA_ERR_SHAPE
    assert fwd_ex(ctypes.byref(o), ws=0) == fm.FMCA_ERR_WORKSPACE
    assert fwd_ex(None, V=P + 0x10000008) == fm.FMCA_ERR_ALIGN


def test_decode_state_bytes_and_validation():
    import ctypes
    nb = fm.flash_mca_decode_state_bytes(2, 32, 64, 16, fm.FMCA_F32)
    a = lambda x: (x + 255) // 256 * 256
    assert nb == a(4 * 2 * 32 * 64) + a(4 * 2 * 16 * 32) + a(4 * 2 * 16 * 64)
    # bf16: the fp32 sum, its bf16 copy, and the bf16 chunk cache
    assert fm.flash_mca_decode_state_bytes(2, 32, 64, 16, fm.FMCA_BF16) == \
        a(4 * 2 * 32 * 64) + a(2 * 2 * 32 * 64) + a(2 * 2 * 16 * 32) + a(2 * 2 * 16 * 64)
    for bad in ((0, 32, 64, 16), (2, 300, 64, 16), (2, 32, 64, 2048), (2, 32, 0, 16)):
        assert fm.flash_mca_decode_state_bytes(*bad, fm.FMCA_F32) == 0
    step = fm.lib.flash_mca_decode_step
    base = dict(z=P, v=P + 0x1000, u=P + 0x2000, g=P + 0x3000, b=P + 0x4000, o=P + 0x5000,
                B=2, s=32, e=64, C=16, t=5, n=64, dt=fm.FMCA_F32, opts=None,
                st=P + 0x100000, stb=nb)

    def call(**kw):
        d = dict(base)
        d.update(kw)
        return step(d["z"], d["v"], d["u"], d["g"], d["b"], d["o"], d["B"], d["s"], d["e"], d["C"],
                    d["t"], d["n"], d["dt"], d["opts"], d["st"], d["stb"], None)
    assert call(t=-1) == fm.FMCA_ERR_INVALID_ARG
    assert call(n=5) == fm.FMCA_ERR_INVALID_ARG          # n_norm must exceed t
    assert call(C=4096) == fm.FMCA_ERR_INVALID_ARG
    assert call(z=0) == fm.FMCA_ERR_INVALID_ARG
    assert call(v=P + 0x1004) == fm.FMCA_ERR_ALIGN
    assert call(stb=nb - 1) == fm.FMCA_ERR_WORKSPACE
    assert call(st=0) == fm.FMCA_ERR_WORKSPACE
    assert call(st=P + 0x100010) == fm.FMCA_ERR_ALIGN
    assert call(o=P + 0x1000) == fm.FMCA_ERR_INVALID_ARG    # o overlaps v
    o = fm.FmcaOptions(0.1, 7)
    assert call(opts=ctypes.byref(o)) == fm.FMCA_ERR_INVALID_ARG
    # the per-position and tokens-summed divisors do not need n_norm
    o = fm.FmcaOptions(0.1, fm.FMCA_LIN_NORM_SUMMED)
    assert call(opts=ctypes.byref(o), n=0, stb=0) == fm.FMCA_ERR_WORKSPACE
    reset = fm.lib.flash_mca_decode_reset
    assert reset(P + 0x100000, nb - 1, 2, 32, 64, 16, fm.FMCA_F32, None) == fm.FMCA_ERR_WORKSPACE
    assert reset(P + 0x100010, nb, 2, 32, 64, 16, fm.FMCA_F32, None) == fm.FMCA_ERR_ALIGN
    assert reset(P + 0x100000, nb, 0, 32, 64, 16, fm.FMCA_F32, None) == fm.FMCA_ERR_INVALID_ARG


def test_backward_workspace_and_validation():
    nb = fm.flash_mca_backward_workspace_bytes(2, 64, 16, 32, 16, 1, fm.FMCA_F32)
    a = lambda x: (x + 255) // 256 * 256
    G, rows = 4, 128
    want = (a(4 * 2 * G * 16 * 32) * 3 + a(4 * rows * 32) + 2 * a(4 * 2 * G * 16 * 16) +
            a(4 * 4 * rows * 16) + a(4 * 8 * 16 * 2))
    assert nb == want
    assert fm.flash_mca_backward_workspace_bytes(2, 64, 16, 32, 60, 1, fm.FMCA_F32) == 0
    f = fm.lib.flash_mca_backward
    base = dict(Z=P, V=P + 0x10000, U=P + 0x20000, g=P + 0x30000, b=P + 0x31000, dO=P + 0x40000,
                dZ=P + 0x50000, dV=P + 0x60000, dU=P + 0x70000, dg=P + 0x80000, db=P + 0x81000,
                B=2, n=64, s=16, e=32, C=16, causal=1, dt=fm.FMCA_F32, opts=None,
                ws=P + 0x100000, wsb=nb)

    def call(**kw):
        d = dict(base)
        d.update(kw)
        return f(d["Z"], d["V"], d["U"], d["g"], d["b"], d["dO"], d["dZ"], d["dV"], d["dU"],
                 d["dg"], d["db"], d["B"], d["n"], d["s"], d["e"], d["C"], d["causal"], d["dt"],
                 d["opts"], d["ws"], d["wsb"], None)
    assert call(C=60) == fm.FMCA_ERR_SHAPE
    assert call(dO=0) == fm.FMCA_ERR_INVALID_ARG
    assert call(dg=0) == fm.FMCA_ERR_INVALID_ARG
    assert call(dV=P + 0x60004) == fm.FMCA_ERR_ALIGN
    assert call(ws=0) == fm.FMCA_ERR_WORKSPACE
    assert call(wsb=nb - 1) == fm.FMCA_ERR_WORKSPACE
    assert call(ws=P + 0x100010) == fm.FMCA_ERR_ALIGN
    assert call(dZ=P + 0x10000) == fm.FMCA_ERR_INVALID_ARG   # dZ overlaps V
    assert call(dU=P + 0x60000) == fm.FMCA_ERR_INVALID_ARG   # dU overlaps dV
    import ctypes
    o = fm.FmcaOptions(0.1, 9)
    assert call(opts=ctypes.byref(o)) == fm.FMCA_ERR_INVALID_ARG


def test_gau_projection_validation():
    f = fm.lib.flash_mca_gau_project
    X, W, U, V, Z = P, P + 0x100000, P + 0x200000, P + 0x300000, P + 0x400000
    assert f(0, W, U, V, Z, 128, 64, 64, 64, None) == fm.FMCA_ERR_INVALID_ARG
    assert f(X, W, U, V, Z, 0, 64, 64, 64, None) == fm.FMCA_ERR_INVALID_ARG
    assert f(X, W, U, V, Z, 128, 60, 64, 64, None) == fm.FMCA_ERR_UNSUPPORTED   # d % 8
    assert f(X, W, U, V, Z, 128, 64, 96, 64, None) == fm.FMCA_ERR_UNSUPPORTED   # e % 64
    assert f(X, W, U, V, Z, 128, 64, 64, 32, None) == fm.FMCA_ERR_UNSUPPORTED   # s % 64
    assert f(X + 8, W, U, V, Z, 128, 64, 64, 64, None) == fm.FMCA_ERR_ALIGN
    assert f(X, W, X, V, Z, 128, 64, 64, 64, None) == fm.FMCA_ERR_INVALID_ARG   # U overlaps X
    assert f(X, W, U, U, Z, 128, 64, 64, 64, None) == fm.FMCA_ERR_INVALID_ARG   # V overlaps U
    g = fm.lib.flash_mca_gau_output
    assert g(X, W, U, 128, 64, 96, None) == fm.FMCA_ERR_UNSUPPORTED             # d % 64
    assert g(X, W, X, 128, 64, 64, None) == fm.FMCA_ERR_INVALID_ARG             # Out overlaps Y
    assert g(X, W, U + 4, 128, 64, 64, None) == fm.FMCA_ERR_ALIGN


def test_backward_saved_validation():
    # the saved mode exists for the tensor-core shapes only: fp32, or bf16 with
    # s != 128, is refused before any pointer is looked at
    f = fm.lib.flash_mca_backward_saved

    def call(B, n, s, e, C, dt):
        return f(P, P, P, P, P, P, P, P, P, P, P, B, n, s, e, C, 1, dt, None, P, 1 << 30, None)
    assert call(2, 64, 16, 32, 16, fm.FMCA_F32) == fm.FMCA_ERR_UNSUPPORTED
    assert call(1, 512, 64, 256, 256, fm.FMCA_BF16) == fm.FMCA_ERR_UNSUPPORTED
    assert call(1, 512, 128, 200, 256, fm.FMCA_BF16) == fm.FMCA_ERR_UNSUPPORTED
    assert call(2, 64, 16, 32, 60, fm.FMCA_F32) == fm.FMCA_ERR_SHAPE   # C does not divide n


def test_backward_launch_count():
    bf, f32 = fm.FMCA_BF16, fm.FMCA_F32
    cnt = fm.flash_mca_backward_launch_count
    # tensor cores: forward kernels (chunk walkers, segment carries, scaled
    # prefix, relu^2 weights, output kernel: 5; 3 when the forward pass's local
    # sums and carries are kept; 2 without a global term), 2 elementwise, 3
    # product launches, the reverse scan (global term only), 2 for dZ /
    # dgamma / dbeta
    assert cnt(2, 1024, 128, 512, 256, True, bf) == 13
    assert cnt(2, 1024, 128, 512, 256, True, bf, saved=True) == 11
    assert cnt(2, 1024, 128, 512, 256, True, bf, lin_norm=fm.FMCA_LIN_NORM_NONE) == 9
    # CUDA cores
    assert cnt(2, 1024, 128, 512, 256, True, f32) == 12
    assert cnt(2, 1024, 128, 512, 256, True, f32, lin_norm=fm.FMCA_LIN_NORM_NONE) == 7
    assert cnt(2, 1024, 128, 512, 256, True, f32, saved=True) == 0
    assert cnt(2, 1024, 128, 512, 60, True, bf) == 0        # C does not divide n


def test_forward_seq_rejects_before_queueing():
    """flash_mca_forward_seq checks its arguments on the host before anything is
    queued: bidirectional attention and the no-global-term variant are not
    covered, the piece must start on a chunk boundary, state pointers must be
    16-byte aligned and state_out must not overlap the other buffers.  The
    pointers here are never dereferenced."""
    import ctypes
    B, n, s, e, C = 1, 512, 128, 256, 256
    P = 0x7F0000000000
    z, v, u, g, b, o = P, P + (1 << 24), P + (2 << 24), P + (3 << 24), P + (3 << 24) + 4096, P + (4 << 24)
    ws = P + (8 << 24)
    nb = fm.flash_mca_workspace_bytes(B, n, s, e, C, 1, fm.FMCA_BF16)
    opts = fm.flash_mca_default_options(C)
    state = P + (16 << 24)

    def call(causal, offset, lin_norm=fm.FMCA_LIN_NORM_N, s_in=state, s_out=state, dt=fm.FMCA_BF16):
        opts.lin_norm = lin_norm
        seq = fm.FmcaSeq(s_in, s_out, offset, 0)
        return fm.lib.flash_mca_forward_seq(z, v, u, g, b, o, B, n, s, e, C, causal, dt, ws, nb,
                                            ctypes.byref(opts), ctypes.byref(seq), None)
    assert call(0, 0) == fm.FMCA_ERR_UNSUPPORTED                      # bidirectional
    assert call(1, 0, lin_norm=fm.FMCA_LIN_NORM_NONE) == fm.FMCA_ERR_UNSUPPORTED
    assert call(1, 0, dt=fm.FMCA_F32) != fm.FMCA_OK                   # not the tensor-core path
    assert call(1, 128) == fm.FMCA_ERR_INVALID_ARG                    # off a chunk boundary
    assert call(1, -256) == fm.FMCA_ERR_INVALID_ARG
    assert call(1, 0, s_in=state + 4) == fm.FMCA_ERR_ALIGN
    assert call(1, 0, s_out=o) == fm.FMCA_ERR_INVALID_ARG             # state_out overlaps O
