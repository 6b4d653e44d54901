"""Python binding of ``libflash_mca.so`` -- the FLASH mixed-chunk attention
forward core on GB300 (sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/flash_mca.h``; the functions
here take torch tensors (device memory, streams) and pass raw pointers and
sizes to the entry points of the same names.  There is no CPU fallback: if the
shared library is missing or fails to load, importing this package raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _buildlib as _build

__all__ = [
    "FMCA_OK", "FMCA_ERR_INVALID_ARG", "FMCA_ERR_SHAPE", "FMCA_ERR_UNSUPPORTED", "FMCA_ERR_ALIGN",
    "FMCA_ERR_WORKSPACE", "FMCA_ERR_CUDA", "FMCA_ERR_TIMEOUT", "FMCA_F32", "FMCA_BF16",
    "FMCA_PATH_AUTO", "FMCA_PATH_SIMT", "FMCA_PATH_TCGEN05", "FmcaError", "lib", "library_path",
    "flash_mca_workspace_bytes", "flash_mca_forward", "flash_mca_forward_path",
    "flash_mca_forward_timed",
    "flash_mca_auto_path", "flash_mca_launch_count", "flash_mca_launch_count_ex",
    "flash_mca_host_arena_bytes",
    "flash_mca_forward_host", "flash_mca_forward_noalloc", "flash_mca_device_status",
    "flash_mca_selftest_timeout", "FMCA_NOALLOC_SCRATCH_BYTES",
    "flash_mca_status_string", "flash_mca_version", "forward", "EXPORTED_SYMBOLS",
    "FMCA_LIN_NORM_N", "FMCA_LIN_NORM_SUMMED", "FMCA_LIN_NORM_POSITION", "FMCA_LIN_NORM_NONE",
    "FmcaOptions",
    "flash_mca_default_options", "flash_mca_forward_ex", "flash_mca_forward_seq", "FmcaSeq",
    "flash_mca_decode_state_bytes",
    "flash_mca_decode_reset", "flash_mca_decode_step", "flash_mca_backward_workspace_bytes",
    "flash_mca_backward", "flash_mca_backward_saved", "flash_mca_backward_launch_count",
    "backward", "flash_mca_gau_project",
    "flash_mca_gau_output",
    "gau_project", "gau_output",
]

FMCA_OK, FMCA_ERR_INVALID_ARG, FMCA_ERR_SHAPE, FMCA_ERR_UNSUPPORTED = 0, 1, 2, 3
FMCA_ERR_ALIGN, FMCA_ERR_WORKSPACE, FMCA_ERR_CUDA, FMCA_ERR_TIMEOUT = 4, 5, 6, 7
FMCA_F32, FMCA_BF16 = 0, 1
FMCA_PATH_AUTO, FMCA_PATH_SIMT, FMCA_PATH_TCGEN05 = 0, 1, 2
# global-term divisors of flash_mca_forward_ex: n; the tokens the sum covers;
# the token's position counted from 1
FMCA_LIN_NORM_N, FMCA_LIN_NORM_SUMMED, FMCA_LIN_NORM_POSITION = 0, 1, 2
FMCA_LIN_NORM_NONE = 3  # no global term (with C = n: FLASH-Quad)
FMCA_NOALLOC_SCRATCH_BYTES = 64 << 20  # size of the fixed scratch of flash_mca_forward_noalloc

library_path = _build.LIB

# Build (or rebuild, when a source is newer) the in-tree library; without it
# the package does not import -- there is no CPU fallback.
try:
    _build.build()
except Exception as exc:  # nvcc missing or the build failed
    if not os.path.exists(library_path):
        raise ImportError(f"{library_path} is missing and could not be built: {exc}") from exc
    raise ImportError(f"{library_path} is out of date and could not be rebuilt: {exc}") from exc
lib = ctypes.CDLL(library_path)

_vp, _sz, _i32, _cp = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_char_p
_int = ctypes.c_int
_fwd_args = [_vp, _vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _int, _int, _i32, _vp, _sz]


class FmcaOptions(ctypes.Structure):
    """``fmca_options`` of the header: intra-chunk weights quad_scale *
    relu(q . k)^2 and the global-term divisor lin_norm (FMCA_LIN_NORM_*)."""
    _fields_ = [("quad_scale", ctypes.c_float), ("lin_norm", _i32)]


class FmcaSeq(ctypes.Structure):
    """``fmca_seq`` of the header: one piece of longer causal sequences
    (carried-in state, state out, the piece's first token, the divisor's
    length)."""
    _fields_ = [("state_in", _vp), ("state_out", _vp), ("token_offset", ctypes.c_int64),
                ("n_norm", ctypes.c_int64)]


# (name, restype, argtypes) for every symbol the header declares
_SIGNATURES = [
    ("flash_mca_workspace_bytes", _sz, [_int] * 6 + [_i32]),
    ("flash_mca_forward", _i32, _fwd_args + [_vp]),
    ("flash_mca_forward_path", _i32, _fwd_args + [_i32, _vp]),
    ("flash_mca_default_options", _i32, [_int, ctypes.POINTER(FmcaOptions)]),
    ("flash_mca_forward_timed", _i32, _fwd_args + [_i32, ctypes.POINTER(FmcaOptions),
                                                   ctypes.POINTER(_vp), _int, _vp]),
    ("flash_mca_forward_ex", _i32, _fwd_args + [_i32, ctypes.POINTER(FmcaOptions), _vp]),
    ("flash_mca_forward_seq", _i32, _fwd_args + [ctypes.POINTER(FmcaOptions),
                                                 ctypes.POINTER(FmcaSeq), _vp]),
    ("flash_mca_decode_state_bytes", _sz, [_int] * 4 + [_i32]),
    ("flash_mca_backward_workspace_bytes", _sz, [_int] * 6 + [_i32]),
    ("flash_mca_gau_project", _i32, [_vp] * 5 + [_int] * 4 + [_vp]),
    ("flash_mca_gau_output", _i32, [_vp] * 3 + [_int] * 3 + [_vp]),
    ("flash_mca_backward", _i32, [_vp] * 11 + [_int] * 6 + [_i32, ctypes.POINTER(FmcaOptions),
                                                          _vp, _sz, _vp]),
    ("flash_mca_backward_saved", _i32, [_vp] * 11 + [_int] * 6 +
     [_i32, ctypes.POINTER(FmcaOptions), _vp, _sz, _vp]),
    ("flash_mca_backward_launch_count", _int,
     [_int] * 6 + [_i32, ctypes.POINTER(FmcaOptions), _int]),
    ("flash_mca_decode_reset", _i32, [_vp, _sz] + [_int] * 4 + [_i32, _vp]),
    ("flash_mca_decode_step", _i32, [_vp] * 6 + [_int] * 6 + [_i32, ctypes.POINTER(FmcaOptions),
                                                             _vp, _sz, _vp]),
    ("flash_mca_auto_path", _int, [_int] * 6 + [_i32]),
    ("flash_mca_launch_count", _int, [_int] * 6 + [_i32, _i32]),
    ("flash_mca_launch_count_ex", _int, [_int] * 6 + [_i32, _i32, ctypes.POINTER(FmcaOptions)]),
    ("flash_mca_host_arena_bytes", _sz, [_int] * 6 + [_i32]),
    ("flash_mca_forward_host", _i32, _fwd_args + [_vp]),
    ("flash_mca_forward_noalloc", _i32, _fwd_args[:13] + [_vp]),
    ("flash_mca_device_status", _i32, [_vp, ctypes.POINTER(_i32)]),
    ("flash_mca_selftest_timeout", _i32, [_int, _vp]),
    ("flash_mca_status_string", _cp, [_i32]),
    ("flash_mca_version", _cp, []),
]
EXPORTED_SYMBOLS = [name for name, _, _ in _SIGNATURES]
for _name, _res, _args in _SIGNATURES:
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args


class FmcaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        msg = lib.flash_mca_status_string(self.status).decode()
        super().__init__(f"{what}: {msg}" if what else msg)


def _check(status: int, what: str) -> None:
    if status != FMCA_OK:
        raise FmcaError(status, what)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return FMCA_BF16
    if t.dtype == torch.float32:
        return FMCA_F32
    raise TypeError(f"unsupported dtype {t.dtype}: use torch.bfloat16 or torch.float32")


def _stream_ptr(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def flash_mca_status_string(status: int) -> str:
    return lib.flash_mca_status_string(int(status)).decode()


def flash_mca_version() -> str:
    return lib.flash_mca_version().decode()


def flash_mca_workspace_bytes(B: int, n: int, s: int, e: int, C: int, causal: bool,
                              dtype: int) -> int:
    return int(lib.flash_mca_workspace_bytes(B, n, s, e, C, int(bool(causal)), dtype))


def flash_mca_host_arena_bytes(B: int, n: int, s: int, e: int, C: int, causal: bool,
                               dtype: int) -> int:
    return int(lib.flash_mca_host_arena_bytes(B, n, s, e, C, int(bool(causal)), dtype))


def flash_mca_auto_path(B: int, n: int, s: int, e: int, C: int, causal: bool, dtype: int) -> int:
    return int(lib.flash_mca_auto_path(B, n, s, e, C, int(bool(causal)), dtype))


def flash_mca_launch_count(B: int, n: int, s: int, e: int, C: int, causal: bool, dtype: int,
                           path: int = FMCA_PATH_AUTO, quad_scale: float | None = None,
                           lin_norm: int | None = None) -> int:
    """Kernels one forward call launches; with ``quad_scale`` or ``lin_norm``
    given, the count of flash_mca_forward_ex with those options."""
    if quad_scale is None and lin_norm is None:
        return int(lib.flash_mca_launch_count(B, n, s, e, C, int(bool(causal)), dtype, path))
    opts = flash_mca_default_options(C)
    if quad_scale is not None:
        opts.quad_scale = float(quad_scale)
    if lin_norm is not None:
        opts.lin_norm = int(lin_norm)
    return int(lib.flash_mca_launch_count_ex(B, n, s, e, C, int(bool(causal)), dtype, path,
                                             ctypes.byref(opts)))


def _shapes(Z: torch.Tensor, V: torch.Tensor, U: torch.Tensor):
    if Z.dim() != 3 or V.dim() != 3 or U.dim() != 3:
        raise ValueError("Z, V, U must be 3-D: [B, n, s], [B, n, e], [B, n, e]")
    B, n, s = Z.shape
    e = V.shape[2]
    if tuple(V.shape) != (B, n, e) or tuple(U.shape) != (B, n, e):
        raise ValueError("V and U must be [B, n, e] with Z [B, n, s]")
    return B, n, s, e


def flash_mca_default_options(C: int) -> FmcaOptions:
    opts = FmcaOptions()
    _check(lib.flash_mca_default_options(int(C), ctypes.byref(opts)), "flash_mca_default_options")
    return opts


def _check_device_args(Z, V, U, gamma, beta, O, workspace):
    B, n, s, e = _shapes(Z, V, U)
    for name, t in (("Z", Z), ("V", V), ("U", U), ("O", O), ("gamma", gamma), ("beta", beta),
                    ("workspace", workspace)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if gamma.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("gamma and beta must be float32 [4, s]")
    if tuple(gamma.shape) != (4, s) or tuple(beta.shape) != (4, s):
        raise ValueError("gamma and beta must be [4, s]")
    dt = _dtype_code(Z)
    if V.dtype != Z.dtype or U.dtype != Z.dtype or O.dtype != Z.dtype:
        raise TypeError("Z, V, U and O must share one dtype")
    if tuple(O.shape) != (B, n, e):
        raise ValueError("O must be [B, n, e]")
    return B, n, s, e, dt, workspace.numel() * workspace.element_size()


def flash_mca_forward_path(Z, V, U, gamma, beta, O, C: int, causal: bool, workspace,
                           path: int = FMCA_PATH_AUTO, stream=None) -> None:
    """Queue the forward pass on ``stream`` (default: torch's current stream)
    with an explicit kernel path; all tensors are CUDA tensors the caller
    owns."""
    B, n, s, e, dt, ws_bytes = _check_device_args(Z, V, U, gamma, beta, O, workspace)
    st = lib.flash_mca_forward_path(Z.data_ptr(), V.data_ptr(), U.data_ptr(), gamma.data_ptr(),
                                    beta.data_ptr(), O.data_ptr(), B, n, s, e, int(C),
                                    int(bool(causal)), dt, workspace.data_ptr(), ws_bytes, path,
                                    _stream_ptr(stream))
    _check(st, "flash_mca_forward_path")


def flash_mca_forward_ex(Z, V, U, gamma, beta, O, C: int, causal: bool, workspace,
                         quad_scale: float | None = None, lin_norm: int = FMCA_LIN_NORM_N,
                         path: int = FMCA_PATH_AUTO, stream=None) -> None:
    """``flash_mca_forward_path`` with the scale and normalisation variants:
    intra-chunk weights quad_scale * relu(q . k)^2 (default 1/C^2) and the
    global-term divisor ``lin_norm`` (FMCA_LIN_NORM_*)."""
    B, n, s, e, dt, ws_bytes = _check_device_args(Z, V, U, gamma, beta, O, workspace)
    opts = flash_mca_default_options(C)
    if quad_scale is not None:
        opts.quad_scale = float(quad_scale)
    opts.lin_norm = int(lin_norm)
    st = lib.flash_mca_forward_ex(Z.data_ptr(), V.data_ptr(), U.data_ptr(), gamma.data_ptr(),
                                  beta.data_ptr(), O.data_ptr(), B, n, s, e, int(C),
                                  int(bool(causal)), dt, workspace.data_ptr(), ws_bytes, path,
                                  ctypes.byref(opts), _stream_ptr(stream))
    _check(st, "flash_mca_forward_ex")


def flash_mca_forward_seq(Z, V, U, gamma, beta, O, C: int, workspace, state_in=None,
                          state_out=None, token_offset: int = 0, n_norm: int = 0,
                          quad_scale: float | None = None, lin_norm: int = FMCA_LIN_NORM_N,
                          stream=None) -> None:
    """``flash_mca_forward_seq``: the causal forward pass on one piece of
    longer sequences.  ``state_in`` / ``state_out``: fp32 CUDA tensors
    [B][s][e] (or None), the sum of T3^T V over the chunks before the piece and
    after it; ``token_offset``: the piece's first token (a multiple of C);
    ``n_norm``: the divisor's length (0: the piece's n)."""
    B, n, s, e, dt, ws_bytes = _check_device_args(Z, V, U, gamma, beta, O, workspace)
    for name, t in (("state_in", state_in), ("state_out", state_out)):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != (B, s, e)
                              or not t.is_contiguous() or t.device != Z.device):
            raise ValueError(f"{name} must be a contiguous float32 [B, s, e] tensor on "
                             f"{Z.device}")
    opts = flash_mca_default_options(C)
    if quad_scale is not None:
        opts.quad_scale = float(quad_scale)
    opts.lin_norm = int(lin_norm)
    seq = FmcaSeq(state_in.data_ptr() if state_in is not None else None,
                  state_out.data_ptr() if state_out is not None else None,
                  int(token_offset), int(n_norm))
    st = lib.flash_mca_forward_seq(Z.data_ptr(), V.data_ptr(), U.data_ptr(), gamma.data_ptr(),
                                   beta.data_ptr(), O.data_ptr(), B, n, s, e, int(C), 1, dt,
                                   workspace.data_ptr(), ws_bytes, ctypes.byref(opts),
                                   ctypes.byref(seq), _stream_ptr(stream))
    _check(st, "flash_mca_forward_seq")


def flash_mca_forward_timed(Z, V, U, gamma, beta, O, C: int, causal: bool, workspace,
                            events, path: int = FMCA_PATH_AUTO, stream=None,
                            quad_scale: float | None = None,
                            lin_norm: int = FMCA_LIN_NORM_N) -> None:
    """``flash_mca_forward_ex`` recording ``events`` (torch.cuda.Event
    objects, launch count + 1 of them) before the first kernel and after each
    kernel on ``stream``.  torch creates an event's CUDA handle on its first
    record; events without a handle yet are recorded once here to create it."""
    B, n, s, e = _shapes(Z, V, U)
    if stream is None:
        stream = torch.cuda.current_stream()
    for ev in events:
        if not ev.cuda_event:
            ev.record(stream)
    handles = (_vp * len(events))(*[ev.cuda_event for ev in events])
    dt = _dtype_code(Z)
    opts = flash_mca_default_options(C)
    if quad_scale is not None:
        opts.quad_scale = float(quad_scale)
    opts.lin_norm = int(lin_norm)
    st = lib.flash_mca_forward_timed(Z.data_ptr(), V.data_ptr(), U.data_ptr(), gamma.data_ptr(),
                                     beta.data_ptr(), O.data_ptr(), B, n, s, e, int(C),
                                     int(bool(causal)), dt, workspace.data_ptr(),
                                     workspace.numel() * workspace.element_size(), path,
                                     ctypes.byref(opts), handles, len(events),
                                     _stream_ptr(stream))
    _check(st, "flash_mca_forward_timed")


def flash_mca_forward(Z, V, U, gamma, beta, O, C: int, causal: bool, workspace,
                      stream=None) -> None:
    """The C entry point of the same name (kernel path chosen automatically)."""
    flash_mca_forward_path(Z, V, U, gamma, beta, O, C, causal, workspace, FMCA_PATH_AUTO, stream)


def flash_mca_forward_host(Z, V, U, gamma, beta, O, C: int, causal: bool, arena,
                           stream=None) -> None:
    """End-to-end call on HOST tensors (ideally pinned): copies in, computes,
    copies O back and waits.  ``arena`` is a CUDA byte buffer of at least
    ``flash_mca_host_arena_bytes`` bytes."""
    B, n, s, e = _shapes(Z, V, U)
    for name, t in (("Z", Z), ("V", V), ("U", U), ("O", O), ("gamma", gamma), ("beta", beta)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor")
    if not arena.is_cuda:
        raise ValueError("arena must be a CUDA tensor")
    dt = _dtype_code(Z)
    st = lib.flash_mca_forward_host(Z.data_ptr(), V.data_ptr(), U.data_ptr(), gamma.data_ptr(),
                                    beta.data_ptr(), O.data_ptr(), B, n, s, e, int(C),
                                    int(bool(causal)), dt, arena.data_ptr(),
                                    arena.numel() * arena.element_size(), _stream_ptr(stream))
    _check(st, "flash_mca_forward_host")


def flash_mca_forward_noalloc(Z, V, U, gamma, beta, O, C: int, causal: bool,
                              stream=None) -> None:
    """The C entry point of the same name: the forward pass with its scratch
    in a fixed array inside the library, for callers that cannot allocate
    device memory (see include/flash_mca.h).  Only the output is passed."""
    B, n, s, e = _shapes(Z, V, U)
    dt = _dtype_code(Z)
    st = lib.flash_mca_forward_noalloc(Z.data_ptr(), V.data_ptr(), U.data_ptr(),
                                       gamma.data_ptr(), beta.data_ptr(), O.data_ptr(), B, n, s,
                                       e, int(C), int(bool(causal)), dt, _stream_ptr(stream))
    _check(st, "flash_mca_forward_noalloc")


def flash_mca_decode_state_bytes(B: int, s: int, e: int, C: int, dtype: int) -> int:
    return int(lib.flash_mca_decode_state_bytes(B, s, e, C, dtype))


def flash_mca_decode_reset(state, B: int, s: int, e: int, C: int, dtype: int,
                           stream=None) -> None:
    """Clear a decode state (a CUDA byte tensor) before position 0."""
    if not state.is_cuda:
        raise ValueError("state must be a CUDA tensor")
    _check(lib.flash_mca_decode_reset(state.data_ptr(), state.numel() * state.element_size(), B,
                                      s, e, C, dtype, _stream_ptr(stream)),
           "flash_mca_decode_reset")


def flash_mca_decode_step(z, v, u, gamma, beta, o, C: int, t: int, state, n_norm: int = 0,
                          quad_scale: float | None = None, lin_norm: int = FMCA_LIN_NORM_N,
                          stream=None) -> None:
    """One decode step for the tokens at position ``t`` of B sequences:
    z [B, s], v, u, o [B, e] CUDA tensors; ``state`` as sized by
    ``flash_mca_decode_state_bytes`` and cleared by ``flash_mca_decode_reset``
    before t = 0.  ``n_norm``: the length n the default divisor uses."""
    if z.dim() != 2 or v.dim() != 2 or u.dim() != 2 or o.dim() != 2:
        raise ValueError("z, v, u, o must be 2-D: [B, s], [B, e], [B, e], [B, e]")
    B, s = z.shape
    e = v.shape[1]
    for name, x in (("z", z), ("v", v), ("u", u), ("o", o), ("gamma", gamma), ("beta", beta),
                    ("state", state)):
        if not x.is_cuda or not x.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if tuple(v.shape) != (B, e) or tuple(u.shape) != (B, e) or tuple(o.shape) != (B, e):
        raise ValueError("v, u and o must be [B, e] with z [B, s]")
    dt = _dtype_code(z)
    if v.dtype != z.dtype or u.dtype != z.dtype or o.dtype != z.dtype:
        raise TypeError("z, v, u and o must share one dtype")
    if gamma.dtype != torch.float32 or tuple(gamma.shape) != (4, s) or tuple(beta.shape) != (4, s):
        raise ValueError("gamma and beta must be float32 [4, s]")
    opts = flash_mca_default_options(C)
    if quad_scale is not None:
        opts.quad_scale = float(quad_scale)
    opts.lin_norm = int(lin_norm)
    st = lib.flash_mca_decode_step(z.data_ptr(), v.data_ptr(), u.data_ptr(), gamma.data_ptr(),
                                   beta.data_ptr(), o.data_ptr(), B, s, e, int(C), int(t),
                                   int(n_norm), dt, ctypes.byref(opts), state.data_ptr(),
                                   state.numel() * state.element_size(), _stream_ptr(stream))
    _check(st, "flash_mca_decode_step")


def flash_mca_backward_workspace_bytes(B: int, n: int, s: int, e: int, C: int, causal: bool,
                                       dtype: int) -> int:
    return int(lib.flash_mca_backward_workspace_bytes(B, n, s, e, C, int(bool(causal)), dtype))


def flash_mca_backward(Z, V, U, gamma, beta, dO, dZ, dV, dU, dgamma, dbeta, C: int,
                       causal: bool, workspace, quad_scale: float | None = None,
                       lin_norm: int = FMCA_LIN_NORM_N, stream=None, saved: bool = False) -> None:
    """Gradients of sum(O * dO) into dZ, dV, dU (I/O dtype) and dgamma, dbeta
    (float32 [4, s]); all CUDA tensors the caller owns.  saved=True calls
    flash_mca_backward_saved: `workspace` holds what flash_mca_forward left in
    it for the same inputs and options."""
    B, n, s, e = _shapes(Z, V, U)
    for name, t in (("dO", dO), ("dZ", dZ), ("dV", dV), ("dU", dU), ("dgamma", dgamma),
                    ("dbeta", dbeta), ("workspace", workspace)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    dt = _dtype_code(Z)
    for name, t, shape in (("dO", dO, (B, n, e)), ("dZ", dZ, (B, n, s)), ("dV", dV, (B, n, e)),
                           ("dU", dU, (B, n, e))):
        if t.dtype != Z.dtype or tuple(t.shape) != shape:
            raise ValueError(f"{name} must be {shape} of Z's dtype")
    if dgamma.dtype != torch.float32 or tuple(dgamma.shape) != (4, s) or \
            tuple(dbeta.shape) != (4, s):
        raise ValueError("dgamma and dbeta must be float32 [4, s]")
    opts = flash_mca_default_options(C)
    if quad_scale is not None:
        opts.quad_scale = float(quad_scale)
    opts.lin_norm = int(lin_norm)
    fn = lib.flash_mca_backward_saved if saved else lib.flash_mca_backward
    st = fn(Z.data_ptr(), V.data_ptr(), U.data_ptr(), gamma.data_ptr(), beta.data_ptr(),
            dO.data_ptr(), dZ.data_ptr(), dV.data_ptr(), dU.data_ptr(), dgamma.data_ptr(),
            dbeta.data_ptr(), B, n, s, e, int(C), int(bool(causal)), dt, ctypes.byref(opts),
            workspace.data_ptr(), workspace.numel() * workspace.element_size(),
            _stream_ptr(stream))
    _check(st, "flash_mca_backward_saved" if saved else "flash_mca_backward")


def flash_mca_backward_launch_count(B: int, n: int, s: int, e: int, C: int, causal: bool,
                                    dtype: int, quad_scale: float | None = None,
                                    lin_norm: int = FMCA_LIN_NORM_N, saved: bool = False) -> int:
    """Kernels one backward call launches (0 for rejected arguments)."""
    opts = flash_mca_default_options(C)
    if quad_scale is not None:
        opts.quad_scale = float(quad_scale)
    opts.lin_norm = int(lin_norm)
    return int(lib.flash_mca_backward_launch_count(B, n, s, e, C, int(bool(causal)), dtype,
                                                   ctypes.byref(opts), int(bool(saved))))


def backward(Z, V, U, gamma, beta, dO, C: int, causal: bool, quad_scale: float | None = None,
             lin_norm: int = FMCA_LIN_NORM_N, stream=None):
    """Convenience wrapper: allocates the outputs and the workspace with torch;
    returns (dZ, dV, dU, dgamma, dbeta)."""
    B, n, s, e = _shapes(Z, V, U)
    dZ, dV, dU = torch.empty_like(Z), torch.empty_like(V), torch.empty_like(U)
    dgamma = torch.empty((4, s), dtype=torch.float32, device=Z.device)
    dbeta = torch.empty_like(dgamma)
    nb = flash_mca_backward_workspace_bytes(B, n, s, e, C, causal, _dtype_code(Z))
    if nb == 0:
        raise FmcaError(FMCA_ERR_SHAPE, "flash_mca_backward_workspace_bytes")
    ws = torch.empty(nb, dtype=torch.uint8, device=Z.device)
    flash_mca_backward(Z, V, U, gamma, beta, dO, dZ, dV, dU, dgamma, dbeta, C, causal, ws,
                       quad_scale, lin_norm, stream)
    return dZ, dV, dU, dgamma, dbeta


def _bf16_cuda(name, t):
    if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be a contiguous bfloat16 CUDA tensor")


def flash_mca_gau_project(X, Wt, U, V, Z, stream=None) -> None:
    """U, V, Z = SiLU(X W_u), SiLU(X W_v), SiLU(X W_z) with Wt = [W_u|W_v|W_z]^T
    ([2e+s, d]); X [M, d], U and V [M, e], Z [M, s], bf16 CUDA tensors."""
    for name, t in (("X", X), ("Wt", Wt), ("U", U), ("V", V), ("Z", Z)):
        _bf16_cuda(name, t)
    M, d = X.shape
    e, s = U.shape[1], Z.shape[1]
    if tuple(Wt.shape) != (2 * e + s, d) or tuple(V.shape) != (M, e) or U.shape[0] != M or \
            Z.shape[0] != M:
        raise ValueError("shapes: X [M, d], Wt [2e+s, d], U and V [M, e], Z [M, s]")
    _check(lib.flash_mca_gau_project(X.data_ptr(), Wt.data_ptr(), U.data_ptr(), V.data_ptr(),
                                     Z.data_ptr(), M, d, e, s, _stream_ptr(stream)),
           "flash_mca_gau_project")


def flash_mca_gau_output(Y, Wo_t, Out, stream=None) -> None:
    """Out = Y W_o with Wo_t = W_o^T ([d, e]); Y [M, e], Out [M, d]."""
    for name, t in (("Y", Y), ("Wo_t", Wo_t), ("Out", Out)):
        _bf16_cuda(name, t)
    M, e = Y.shape
    d = Wo_t.shape[0]
    if tuple(Wo_t.shape) != (d, e) or tuple(Out.shape) != (M, d):
        raise ValueError("shapes: Y [M, e], Wo_t [d, e], Out [M, d]")
    _check(lib.flash_mca_gau_output(Y.data_ptr(), Wo_t.data_ptr(), Out.data_ptr(), M, e, d,
                                    _stream_ptr(stream)), "flash_mca_gau_output")


def gau_project(X, Wt, e: int, s: int, stream=None):
    """Allocating wrapper of flash_mca_gau_project: returns (U, V, Z)."""
    M = X.shape[0]
    U = torch.empty((M, e), dtype=torch.bfloat16, device=X.device)
    V = torch.empty_like(U)
    Z = torch.empty((M, s), dtype=torch.bfloat16, device=X.device)
    flash_mca_gau_project(X, Wt, U, V, Z, stream)
    return U, V, Z


def gau_output(Y, Wo_t, stream=None):
    """Allocating wrapper of flash_mca_gau_output."""
    Out = torch.empty((Y.shape[0], Wo_t.shape[0]), dtype=torch.bfloat16, device=Y.device)
    flash_mca_gau_output(Y, Wo_t, Out, stream)
    return Out


def flash_mca_device_status(stream=None) -> tuple[int, int]:
    """(status, where) recorded by the kernels since the last read; clears it."""
    where = _i32(0)
    st = lib.flash_mca_device_status(_stream_ptr(stream), ctypes.byref(where))
    return int(st), int(where.value)


def flash_mca_selftest_timeout(limit_us: int, stream=None) -> None:
    _check(lib.flash_mca_selftest_timeout(int(limit_us), _stream_ptr(stream)),
           "flash_mca_selftest_timeout")


def forward(Z, V, U, gamma, beta, C: int, causal: bool, workspace=None, out=None,
            path: int = FMCA_PATH_AUTO, stream=None, quad_scale: float | None = None,
            lin_norm: int = FMCA_LIN_NORM_N) -> torch.Tensor:
    """Convenience wrapper: allocates O (and the workspace, if not given) with
    torch and calls ``flash_mca_forward_ex``."""
    B, n, s, e = _shapes(Z, V, U)
    if out is None:
        out = torch.empty((B, n, e), dtype=Z.dtype, device=Z.device)
    if workspace is None:
        nb = flash_mca_workspace_bytes(B, n, s, e, C, causal, _dtype_code(Z))
        if nb == 0:
            raise FmcaError(FMCA_ERR_SHAPE, "flash_mca_workspace_bytes")
        workspace = torch.empty(nb, dtype=torch.uint8, device=Z.device)
    flash_mca_forward_ex(Z, V, U, gamma, beta, out, C, causal, workspace, quad_scale, lin_norm,
                         path, stream)
    return out
