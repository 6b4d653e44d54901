"""fp64 CPU oracle of the FLASH mixed-chunk attention forward core.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
and its Python binding never import, load or call it, and it shares no code with
them: the arithmetic lives in ``mca_oracle.c`` (plain fp64 C, one loop per step
of the definition), this module only compiles it and marshals numpy arrays.

The definition it follows is stated step by step at the top of ``mca_oracle.c``
("FLASH: Possibly the Most Interesting Efficient Transformer Design Recently",
sections "Weak Attention" and "Mixed Chunk").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mca_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``mca_oracle.c`` into ``oracle/liboracle.so`` (fp64, OpenMP,
    no fast-math, no FMA contraction) and return its path."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d = ctypes.POINTER(ctypes.c_double)
            i = ctypes.c_int
            lib.mca_oracle_forward.argtypes = [d, d, d, d, d, d, i, i, i, i, i, i, i]
            lib.mca_oracle_forward.restype = i
            lib.mca_oracle_rows.argtypes = [d, d, d, d, d, i, i, i, i, i, i, i,
                                            ctypes.POINTER(ctypes.c_int64), d, i]
            lib.mca_oracle_rows.restype = i
            lib.mca_oracle_forward_ex.argtypes = [d, d, d, d, d, d, i, i, i, i, i, i,
                                                  ctypes.c_double, i, i]
            lib.mca_oracle_forward_ex.restype = i
            lib.mca_oracle_rows_ex.argtypes = [d, d, d, d, d, i, i, i, i, i, i,
                                               ctypes.c_double, i, i,
                                               ctypes.POINTER(ctypes.c_int64), d, i]
            lib.mca_oracle_rows_ex.restype = i
            lib.mca_oracle_max_threads.argtypes = []
            lib.mca_oracle_max_threads.restype = i
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Exact fp64 copy of an input (numpy array or torch tensor of any float
    dtype): the oracle sees the values the GPU sees, without rounding."""
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(_load().mca_oracle_max_threads())


# Global-term divisors of the variants (see the top of mca_oracle.c).
LIN_NORM_N = 0         # 1/n
LIN_NORM_SUMMED = 1    # 1/(tokens the sum covers): g*C for causal chunk g, n otherwise
LIN_NORM_POSITION = 2  # 1/(t+1) for the token at position t
LIN_NORM_NONE = 3      # no global term (with C = n: FLASH-Quad)


def forward(Z, V, U, gamma, beta, C: int, causal: bool, nthreads: int = 0,
            quad_scale: float | None = None, lin_norm: int | None = None) -> np.ndarray:
    """O[B, n, e] in fp64 for Z[B, n, s], V/U[B, n, e], gamma/beta[4, s].

    With ``quad_scale`` or ``lin_norm`` given, the variant form: intra-chunk
    weights quad_scale * relu(q . k)^2 (default 1/C^2, i.e. relu(x/C)^2) and
    the global-term divisor ``lin_norm`` (LIN_NORM_*)."""
    Z, V, U, gamma, beta = (_f64(t) for t in (Z, V, U, gamma, beta))
    B, n, s = Z.shape
    e = V.shape[2]
    if V.shape != (B, n, e) or U.shape != (B, n, e):
        raise ValueError("V and U must be [B, n, e] with Z [B, n, s]")
    if gamma.shape != (4, s) or beta.shape != (4, s):
        raise ValueError("gamma and beta must be [4, s]")
    O = np.zeros((B, n, e), dtype=np.float64)
    if quad_scale is None and lin_norm is None:
        rc = _load().mca_oracle_forward(_ptr(Z), _ptr(V), _ptr(U), _ptr(gamma), _ptr(beta),
                                        _ptr(O), B, n, s, e, int(C), int(bool(causal)),
                                        int(nthreads))
    else:
        qs = 1.0 / (float(C) * float(C)) if quad_scale is None else float(quad_scale)
        rc = _load().mca_oracle_forward_ex(_ptr(Z), _ptr(V), _ptr(U), _ptr(gamma),
                                           _ptr(beta), _ptr(O), B, n, s, e, int(C),
                                           int(bool(causal)), qs, int(lin_norm or 0),
                                           int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return O


def rows(Z, V, U, gamma, beta, C: int, causal: bool, row_ids, nthreads: int = 0,
         quad_scale: float | None = None, lin_norm: int | None = None) -> np.ndarray:
    """O at selected flat token indices ``row_ids`` (b*n + t): array [len, e]
    (variant arguments as for ``forward``)."""
    Z, V, U, gamma, beta = (_f64(t) for t in (Z, V, U, gamma, beta))
    B, n, s = Z.shape
    e = V.shape[2]
    ids = np.ascontiguousarray(np.asarray(row_ids, dtype=np.int64).reshape(-1))
    out = np.zeros((ids.size, e), dtype=np.float64)
    idp = ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    if quad_scale is None and lin_norm is None:
        rc = _load().mca_oracle_rows(_ptr(Z), _ptr(V), _ptr(U), _ptr(gamma), _ptr(beta),
                                     B, n, s, e, int(C), int(bool(causal)), int(ids.size),
                                     idp, _ptr(out), int(nthreads))
    else:
        qs = 1.0 / (float(C) * float(C)) if quad_scale is None else float(quad_scale)
        rc = _load().mca_oracle_rows_ex(_ptr(Z), _ptr(V), _ptr(U), _ptr(gamma), _ptr(beta),
                                        B, n, s, e, int(C), int(bool(causal)), qs,
                                        int(lin_norm or 0), int(ids.size), idp, _ptr(out),
                                        int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out
