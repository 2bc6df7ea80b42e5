"""The oracle: a plain, slow float64 CPU implementation of the W4A16 GEMM.

TEST INFRASTRUCTURE ONLY. Only `tests/`, `__graft_entry__.smoke()` and the
benchmark's CPU-baseline leg may import this package. It shares no code with the
CUDA library and never imports it.

Follows the "Validation" section of the MatMulNBits Marlin pull request
(github.com/justinchuby/onnx-genai pull 960): an f64 dequant -> GEMM reference,
here written out in C (`w4a16_oracle.c`) with plain loops. This module widens the
float16/float32 inputs to float64 (lossless) and calls that C code through ctypes.
The repacked-layout reference lives in `repack_layout.py`.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

from . import repack_layout  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (-O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            u8p = ctypes.POINTER(ctypes.c_uint8)
            i32p = ctypes.POINTER(ctypes.c_int32)
            ci = ctypes.c_int
            lib.oracle_dequant.argtypes = [u8p, dp, u8p, ci, ci, ci, dp]
            lib.oracle_gemm.argtypes = [dp, ci, ci, u8p, dp, u8p, ci, ci,
                                        i32p, ci, i32p, ci, dp, ci]
            lib.oracle_gemm_swiglu.argtypes = [dp, ci, ci, u8p, dp, u8p, u8p, dp, u8p, ci, ci,
                                               i32p, ci, i32p, ci, dp, ci]
            for f in (lib.oracle_dequant, lib.oracle_gemm, lib.oracle_gemm_swiglu):
                f.restype = ci
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def _ptr(a: Optional[np.ndarray], ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.float64)


def _u8(a) -> Optional[np.ndarray]:
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a), dtype=np.uint8)


def _idx(ix, n):
    if ix is None:
        return None, n
    arr = np.ascontiguousarray(np.asarray(ix), dtype=np.int32)
    return arr, int(arr.size)


def _check_meta(bq, scales, zp, K, group):
    N = bq.shape[0]
    G = K // group
    if bq.shape != (N, K // 2):
        raise ValueError("bq must be [N, K/2]")
    if scales.shape != (N, G):
        raise ValueError("scales must be [N, K/group]")
    if zp is not None and zp.shape != (N, (G + 1) // 2):
        raise ValueError("zp must be [N, ceil(G/2)]")


def dequant(bq, scales, zp, K: int, group: int) -> np.ndarray:
    """W[n, k] = (q - zp) * scale in float64, shape [N, K]."""
    bq, zp, s = _u8(bq), _u8(zp), _f64(scales)
    _check_meta(bq, s, zp, K, group)
    N = bq.shape[0]
    W = np.empty((N, K), dtype=np.float64)
    rc = _load().oracle_dequant(_ptr(bq, ctypes.c_uint8), _ptr(s, ctypes.c_double),
                                _ptr(zp, ctypes.c_uint8), N, K, group,
                                _ptr(W, ctypes.c_double))
    if rc:
        raise RuntimeError(f"oracle_dequant failed ({rc})")
    return W


def gemm(A, bq, scales, zp, group: int, rows: Optional[Sequence[int]] = None,
         cols: Optional[Sequence[int]] = None, nthreads: Optional[int] = None) -> np.ndarray:
    """Y = A . dequant(Bq)^T in float64; optional row (m) and column (n) subsets."""
    A64, bq, zp, s = _f64(A), _u8(bq), _u8(zp), _f64(scales)
    M, K = A64.shape
    _check_meta(bq, s, zp, K, group)
    N = bq.shape[0]
    r, nr = _idx(rows, M)
    c, nc = _idx(cols, N)
    Y = np.empty((nr, nc), dtype=np.float64)
    rc = _load().oracle_gemm(_ptr(A64, ctypes.c_double), M, K,
                             _ptr(bq, ctypes.c_uint8), _ptr(s, ctypes.c_double),
                             _ptr(zp, ctypes.c_uint8), N, group,
                             _ptr(r, ctypes.c_int32), nr, _ptr(c, ctypes.c_int32), nc,
                             _ptr(Y, ctypes.c_double), nthreads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_gemm failed ({rc})")
    return Y


def gemm_swiglu(A, gate, up, group: int, rows=None, cols=None,
                nthreads: Optional[int] = None) -> np.ndarray:
    """Y = silu(A . Wg^T) * (A . Wu^T) in float64. gate/up = (bq, scales, zp)."""
    A64 = _f64(A)
    M, K = A64.shape
    bg, sg, zg = _u8(gate[0]), _f64(gate[1]), _u8(gate[2])
    bu, su, zu = _u8(up[0]), _f64(up[1]), _u8(up[2])
    _check_meta(bg, sg, zg, K, group)
    _check_meta(bu, su, zu, K, group)
    N = bg.shape[0]
    r, nr = _idx(rows, M)
    c, nc = _idx(cols, N)
    Y = np.empty((nr, nc), dtype=np.float64)
    rc = _load().oracle_gemm_swiglu(_ptr(A64, ctypes.c_double), M, K,
                                    _ptr(bg, ctypes.c_uint8), _ptr(sg, ctypes.c_double),
                                    _ptr(zg, ctypes.c_uint8),
                                    _ptr(bu, ctypes.c_uint8), _ptr(su, ctypes.c_double),
                                    _ptr(zu, ctypes.c_uint8), N, group,
                                    _ptr(r, ctypes.c_int32), nr, _ptr(c, ctypes.c_int32), nc,
                                    _ptr(Y, ctypes.c_double), nthreads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_gemm_swiglu failed ({rc})")
    return Y


def rmsnorm(A, gamma, eps: float) -> np.ndarray:
    """RMS normalisation of each activation row, float64 (the RMS-norm prologue
    of the same pull request, "Update -- fused RMS-norm epilogue + e2e PASS" and
    "Update -- P1 COMPLETE": the normalised activation is staged, then the GEMM
    runs on it). Reading of the pages, which give no formula: the ONNX
    SimplifiedLayerNormalization that the prologue replaces,

        out[m, k] = A[m, k] / sqrt(mean_k(A[m, k]^2) + eps) * gamma[k].

    Plain float64 arithmetic on the widened inputs; no rounding of the result."""
    A64 = _f64(A)
    g64 = _f64(gamma).reshape(-1)
    if A64.ndim != 2 or g64.size != A64.shape[1]:
        raise ValueError("A must be [M, K] and gamma [K]")
    M, K = A64.shape
    out = np.empty_like(A64)
    for m in range(M):
        row = A64[m]
        r = 1.0 / np.sqrt(float(np.dot(row, row)) / K + float(eps))
        out[m] = row * r * g64
    return out


def _rows_of(A, rows):
    A = np.asarray(A)
    return A if rows is None else A[np.asarray(rows)]


def gemm_rmsnorm(A, gamma, eps: float, bq, scales, zp, group: int, rows=None, cols=None,
                 nthreads: Optional[int] = None) -> np.ndarray:
    """Y = rmsnorm(A) . dequant(Bq)^T in float64 (optionally only some rows of A)."""
    return gemm(rmsnorm(_rows_of(A, rows), gamma, eps), bq, scales, zp, group, cols=cols,
                nthreads=nthreads)


def gemm_swiglu_rmsnorm(A, gamma, eps: float, gate, up, group: int, rows=None, cols=None,
                        nthreads: Optional[int] = None) -> np.ndarray:
    """Y = silu(rmsnorm(A) . Wg^T) * (rmsnorm(A) . Wu^T) in float64."""
    return gemm_swiglu(rmsnorm(_rows_of(A, rows), gamma, eps), gate, up, group, cols=cols,
                       nthreads=nthreads)


def repack(bq) -> np.ndarray:
    return repack_layout.repack(_u8(bq))


def unpack(rep, N: int, K: int) -> np.ndarray:
    return repack_layout.unpack(rep, N, K)
