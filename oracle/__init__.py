"""CPU oracle -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it.

* ``gemm``: the fp64 plain-definition GEMM with the fused epilogue
  (``gemm_oracle.c``, compiled here with gcc + OpenMP).
* ``pointwise``: the fp64 named-layout pointwise program (numpy, row by row).
* ``layouts``: brute-force GF(2) layout evaluation and the pages' ownership
  rules written out directly (``layout_oracle.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compiles the C oracle (host code only, portable C: builds on x86 and Arm)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp,
                        _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_gemm.argtypes = [i64, i64, i64, p, i64, ctypes.c_int, p, i64, ctypes.c_int,
                                    ctypes.c_int, p, p, ctypes.c_int, p, i64, i64, i64, p,
                                    ctypes.c_int]
        lib.oracle_gemm.restype = ctypes.c_int
        lib.oracle_decode.argtypes = [p, i64, ctypes.c_int, p]
        lib.oracle_decode.restype = None
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    """fp64 values of 16-bit patterns, by the oracle's own decoders."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_decode(_ptr(bits), bits.size, dtype, _ptr(out))
    return out


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def gemm(p: dict, rows: tuple[int, int] | None = None, relu: bool | None = None,
         threads: int = 0) -> np.ndarray:
    """y(m, n) in fp64 for rows[0] <= m < rows[1] of the problem dict ``p``.

    ``p`` holds the storage buffers and sizes (the keys of
    ``synthetic.gemm_problem``; a ``relu`` key may be present).
    """
    M, N, K = p["M"], p["N"], p["K"]
    r0, r1 = (0, M) if rows is None else rows
    relu = bool(p.get("relu", False)) if relu is None else relu
    arrs = {k: (None if p.get(k) is None else np.ascontiguousarray(p[k], dtype=np.uint16))
            for k in ("A", "B", "bias", "scale", "R")}
    y = np.empty((r1 - r0, N), dtype=np.float64)
    rc = _load().oracle_gemm(M, N, K, _ptr(arrs["A"]), p["lda"], p["permA"],
                             _ptr(arrs["B"]), p["ldb"], p["permB"], p["dtype"],
                             _ptr(arrs["bias"]), _ptr(arrs["scale"]), int(relu),
                             _ptr(arrs["R"]), p.get("ldr", 0) or 0, r0, r1, _ptr(y), threads)
    if rc != 0:
        raise ValueError("oracle_gemm rejected its arguments")
    return y


def pointwise(p: dict) -> np.ndarray:
    """y(m, n) in fp64 of the named-layout pointwise program
    (ninetoothed.org "Named layouts": pointwise work, missing-axis
    broadcasting, reordering, bias/ReLU/residual postprocessing).

    x = X(m, n), read through the explicit permute (permX = 0: X[m, n] of an
    M x ldx buffer; permX = 1: X[n, m] of an N x ldx buffer), then the GEMM's
    epilogue in its order: x *= scale_m[m]; x += bias_n[n]; x = max(x, 0);
    x += R[m, n].  An absent operand is the identity; scale_m (axes "m") is
    the same for every n of a row, bias_n (axes "n") the same for every m of
    a column.  Unrounded.  ``p`` holds the keys of
    ``synthetic.pointwise_problem``.
    """
    M, N, dt = p["M"], p["N"], p["dtype"]
    X = decode(p["X"], dt)
    bias = None if p.get("bias") is None else decode(p["bias"], dt)
    scale = None if p.get("scale") is None else decode(p["scale"], dt)
    R = None if p.get("R") is None else decode(p["R"], dt)
    y = np.empty((M, N), dtype=np.float64)
    for m in range(M):
        row = X[m, :N].copy() if p["permX"] == 0 else X[:N, m].copy()
        if scale is not None:
            row *= scale[m]
        if bias is not None:
            row += bias[:N]
        if p.get("relu", False):
            row = np.maximum(row, 0.0)
        if R is not None:
            row += R[m, :N]
        y[m] = row
    return y
