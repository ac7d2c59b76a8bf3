"""CPU oracle -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it.

* ``gemm``: the fp64 plain-definition GEMM with the fused epilogue
  (``gemm_oracle.c``, compiled here with gcc + OpenMP).
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
