"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench.

This module holds no GEMM or layout arithmetic: it only draws numbers and rounds
them to the 16-bit storage types.  Both sides of every parity check (the CPU
oracle under ``oracle/`` and the CUDA library) read the buffers it returns.

Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014).  It is counter based: draw ``i`` of a stream seeded
with ``s`` is ``mix(s + (i + 1) * 0x9E3779B97F4A7C15)``, so any slice of a stream
can be produced directly and in vectorised form.

* ``uniform[-1, 1]``: ``2 * u - 1`` with ``u = (x >> 11) * 2**-53``.
* ``normal(0, sigma)``: Box-Muller on two consecutive draws,
  ``sigma * sqrt(-2 ln(1 - u1)) * cos(2 pi u2)``.
* Each value is drawn in fp64 and rounded once, to nearest-even, to fp16 or
  bf16.  Buffers are returned as ``uint16`` bit patterns in storage order
  (row-major over the physical rows, padding included).
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

F16, BF16 = 0, 1
DTYPE_NAMES = {F16: "f16", BF16: "bf16"}


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of the SplitMix64 stream seeded with ``seed``."""
    idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + idx * GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def unit_interval(seed: int, start: int, count: int) -> np.ndarray:
    """u in [0, 1) with 53 random bits."""
    x = splitmix64(seed, start, count)
    return (x >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def round_f64_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> IEEE binary16, one round-to-nearest-even (numpy's cast rounds once)."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def round_f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> bfloat16, one round-to-nearest-even, straight from the fp64 bits.

    Handles normal results and exact zeros, which is all the generators produce
    (|x| <= 4 and |x| >= 2**-53 or x == 0); anything that would need bf16
    subnormals, overflow or NaN raises instead of being silently wrong.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    nz = ax != 0
    if np.any(~np.isfinite(x)) or np.any(ax[nz] < 2.0 ** -126) or np.any(ax >= 2.0 ** 127):
        raise ValueError("value outside the normal bf16 range")
    bits = x.view(np.uint64)
    sign = (bits >> np.uint64(63)).astype(np.uint16)
    # round the 52-bit mantissa to 7 bits, ties to even (carry may bump the exponent)
    lsb = (bits >> np.uint64(45)) & np.uint64(1)
    with np.errstate(over="ignore"):
        r = bits + np.uint64((1 << 44) - 1) + lsb
    exp = ((r >> np.uint64(52)) & np.uint64(0x7FF)).astype(np.int64) - 1023 + 127
    man = ((r >> np.uint64(45)) & np.uint64(0x7F)).astype(np.uint16)
    out = (sign << np.uint16(15)) | (exp.astype(np.uint16) << np.uint16(7)) | man
    return np.where(nz, out, sign << np.uint16(15)).astype(np.uint16)


def round_to_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == F16:
        return round_f64_to_f16_bits(x)
    if dtype == BF16:
        return round_f64_to_bf16_bits(x)
    raise ValueError(f"unknown dtype {dtype}")


class Stream:
    """A SplitMix64 stream consumed in draw order (A, B, bias, scale, R)."""

    def __init__(self, seed: int):
        self.seed = int(seed)
        self.pos = 0

    def uniform(self, count: int, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
        u = unit_interval(self.seed, self.pos, count)
        self.pos += count
        return lo + (hi - lo) * u

    def normal(self, count: int, sigma: float) -> np.ndarray:
        u = unit_interval(self.seed, self.pos, 2 * count)
        self.pos += 2 * count
        u1, u2 = u[0::2], u[1::2]
        return sigma * np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * np.pi * u2)

    def matrix(self, rows: int, ld: int, dtype: int, dist: str = "uniform",
               sigma: float = 0.5) -> np.ndarray:
        """A rows x ld storage buffer of 16-bit patterns (padding columns drawn too)."""
        n = rows * ld
        v = self.uniform(n) if dist == "uniform" else self.normal(n, sigma)
        return round_to_bits(v, dtype).reshape(rows, ld)

    def vector(self, n: int, dtype: int, dist: str = "uniform", sigma: float = 0.5) -> np.ndarray:
        v = self.uniform(n) if dist == "uniform" else self.normal(n, sigma)
        return round_to_bits(v, dtype)


def gemm_problem(M: int, N: int, K: int, dtype: int, seed: int, *, permA: int = 0,
                 permB: int = 0, lda: int | None = None, ldb: int | None = None,
                 dist: str = "uniform", sigma: float = 0.5, bias: bool = False,
                 scale: bool = False, residual: bool = False,
                 ldr: int | None = None) -> dict:
    """Storage buffers for one GEMM problem, drawn in the order A, B, bias, scale, R.

    permA = 0: A is an M x lda buffer (A(m,k) = A[m, k]); permA = 1: a K x lda
    buffer holding the transpose (A(m,k) = A[k, m]).  permB = 0: B is K x ldb
    (B(k,n) = B[k, n]); permB = 1: N x ldb (B(k,n) = B[n, k]).
    """
    a_rows, a_w = (M, K) if permA == 0 else (K, M)
    b_rows, b_w = (K, N) if permB == 0 else (N, K)
    lda = a_w if lda is None else lda
    ldb = b_w if ldb is None else ldb
    s = Stream(seed)
    out = {"M": M, "N": N, "K": K, "dtype": dtype, "permA": permA, "permB": permB,
           "lda": lda, "ldb": ldb}
    out["A"] = s.matrix(a_rows, lda, dtype, dist, sigma)
    out["B"] = s.matrix(b_rows, ldb, dtype, dist, sigma)
    out["bias"] = s.vector(N, dtype, dist, sigma) if bias else None
    out["scale"] = s.vector(M, dtype, dist, sigma) if scale else None
    if residual:
        ldr = N if ldr is None else ldr
        out["R"] = s.matrix(M, ldr, dtype, dist, sigma)
        out["ldr"] = ldr
    else:
        out["R"] = None
        out["ldr"] = 0
    return out


def pointwise_problem(M: int, N: int, dtype: int, seed: int, *, permX: int = 0,
                      ldx: int | None = None, dist: str = "uniform", sigma: float = 0.5,
                      bias: bool = False, scale: bool = False, residual: bool = False,
                      ldr: int | None = None) -> dict:
    """Storage buffers for one pointwise program, drawn in the order X, bias,
    scale, R.  permX = 0: X is an M x ldx buffer (X(m,n) = X[m, n]);
    permX = 1: an N x ldx buffer holding the transpose (X(m,n) = X[n, m])."""
    x_rows, x_w = (M, N) if permX == 0 else (N, M)
    ldx = x_w if ldx is None else ldx
    s = Stream(seed)
    out = {"M": M, "N": N, "dtype": dtype, "permX": permX, "ldx": ldx}
    out["X"] = s.matrix(x_rows, ldx, dtype, dist, sigma)
    out["bias"] = s.vector(N, dtype, dist, sigma) if bias else None
    out["scale"] = s.vector(M, dtype, dist, sigma) if scale else None
    if residual:
        ldr = N if ldr is None else ldr
        out["R"] = s.matrix(M, ldr, dtype, dist, sigma)
        out["ldr"] = ldr
    else:
        out["R"] = None
        out["ldr"] = 0
    return out
