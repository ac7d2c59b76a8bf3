"""Shared test helpers: device buffers holding 16-bit patterns, the GEMM call
through the C ABI, and the elementwise tolerance check against the oracle."""
from __future__ import annotations

import numpy as np

SENTINEL = 0x7E00  # fp16 NaN / large bf16: padding of C that must survive every call
RTOL = 1e-2        # |gpu - oracle| <= 1e-2 * max(1, |oracle|), inputs in [-1, 1], K <= 8192


def dev(bits: np.ndarray):
    """uint16 pattern array -> int16 CUDA tensor with the same bits."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def host_bits(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    """fp16 via numpy's half type, bf16 by widening to fp32 (library routines)."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == 0:
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run_gemm(tg, p: dict, ldc: int | None = None, stream=None, force: str | None = None):
    """Runs tg_gemm on the problem dict ``p`` (synthetic.gemm_problem keys).

    Returns (C storage bits as uint16 [M, ldc], status).  C is pre-filled with
    SENTINEL so writes outside the M x N window are visible.
    """
    import os
    import torch
    M, N, K = p["M"], p["N"], p["K"]
    ldc = N if ldc is None else ldc
    A, B = dev(p["A"]), dev(p["B"])
    bias = dev(p["bias"]) if p.get("bias") is not None else None
    scale = dev(p["scale"]) if p.get("scale") is not None else None
    R = dev(p["R"]) if p.get("R") is not None else None
    C = torch.full((M, ldc), SENTINEL, dtype=torch.int16, device="cuda")
    epi = tg.make_epilogue(bias, scale, bool(p.get("relu", False)), R, p.get("ldr", 0) or 0)
    old = os.environ.get("TG_FORCE_CONFIG")
    if force is not None:
        os.environ["TG_FORCE_CONFIG"] = force
    try:
        rc = tg.tg_gemm(M, N, K, A, p["lda"], p["permA"], B, p["ldb"], p["permB"], C, ldc,
                        p["dtype"], epi, stream)
    finally:
        if force is not None:
            if old is None:
                del os.environ["TG_FORCE_CONFIG"]
            else:
                os.environ["TG_FORCE_CONFIG"] = old
    torch.cuda.synchronize()
    return host_bits(C), rc


def check_close(gpu_bits: np.ndarray, ref: np.ndarray, dtype: int, rows=None, what=""):
    """Elementwise |gpu - ref| <= RTOL * max(1, |ref|); returns the max normalised error."""
    M, N = ref.shape
    g = decode(gpu_bits[:, :N] if rows is None else gpu_bits[rows, :N], dtype)
    err = np.abs(g - ref) / np.maximum(1.0, np.abs(ref))
    bad = ~(err <= RTOL)  # NaN counts as bad
    if bad.any():
        i, j = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at "
                             f"({i},{j}) gpu={g[i, j]!r} oracle={ref[i, j]!r}, max err {np.nanmax(err)}")
    return float(err.max())


def check_padding(gpu_bits: np.ndarray, N: int):
    if gpu_bits.shape[1] > N:
        assert np.all(gpu_bits[:, N:] == SENTINEL), "write outside the M x N window"
