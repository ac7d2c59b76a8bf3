"""tg_gemm_static_ws: the stream-K GEMM with library-owned static scratch, for
callers that cannot allocate device memory (inside a stream capture, under an
outside allocator).  Its results must match tg_gemm_ws with a caller
workspace, call after call, although every call reuses the same array.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import os

import numpy as np
import pytest

import synthetic
from synthetic import F16, BF16
from helpers import SENTINEL, check_close, decode, dev, host_bits

pytestmark = pytest.mark.gpu

CAPACITY = 40 << 20


class forced:
    def __init__(self, cfg):
        self.cfg = cfg

    def __enter__(self):
        self.old = os.environ.get("TG_FORCE_CONFIG")
        if self.cfg is None:
            os.environ.pop("TG_FORCE_CONFIG", None)
        else:
            os.environ["TG_FORCE_CONFIG"] = self.cfg

    def __exit__(self, *exc):
        if self.old is None:
            os.environ.pop("TG_FORCE_CONFIG", None)
        else:
            os.environ["TG_FORCE_CONFIG"] = self.old


def operands(tg, p):
    bias = dev(p["bias"]) if p.get("bias") is not None else None
    scale = dev(p["scale"]) if p.get("scale") is not None else None
    R = dev(p["R"]) if p.get("R") is not None else None
    epi = tg.make_epilogue(bias, scale, bool(p.get("relu", False)), R, p.get("ldr", 0) or 0)
    return dev(p["A"]), dev(p["B"]), epi, (bias, scale, R)


def with_workspace(tg, p):
    """Reference: the existing entry point with a caller-allocated workspace."""
    import torch
    A, B, epi, keep = operands(tg, p)
    M, N, K = p["M"], p["N"], p["K"]
    need = tg.tg_gemm_workspace_size(M, N, K, p["dtype"], p["permA"], p["permB"], epi)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
    C = torch.full((M, N), SENTINEL, dtype=torch.int16, device="cuda")
    rc = tg.tg_gemm_ws(M, N, K, A, p["lda"], p["permA"], B, p["ldb"], p["permB"], C, N,
                       p["dtype"], epi, ws if need else None, need)
    torch.cuda.synchronize()
    assert rc == tg.TG_OK, tg.tg_status_string(rc)
    return host_bits(C), need


def static_scratch(tg, p):
    import torch
    A, B, epi, keep = operands(tg, p)
    M, N, K = p["M"], p["N"], p["K"]
    C = torch.full((M, N), SENTINEL, dtype=torch.int16, device="cuda")
    rc = tg.tg_gemm_static_ws(M, N, K, A, p["lda"], p["permA"], B, p["ldb"], p["permB"], C, N,
                              p["dtype"], epi)
    torch.cuda.synchronize()
    assert rc == tg.TG_OK, tg.tg_status_string(rc)
    st, code = tg.tg_debug_status()
    assert st == tg.TG_OK, hex(code)
    return host_bits(C)


def same_within_tolerance(got, ref, dtype, what):
    check_close(got, decode(ref, dtype), dtype, what=what)


def test_static_scratch_matches_caller_workspace_two_calls_in_a_row(tg):
    # two different split shapes, each called twice: the shared array keeps the
    # previous call's contents, which must never leak into the next result
    cases = [
        (synthetic.gemm_problem(1000, 520, 1200, F16, 301), "pair=1,bn=256,grid=10,sk=1"),
        (synthetic.gemm_problem(700, 312, 1000, BF16, 302, bias=True, scale=True,
                                residual=True), "pair=0,bn=128,grid=4,sk=1"),
    ]
    cases[1][0]["relu"] = True
    for p, cfg in cases:
        with forced(cfg):
            ref, need = with_workspace(tg, p)
            assert 0 < need <= CAPACITY  # the case really uses scratch
            first = static_scratch(tg, p)
            second = static_scratch(tg, p)
        same_within_tolerance(first, ref, p["dtype"], f"{cfg}, first call")
        same_within_tolerance(second, ref, p["dtype"], f"{cfg}, second call")


def test_static_scratch_default_selection_headline_shape(tg):
    # the 4096^3 fp16 GEMM picks a stream-K split whose scratch fits the array
    p = synthetic.gemm_problem(4096, 4096, 4096, F16, 1002)
    with forced(None):
        ref, need = with_workspace(tg, p)
        assert 0 < need <= CAPACITY
        for call in ("first", "second"):
            got = static_scratch(tg, p)
            same_within_tolerance(got, ref, F16, f"4096^3, {call} call")


def test_static_scratch_rejects_splits_beyond_capacity(tg):
    import torch
    # 16 CTA-pair tiles dealt out over 76 clusters: six partial slots per
    # split tile, about 114 MB of scratch, more than the static array holds
    p = synthetic.gemm_problem(1024, 1024, 4096, F16, 303)
    A, B, epi, keep = operands(tg, p)
    C = torch.zeros((1024, 1024), dtype=torch.int16, device="cuda")
    with forced("pair=1,bn=256,sk=1"):
        need = tg.tg_gemm_workspace_size(1024, 1024, 4096, F16)
        if need <= CAPACITY:
            pytest.skip(f"this GPU's split needs only {need} bytes")
        rc = tg.tg_gemm_static_ws(1024, 1024, 4096, A, 4096, 0, B, 1024, 0, C, 1024, F16)
    assert rc == tg.TG_ERR_BUFFER
