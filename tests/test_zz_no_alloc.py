"""tg_gemm_static_ws: the stream-K GEMM with library-owned static scratch, for
callers that cannot allocate device memory (code under an outside allocator
that owns the device's memory, plugins whose host framework forbids device
allocations, host paths that cannot take cudaMalloc's implicit
synchronisation).  Its results must match tg_gemm_ws with a caller workspace
and the fp64 oracle, call after call, although every call reuses the same
array.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import os

import numpy as np
import pytest

import oracle
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


def args_of(p, A, B, C, epi):
    return (p["M"], p["N"], p["K"], A, p["lda"], p["permA"], B, p["ldb"], p["permB"], C,
            p["N"], p["dtype"], epi)


def with_workspace(tg, p):
    """The existing entry point, with a workspace the caller allocates."""
    import torch
    A, B, epi, keep = operands(tg, p)
    C = torch.full((p["M"], p["N"]), SENTINEL, dtype=torch.int16, device="cuda")
    args = args_of(p, A, B, C, epi)
    need = tg.tg_gemm_workspace_size_ex(*args)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
    rc = tg.tg_gemm_ws(*args, ws if need else None, need)
    torch.cuda.synchronize()
    assert rc == tg.TG_OK, tg.tg_status_string(rc)
    return host_bits(C), need


def static_scratch(tg, p):
    import torch
    A, B, epi, keep = operands(tg, p)
    C = torch.full((p["M"], p["N"]), SENTINEL, dtype=torch.int16, device="cuda")
    rc = tg.tg_gemm_static_ws(*args_of(p, A, B, C, epi))
    torch.cuda.synchronize()
    assert rc == tg.TG_OK, tg.tg_status_string(rc)
    st, code = tg.tg_debug_status()
    assert st == tg.TG_OK, hex(code)
    return host_bits(C)


def agree(got, ref_bits, want, dtype, what):
    """Within the parity tolerance of the caller-workspace call and of the oracle."""
    check_close(got, decode(ref_bits, dtype), dtype, what=f"{what} vs tg_gemm_ws")
    check_close(got, want, dtype, what=f"{what} vs oracle")


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
        want = oracle.gemm(p)
        with forced(cfg):
            ref, need = with_workspace(tg, p)
            assert 0 < need <= CAPACITY  # the case really uses scratch
            first = static_scratch(tg, p)
            second = static_scratch(tg, p)
        agree(first, ref, want, p["dtype"], f"{cfg}, first call")
        agree(second, ref, want, p["dtype"], f"{cfg}, second call")


def test_static_scratch_stages_unaligned_operands(tg):
    # a row stride that is not a whole number of 16-byte units: B is copied
    # into an aligned image inside the static array, after the split's region
    p = synthetic.gemm_problem(640, 264, 960, F16, 304, ldb=264 + 3, bias=True)
    want = oracle.gemm(p)
    with forced("pair=0,bn=128,grid=6,sk=1"):
        ref, need = with_workspace(tg, p)
        assert need > tg.tg_gemm_workspace_size(640, 264, 960, F16)  # staging on top of the split
        first = static_scratch(tg, p)
        second = static_scratch(tg, p)
    agree(first, ref, want, F16, "unaligned ldb, first call")
    agree(second, ref, want, F16, "unaligned ldb, second call")


def test_static_scratch_default_selection_headline_shape(tg):
    # the 4096^3 fp16 GEMM picks a stream-K split whose scratch fits the array
    p = synthetic.gemm_problem(4096, 4096, 4096, F16, 1002)
    want = oracle.gemm(p)
    with forced(None):
        ref, need = with_workspace(tg, p)
        assert 0 < need <= CAPACITY
        for call in ("first", "second"):
            got = static_scratch(tg, p)
            agree(got, ref, want, F16, f"4096^3, {call} call")


def test_static_scratch_rejects_splits_beyond_capacity(tg):
    import torch
    # 16 CTA-pair tiles forced to be dealt out over 76 clusters: six partial
    # slots per split tile, about 114 MB of scratch, more than the array holds
    p = synthetic.gemm_problem(1024, 1024, 4096, F16, 303)
    A, B, epi, keep = operands(tg, p)
    C = torch.zeros((1024, 1024), dtype=torch.int16, device="cuda")
    with forced("pair=1,bn=256,sk=1"):
        need = tg.tg_gemm_workspace_size(1024, 1024, 4096, F16)
        if need <= CAPACITY:
            pytest.skip(f"this GPU's split needs only {need} bytes")
        rc = tg.tg_gemm_static_ws(1024, 1024, 4096, A, 4096, 0, B, 1024, 0, C, 1024, F16)
    assert rc == tg.TG_ERR_BUFFER
