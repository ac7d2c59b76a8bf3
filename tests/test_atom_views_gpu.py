"""MN-major operands whose extent is not a whole number of 64-element swizzle
atoms (A given as a permuted K x M buffer with M mod 64 != 0, B row-major
with N mod 64 != 0).

Such an operand's stage arrives as one 2-D TMA box per 64-element atom; the
tensor map bounds every box at M (or N) and K, so the partial last atom is
zero-filled and nothing past the operand is read.  Results must match the
fp64 oracle on every element, under several tile configurations; one case
puts A flush against the end of a raw driver allocation, so that a read
past its last byte would fault instead of landing in an allocator's slack.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synthetic
from synthetic import F16, BF16
from helpers import SENTINEL, check_close, check_padding, dev, host_bits, run_gemm

pytestmark = pytest.mark.gpu


def _driver():
    lib = ctypes.CDLL("libcuda.so.1")
    lib.cuMemAlloc_v2.argtypes = [ctypes.POINTER(ctypes.c_uint64), ctypes.c_size_t]
    lib.cuMemFree_v2.argtypes = [ctypes.c_uint64]
    lib.cuMemcpyHtoD_v2.argtypes = [ctypes.c_uint64, ctypes.c_void_p, ctypes.c_size_t]
    return lib


class TightBuffer:
    """A driver allocation of exactly `nbytes` (a multiple of 2 MiB) holding
    `bits` flush against its end."""

    def __init__(self, bits: np.ndarray, nbytes: int):
        import torch
        torch.zeros(1, device="cuda")  # the primary context is current on this thread
        self.lib = _driver()
        flat = np.ascontiguousarray(bits).reshape(-1).view(np.uint16)
        assert flat.nbytes <= nbytes and nbytes % (2 << 20) == 0
        self.base = ctypes.c_uint64(0)
        assert self.lib.cuMemAlloc_v2(ctypes.byref(self.base), nbytes) == 0
        self.addr = self.base.value + nbytes - flat.nbytes
        assert self.addr % 16 == 0
        assert self.lib.cuMemcpyHtoD_v2(self.addr, flat.ctypes.data, flat.nbytes) == 0

    def free(self):
        self.lib.cuMemFree_v2(self.base.value)


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("force", [None, "pair=1,bn=256", "pair=0,bn=128"])
def test_permuted_a_with_partial_atom(tg, dtype, force):
    # lda = M = 1000: the last atom of each storage row holds 40 of 64 elements
    M, N, K = 1000, 512, 1048
    p = synthetic.gemm_problem(M, N, K, dtype, 41, permA=1, bias=True)
    c, rc = run_gemm(tg, p, ldc=N + 8, force=force)
    assert rc == tg.TG_OK, tg.tg_status_string(rc)
    check_close(c, oracle.gemm(p), dtype, what=f"permA partial atom {force}")
    check_padding(c, N)


@pytest.mark.parametrize("force", [None, "pair=1,bn=256", "pair=0,bn=192"])
def test_row_major_b_with_partial_atom(tg, force):
    # N = 1000 with ldb = 1008: the last atom holds 40 of 64 columns
    M, N, K = 640, 1000, 900
    p = synthetic.gemm_problem(M, N, K, F16, 42, lda=904, ldb=1008, scale=True)
    c, rc = run_gemm(tg, p, ldc=N + 8, force=force)
    assert rc == tg.TG_OK, tg.tg_status_string(rc)
    check_close(c, oracle.gemm(p), F16, what=f"B partial atom {force}")
    check_padding(c, N)


@pytest.mark.parametrize("force", [None, "pair=1,bn=256"])
def test_operand_flush_against_the_end_of_its_allocation(tg, force):
    import os
    import torch
    # A's storage (K x M, lda = M) ends exactly at the end of its allocation
    M, N, K = 1000, 512, 1048
    p = synthetic.gemm_problem(M, N, K, F16, 43, permA=1)
    buf = TightBuffer(p["A"], 2 << 20)
    try:
        B = dev(p["B"])
        C = torch.full((M, N + 8), SENTINEL, dtype=torch.int16, device="cuda")
        old = os.environ.get("TG_FORCE_CONFIG")
        if force:
            os.environ["TG_FORCE_CONFIG"] = force
        try:
            rc = tg.tg_gemm(M, N, K, buf.addr, M, 1, B, N, 0, C, N + 8, F16, None)
        finally:
            if force:
                if old is None:
                    del os.environ["TG_FORCE_CONFIG"]
                else:
                    os.environ["TG_FORCE_CONFIG"] = old
        torch.cuda.synchronize()
        assert rc == tg.TG_OK, tg.tg_status_string(rc)
        c = host_bits(C)
    finally:
        buf.free()
    check_close(c, oracle.gemm(p), F16, what="tight allocation")
    check_padding(c, N)
