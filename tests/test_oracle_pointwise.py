"""Pins of the pointwise oracle (no GPU): it must agree with things other
than itself -- the GEMM oracle with an identity right operand (an exact fp64
reduction of the same epilogue), closed forms of the broadcasting rules, and
the epilogue's order on hand-picked values."""
import numpy as np
import pytest

import oracle
import synthetic
from synthetic import F16, BF16

ONE = {F16: 0x3C00, BF16: 0x3F80}
TWO = {F16: 0x4000, BF16: 0x4000}
MINUS_ONE = {F16: 0xBC00, BF16: 0xBF80}
HALF = {F16: 0x3800, BF16: 0x3F00}


def identity_bits(n, dtype):
    b = np.zeros((n, n), dtype=np.uint16)
    np.fill_diagonal(b, ONE[dtype])
    return b


@pytest.mark.parametrize("permX", [0, 1])
@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("epi", [{}, dict(bias=True), dict(scale=True, relu=True),
                                 dict(bias=True, scale=True, residual=True, relu=True)])
def test_equals_gemm_with_identity(permX, dtype, epi):
    M, N = 7, 13
    flags = dict(epi)
    relu = flags.pop("relu", False)
    p = synthetic.pointwise_problem(M, N, dtype, 11 + permX, permX=permX, ldx=(N if permX == 0 else M) + 3,
                                    **flags)
    p["relu"] = relu
    g = {"M": M, "N": N, "K": N, "dtype": dtype, "permA": permX, "permB": 0,
         "A": p["X"], "lda": p["ldx"], "B": identity_bits(N, dtype), "ldb": N,
         "bias": p["bias"], "scale": p["scale"], "R": p["R"], "ldr": p["ldr"], "relu": relu}
    # X(m,n) = sum_k X(m,k) I(k,n) exactly in fp64, then the same epilogue
    assert np.array_equal(oracle.pointwise(p), oracle.gemm(g))


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_broadcast_axes(dtype):
    M, N = 5, 6
    p = synthetic.pointwise_problem(M, N, dtype, 3, scale=True)
    p["X"][:] = ONE[dtype]
    y = oracle.pointwise(p)  # all-ones X: every row is its scale_m, constant along n
    s = oracle.decode(p["scale"], dtype)
    assert np.array_equal(y, np.repeat(s[:, None], N, axis=1))
    q = synthetic.pointwise_problem(M, N, dtype, 4, bias=True)
    q["X"][:] = 0
    y = oracle.pointwise(q)  # zero X: every column is its bias_n, constant along m
    b = oracle.decode(q["bias"], dtype)
    assert np.array_equal(y, np.repeat(b[None, :], M, axis=0))


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_permute_equals_materialised_transpose(dtype):
    M, N = 9, 4
    p = synthetic.pointwise_problem(M, N, dtype, 5, permX=1, ldx=M + 2, bias=True)
    q = dict(p)
    q["permX"], q["ldx"] = 0, N
    q["X"] = np.ascontiguousarray(p["X"][:N, :M].T)
    assert np.array_equal(oracle.pointwise(p), oracle.pointwise(q))


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_epilogue_order(dtype):
    # x = 1, scale 2, bias -1: scale first gives 1 (bias first would give 0)
    p = synthetic.pointwise_problem(1, 1, dtype, 6, scale=True, bias=True, residual=True)
    p["X"][:] = ONE[dtype]
    p["scale"][:] = TWO[dtype]
    p["bias"][:] = MINUS_ONE[dtype]
    p["R"][:] = HALF[dtype]
    p["relu"] = True
    assert oracle.pointwise(p)[0, 0] == 1.5  # relu(2*1 - 1) + 0.5
    p["X"][:] = MINUS_ONE[dtype]  # relu before residual: relu(-2 - 1) + 0.5
    assert oracle.pointwise(p)[0, 0] == 0.5
    p["relu"] = False
    assert oracle.pointwise(p)[0, 0] == -2.5


def test_plain_is_the_decoded_input():
    p = synthetic.pointwise_problem(4, 8, F16, 7)
    assert np.array_equal(oracle.pointwise(p), p["X"].view(np.float16).astype(np.float64))
