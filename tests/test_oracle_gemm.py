"""Pins for the fp64 GEMM oracle (no GPU).

Each check ties the oracle to something other than itself: library decoders
for every 16-bit pattern, closed forms (all-ones, identities, outer products),
and exact rational brute force on tiny shapes with inputs that fp64 represents
exactly, so a dropped term, a wrong sign, a wrong index or a transposed operand
anywhere in the oracle fails at least one of them.
"""
from fractions import Fraction
import itertools

import numpy as np
import pytest

import oracle
import synthetic
from synthetic import F16, BF16
from conftest import load_golden

NAN_F16 = 0x7E00
NAN_BF16 = 0x7FC0


def bits(values, dtype):
    return synthetic.round_to_bits(np.asarray(values, dtype=np.float64), dtype)


def problem(A, B, dtype, permA=0, permB=0, lda=None, ldb=None, bias=None, scale=None,
            relu=False, R=None, ldr=None):
    """Wraps logical fp64 matrices (exact in dtype) into storage buffers.

    Padding columns are filled with NaN patterns: if the oracle ever reads one,
    the result turns NaN and the exact comparisons fail.
    """
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    nan = NAN_F16 if dtype == F16 else NAN_BF16
    sa = A if permA == 0 else A.T
    sb = B if permB == 0 else B.T
    lda = sa.shape[1] if lda is None else lda
    ldb = sb.shape[1] if ldb is None else ldb
    bufA = np.full((sa.shape[0], lda), nan, dtype=np.uint16)
    bufA[:, :sa.shape[1]] = bits(sa, dtype)
    bufB = np.full((sb.shape[0], ldb), nan, dtype=np.uint16)
    bufB[:, :sb.shape[1]] = bits(sb, dtype)
    p = {"M": M, "N": N, "K": K, "dtype": dtype, "permA": permA, "permB": permB,
         "lda": lda, "ldb": ldb, "A": bufA, "B": bufB, "relu": relu,
         "bias": None if bias is None else bits(bias, dtype),
         "scale": None if scale is None else bits(scale, dtype), "R": None, "ldr": 0}
    if R is not None:
        R = np.asarray(R, dtype=np.float64)
        ldr = N if ldr is None else ldr
        bufR = np.full((M, ldr), nan, dtype=np.uint16)
        bufR[:, :N] = bits(R, dtype)
        p["R"], p["ldr"] = bufR, ldr
    return p


# --- decoders ---------------------------------------------------------------

def test_decode_f16_every_pattern_matches_numpy():
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode(allbits, F16)
    ref = allbits.view(np.float16).astype(np.float64)
    np.testing.assert_array_equal(ours, ref)  # NaN positions compare equal


def test_decode_bf16_every_pattern_matches_fp32_widening():
    allbits = np.arange(65536, dtype=np.uint32)
    ours = oracle.decode(allbits.astype(np.uint16), BF16)
    ref = (allbits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    np.testing.assert_array_equal(ours, ref)


# --- generator --------------------------------------------------------------

def test_splitmix64_published_vector():
    g = load_golden("splitmix64.json")
    got = [int(v) for v in synthetic.splitmix64(g["seed"], 0, len(g["outputs"]))]
    assert got == [int(v) for v in g["outputs"]]


def _nearest_even_bf16(x: float) -> int:
    """Brute force: the bf16 value nearest to x (exact rationals), ties to even."""
    f = Fraction(x)
    if f == 0:
        return 0
    sign = 0x8000 if f < 0 else 0
    a = abs(f)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (e - 7)
    q, r = divmod(a, ulp)
    q = int(q)
    if r * 2 > ulp or (r * 2 == ulp and q % 2 == 1):
        q += 1
    if q == 256:
        q, e = 128, e + 1
    return sign | ((e + 127) << 7) | (q - 128)


def test_bf16_rounding_matches_exact_nearest_even():
    rng = np.random.default_rng(5)
    xs = list(rng.uniform(-4, 4, 3000)) + list(synthetic.Stream(3).normal(500, 0.5))
    # exact ties and their neighbours
    for m in range(128, 256, 7):
        for e in (-3, 0, 1):
            mid = (m + 0.5) * 2.0 ** (e - 7)
            xs += [mid, -mid, np.nextafter(mid, 0), np.nextafter(mid, 10)]
    ours = synthetic.round_f64_to_bf16_bits(np.array(xs))
    ref = np.array([_nearest_even_bf16(x) for x in xs], dtype=np.uint16)
    np.testing.assert_array_equal(ours, ref)


# --- closed forms -----------------------------------------------------------

@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (5, 7, 37), (16, 9, 128), (3, 130, 1000)])
def test_all_ones_gives_K(dtype, M, N, K):
    p = problem(np.ones((M, K)), np.ones((K, N)), dtype)
    y = oracle.gemm(p)
    assert np.all(y == K)


@pytest.mark.parametrize("permA,permB", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_identity_A_returns_B(permA, permB):
    K, N = 13, 11
    B = synthetic.Stream(1).uniform(K * N).reshape(K, N)
    B = synthetic.round_to_bits(B, F16).view(np.float16).astype(np.float64)
    p = problem(np.eye(K), B, F16, permA=permA, permB=permB, lda=K + 5 if permA else None,
                ldb=(N + 3) if permB == 0 else K + 2)
    np.testing.assert_array_equal(oracle.gemm(p), B)


@pytest.mark.parametrize("permA,permB", [(0, 0), (1, 1)])
def test_identity_B_returns_A(permA, permB):
    M, K = 9, 12
    A = synthetic.Stream(2).uniform(M * K).reshape(M, K)
    A = synthetic.round_to_bits(A, BF16)
    A = oracle.decode(A, BF16)
    p = problem(A, np.eye(K), BF16, permA=permA, permB=permB)
    np.testing.assert_array_equal(oracle.gemm(p), A)


def test_K1_outer_product():
    a = np.array([[0.5], [-2.0], [3.0], [0.25]])
    b = np.array([[1.0, -1.5, 4.0, 0.125, 8.0]])
    y = oracle.gemm(problem(a, b, F16))
    np.testing.assert_array_equal(y, a @ b)  # products of dyadics: exact


def test_single_nonzero_column():
    M, N, K, k0 = 6, 5, 9, 4
    A = np.zeros((M, K))
    A[:, k0] = [1, -2, 3, -4, 5, -6]
    B = np.arange(K * N, dtype=np.float64).reshape(K, N) - 20
    y = oracle.gemm(problem(A, B, F16))
    np.testing.assert_array_equal(y, np.outer(A[:, k0], B[k0, :]))


# --- exact brute force ------------------------------------------------------

def _brute(A, B, bias, scale, relu, R):
    M, K = len(A), len(A[0])
    N = len(B[0])
    Y = [[None] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                acc += Fraction(A[m][k]) * Fraction(B[k][n])
            if scale is not None:
                acc *= Fraction(scale[m])
            if bias is not None:
                acc += Fraction(bias[n])
            if relu:
                acc = max(acc, Fraction(0))
            if R is not None:
                acc += Fraction(R[m][n])
            Y[m][n] = acc
    return Y


@pytest.mark.parametrize("seed", range(12))
def test_bruteforce_exact_tiny(seed):
    rng = np.random.default_rng(100 + seed)
    dims = [1, 2, 3, 5, 7, 9]
    M, N, K = (int(rng.choice(dims)) for _ in range(3))
    dtype = F16 if seed % 2 == 0 else BF16
    # small integers and dyadic fractions: exact in both dtypes and in fp64 sums
    A = rng.integers(-6, 7, (M, K)) / rng.choice([1, 2, 4, 8], (M, K))
    B = rng.integers(-6, 7, (K, N)) / rng.choice([1, 2, 4, 8], (K, N))
    bias = rng.integers(-8, 9, N) / 4 if seed % 3 else None
    scale = rng.integers(-4, 5, M) / 2 if seed % 4 else None
    relu = bool(seed % 2)
    R = rng.integers(-8, 9, (M, N)) / 8 if seed % 5 else None
    permA, permB = seed % 2, (seed // 2) % 2
    p = problem(A, B, dtype, permA=permA, permB=permB,
                lda=(K if permA == 0 else M) + seed % 3,
                ldb=(N if permB == 0 else K) + (seed + 1) % 3,
                bias=bias, scale=scale, relu=relu, R=R, ldr=N + seed % 2 if R is not None else None)
    y = oracle.gemm(p)
    ref = _brute(A.tolist(), B.tolist(), None if bias is None else bias.tolist(),
                 None if scale is None else scale.tolist(), relu,
                 None if R is None else R.tolist())
    for m in range(M):
        for n in range(N):
            assert Fraction(y[m, n]) == ref[m][n], (m, n)


# --- layout handling and epilogue special cases -----------------------------

def test_permute_equals_materialised_transpose():
    p = synthetic.gemm_problem(37, 23, 41, F16, 7, lda=45, ldb=29)
    y0 = oracle.gemm(p)
    q = dict(p)
    q["A"] = np.ascontiguousarray(p["A"][:, :41].T)
    q["permA"], q["lda"] = 1, 37
    q["B"] = np.ascontiguousarray(p["B"][:, :23].T)
    q["permB"], q["ldb"] = 1, 41
    np.testing.assert_array_equal(oracle.gemm(q), y0)


def test_row_range_is_a_slice():
    p = synthetic.gemm_problem(40, 17, 33, BF16, 8, bias=True, scale=True, residual=True)
    p["relu"] = True
    full = oracle.gemm(p)
    np.testing.assert_array_equal(oracle.gemm(p, rows=(11, 29)), full[11:29])


def test_neutral_epilogue_is_plain_gemm():
    M, N, K = 10, 12, 50
    p = synthetic.gemm_problem(M, N, K, F16, 9)
    plain = oracle.gemm(p)
    q = dict(p, bias=bits(np.zeros(N), F16), scale=bits(np.ones(M), F16), relu=False,
             R=bits(np.zeros((M, N)), F16), ldr=N)
    np.testing.assert_array_equal(oracle.gemm(q), plain)


def test_zero_A_gives_relu_bias_plus_residual():
    M, N, K = 7, 9, 20
    rng = np.random.default_rng(3)
    bias = rng.integers(-8, 9, N) / 4
    R = rng.integers(-8, 9, (M, N)) / 8
    p = problem(np.zeros((M, K)), rng.integers(-3, 4, (K, N)).astype(float), F16,
                bias=bias, relu=True, R=R)
    np.testing.assert_array_equal(oracle.gemm(p), np.maximum(bias, 0)[None, :] + R)


def test_negative_products_under_relu_leave_residual():
    M, N, K = 5, 6, 31
    R = np.arange(M * N).reshape(M, N) / 16 - 1
    p = problem(-np.ones((M, K)), np.ones((K, N)), BF16, relu=True, R=R)
    np.testing.assert_array_equal(oracle.gemm(p), R)


def test_scale_then_bias_order():
    # scale is applied to the product before the bias: y = s*acc + b, not s*(acc + b)
    p = problem(np.full((1, 4), 1.0), np.full((4, 1), 1.0), F16, bias=[3.0], scale=[2.0])
    assert oracle.gemm(p)[0, 0] == 2.0 * 4 + 3.0


def test_rejects_bad_arguments():
    p = synthetic.gemm_problem(4, 4, 4, F16, 1)
    with pytest.raises(ValueError):
        oracle.gemm(p, rows=(0, 5))
    with pytest.raises(ValueError):
        oracle.gemm(dict(p, dtype=2))
