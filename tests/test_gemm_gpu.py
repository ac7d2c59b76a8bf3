"""Parity of the tcgen05 GEMM (through the C ABI) with the fp64 oracle.

Small and ragged shapes are compared on every element; the full-size
workloads on sampled rows that the oracle computes one by one.  Tolerance:
|gpu - oracle| <= 1e-2 * max(1, |oracle|) with inputs of magnitude <= ~2 and
K <= 16384 (fp32 accumulation; fp16/bf16 output rounding is at most 2^-9
relative).  The cases follow the GPU execution tests listed in
pbelevich.github.io "My Triton From Scratch Part 16: Register Tiles"
("Tests cover the mapping as a contract": one K tile, several K tiles,
partial M, N and K edges) plus the operand permutes, strides and epilogue
operands of ninetoothed.org "Named layouts".
"""
import numpy as np
import pytest

import oracle
import synthetic
from synthetic import F16, BF16
from helpers import run_gemm, check_close, check_padding

pytestmark = pytest.mark.gpu


def full_check(tg, p, ldc=None, force=None, what=""):
    c, rc = run_gemm(tg, p, ldc=ldc, force=force)
    assert rc == tg.TG_OK, tg.tg_status_string(rc)
    ref = oracle.gemm(p)
    err = check_close(c, ref, p["dtype"], what=what)
    check_padding(c, p["N"])
    st, code = tg.tg_debug_status()
    assert st == tg.TG_OK, hex(code)
    return err


def test_small_128_cube(tg):
    # the 128^3 fp16 row-major workload (seed 1000 + config index)
    p = synthetic.gemm_problem(128, 128, 128, F16, 1001)
    full_check(tg, p, what="128^3")


@pytest.mark.parametrize("M,N,K", [
    (128, 256, 64),     # one K tile
    (256, 128, 320),    # several K tiles, K multiple of 64
    (200, 130, 100),    # partial M, N, K edges
    (17, 40, 72),       # M and N below one tile
    (130, 70, 8),       # K below the 64-wide K block
    (64, 64, 1),        # K = 1 (outer product), lda padded to 8
    (333, 517, 1111),   # several tiles, all edges ragged
])
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_edges(tg, M, N, K, dtype):
    lda = max(8, -(-K // 8) * 8)
    p = synthetic.gemm_problem(M, N, K, dtype, 7 + M + N + K, lda=lda, ldb=-(-N // 8) * 8 + 8)
    full_check(tg, p, ldc=-(-N // 8) * 8 + 16, what=f"{M}x{N}x{K}")


@pytest.mark.parametrize("permA,permB", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_permutes_and_strides(tg, permA, permB, dtype):
    M, N, K = 300, 260, 400
    up8 = lambda x: -(-x // 8) * 8  # row strides must be whole 16-byte units
    lda = up8(K if permA == 0 else M) + 24
    ldb = up8(N if permB == 0 else K) + 64
    p = synthetic.gemm_problem(M, N, K, dtype, 11 + 2 * permA + permB, permA=permA, permB=permB,
                               lda=lda, ldb=ldb, dist="normal", sigma=0.5)
    full_check(tg, p, ldc=up8(N) + 8, what=f"perm {permA}{permB}")


EPILOGUES = [
    dict(bias=True), dict(scale=True), dict(relu=True), dict(residual=True),
    dict(bias=True, scale=True, relu=True, residual=True),
    dict(scale=True, relu=True), dict(bias=True, residual=True),
]


@pytest.mark.parametrize("epi", EPILOGUES)
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_epilogue_combinations(tg, epi, dtype):
    M, N, K = 260, 200, 192
    flags = dict(epi)
    relu = flags.pop("relu", False)
    p = synthetic.gemm_problem(M, N, K, dtype, 21, ldr=N + 8 if flags.get("residual") else None,
                               **flags)
    p["relu"] = relu
    full_check(tg, p, ldc=N + 24, what=str(epi))  # N = 200: both strides whole 16-byte units


CONFIGS = [
    "pair=0,bn=32,swap=1", "pair=0,bn=64,swap=1", "pair=0,bn=128,swap=1", "pair=0,bn=256,swap=1",
    "pair=0,bn=64,swap=0", "pair=0,bn=128,swap=0", "pair=0,bn=192,swap=0", "pair=0,bn=224,swap=0",
    "pair=0,bn=256,swap=0", "pair=0,bn=128,group_m=1", "pair=0,bn=256,grid=7",
    "pair=1,bn=128,swap=0", "pair=1,bn=192,swap=0", "pair=1,bn=224,swap=0", "pair=1,bn=256,swap=0",
    "pair=1,bn=224,swap=1", "pair=1,bn=256,swap=1", "pair=1,bn=256,grid=6", "pair=1,bn=128,group_m=1",
]


def test_selector_reports_forced_configuration(tg):
    import os
    old = os.environ.get("TG_FORCE_CONFIG")
    try:
        os.environ["TG_FORCE_CONFIG"] = "pair=1,bn=224,swap=0"
        cfg = tg.parse_config(tg.tg_query_config(4096, 4096, 4096, F16))
        assert (cfg["pair"], cfg["bn"], cfg["bm"], cfg["swap"]) == (1, 224, 256, 0)
        assert cfg["grid"] % 2 == 0
    finally:
        if old is None:
            os.environ.pop("TG_FORCE_CONFIG", None)
        else:
            os.environ["TG_FORCE_CONFIG"] = old


@pytest.mark.parametrize("force", CONFIGS)
@pytest.mark.parametrize("permA,permB", [(0, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [
    (184, 328, 264),  # ragged against every tile; dense strides stay 16-byte units
    (320, 448, 200),  # M, N whole 64-wide atoms (MN-major stages as one 3-D box), K ragged
    (712, 696, 136),  # partial last atom in M and N: that CTA's stages use 2-D boxes, the rest 3-D
])
def test_every_tile_configuration(tg, force, permA, permB, M, N, K):
    p = synthetic.gemm_problem(M, N, K, BF16, 31, permA=permA, permB=permB,
                               bias=True, scale=True, residual=True)
    p["relu"] = True
    full_check(tg, p, force=force, what=force)


@pytest.mark.parametrize("force", ["pair=1,bn=224,swap=0", "pair=0,bn=224,swap=0", "pair=1,bn=256,swap=0",
                                   "pair=1,bn=224,grid=4,swap=0"])
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_column_bias_across_tiles(tg, force, dtype):
    # Each lane loads its column's bias once per tile; a chunk broadcasts the
    # values to its rows.  N spans several tile columns (odd ones included)
    # and ends mid-chunk; grid=4 gives every worker several tiles, so the
    # main and helper warps split only the last one.
    p = synthetic.gemm_problem(520, 712, 200, dtype, 71, bias=True)
    full_check(tg, p, force=force, what=f"bias {force}")


@pytest.mark.parametrize("force", ["pair=1,bn=256,swap=0", "pair=0,bn=128,swap=0", "pair=0,bn=192,swap=0",
                                   "pair=0,bn=256,swap=0", "pair=1,bn=256,grid=4,swap=0"])
@pytest.mark.parametrize("K", [384, 448])
def test_two_kblock_boxes(tg, force, K):
    # Whole-tile kernels fill two ring slots per barrier transaction; with A
    # K-major, B N-major (N a multiple of 64) and K a multiple of 64, each
    # operand's pair of K-blocks arrives as one 3-D (A) or 4-D (B) box.  K =
    # 448 leaves an odd last K-block, which takes the one-block boxes; M is
    # ragged (rows past M read as zeros).
    p = synthetic.gemm_problem(600, 704, K, F16, 81, bias=True, residual=True)
    full_check(tg, p, force=force, what=f"2k {force}")


def test_swap_selected_for_small_M(tg):
    cfg = tg.parse_config(tg.tg_query_config(32, 16384, 16384, BF16))
    assert cfg["swap"] == 1
    p = synthetic.gemm_problem(32, 2048, 1024, BF16, 41, scale=True)
    full_check(tg, p, what="swap")


def test_repeatable_bits(tg):
    p = synthetic.gemm_problem(384, 512, 640, F16, 51, bias=True)
    c1, _ = run_gemm(tg, p)
    c2, _ = run_gemm(tg, p)
    assert np.array_equal(c1, c2)


def test_inputs_are_not_modified(tg):
    import torch
    from helpers import dev, host_bits
    p = synthetic.gemm_problem(256, 256, 256, F16, 61, bias=True, scale=True, residual=True)
    A, B = dev(p["A"]), dev(p["B"])
    bias, scale, R = dev(p["bias"]), dev(p["scale"]), dev(p["R"])
    C = torch.empty((256, 256), dtype=torch.int16, device="cuda")
    epi = tg.make_epilogue(bias, scale, True, R, 256)
    tg.gemm(256, 256, 256, A, 256, 0, B, 256, 0, C, 256, F16, epi)
    torch.cuda.synchronize()
    for t, ref in [(A, p["A"]), (B, p["B"]), (bias, p["bias"]), (scale, p["scale"]), (R, p["R"])]:
        assert np.array_equal(host_bits(t), ref)


def test_runs_on_a_side_stream(tg):
    import torch
    from helpers import dev, host_bits
    p = synthetic.gemm_problem(256, 384, 512, BF16, 71)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        A, B = dev(p["A"]), dev(p["B"])
        C = torch.empty((256, 384), dtype=torch.int16, device="cuda")
        tg.gemm(256, 384, 512, A, 512, 0, B, 384, 0, C, 384, BF16, None, s)
    s.synchronize()
    check_close(host_bits(C), oracle.gemm(p), BF16, what="side stream")


def test_pointer_checks_on_device(tg):
    import torch
    A = torch.zeros((64, 64), dtype=torch.int16, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.int16, device="cuda")
    host = torch.zeros((64, 64), dtype=torch.int16)
    # host memory is rejected, not dereferenced
    assert tg.tg_gemm(64, 64, 64, host, 64, 0, A, 64, 0, C, 64, F16) == tg.TG_ERR_POINTER
    # an operand extent that runs past the end of its allocation is rejected
    big = 1 << 30
    rc = tg.tg_gemm(64, 64, big, A, big, 0, A, 64, 0, C, 64, F16)
    assert rc in (tg.TG_ERR_POINTER, tg.TG_ERR_OVERLAP)
    assert tg.tg_gemm(64, 64, 64, A, 64, 0, A, 64, 0, A, 64, F16) == tg.TG_ERR_OVERLAP


@pytest.mark.parametrize("force", ["pair=0,bn=128", "pair=1,bn=256"])
def test_watchdog_expires_and_context_survives(tg, force):
    """A producer that never arms one k-block makes the MMA wait run out: the
    kernel must return with TG_ERR_TIMEOUT instead of hanging, and the next
    call must work normally."""
    p = synthetic.gemm_problem(256, 256, 1024, F16, 81)
    assert tg.tg_debug_configure(1_000_000, 3) == tg.TG_OK
    try:
        _, rc = run_gemm(tg, p, force=force)
        assert rc == tg.TG_OK
        st, code = tg.tg_debug_status()
        assert st == tg.TG_ERR_TIMEOUT and code != 0
    finally:
        assert tg.tg_debug_configure(0, -1) == tg.TG_OK
    full_check(tg, p, what="after watchdog")
