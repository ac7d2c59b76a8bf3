"""tg_gemm_host: A, B, C and the epilogue operands in page-locked host memory,
copies overlapped with the block GEMMs.  Every element against the oracle,
across block boundaries (whole 256-row blocks and a ragged last block), both
perms, padded host strides and every epilogue operand; C's host padding must
survive; and the argument checks (pageable or device memory where host
memory is wanted, a short or misplaced workspace, overlap)."""
import os

import numpy as np
import pytest

import oracle
import synthetic
from synthetic import F16, BF16
from helpers import SENTINEL, check_close, check_padding

pytestmark = pytest.mark.gpu


def pinned(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).pin_memory()


def run_host(tg, p, ldc, block_rows=None, stream=None, ws_shrink=0):
    """Runs p through tg_gemm_host; returns (host C bits [M, ldc], status)."""
    import torch
    M, N, K = p["M"], p["N"], p["K"]
    h = {k: (None if p.get(k) is None else pinned(p[k])) for k in ("A", "B", "bias", "scale", "R")}
    hC = torch.full((M, ldc), SENTINEL, dtype=torch.int16).pin_memory()
    epi = tg.make_epilogue(h["bias"], h["scale"], bool(p.get("relu", False)), h["R"],
                           p.get("ldr", 0) or 0)
    old = os.environ.get("TG_HOST_BLOCK_ROWS")
    if block_rows is not None:
        os.environ["TG_HOST_BLOCK_ROWS"] = str(block_rows)
    try:
        need = tg.tg_gemm_host_workspace_size(M, N, K, p["dtype"], p["permA"], p["permB"], epi)
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        rc = tg.tg_gemm_host(M, N, K, h["A"], p["lda"], p["permA"], h["B"], p["ldb"], p["permB"],
                             hC, ldc, p["dtype"], epi, ws, need - ws_shrink, stream)
    finally:
        if block_rows is not None:
            if old is None:
                del os.environ["TG_HOST_BLOCK_ROWS"]
            else:
                os.environ["TG_HOST_BLOCK_ROWS"] = old
    torch.cuda.synchronize()
    return hC.numpy().view(np.uint16).copy(), rc


CASES = [
    # (M, N, K, permA, permB, lda pad, ldb pad, ldc pad, epilogue, block rows)
    (1, 1, 1, 0, 0, 0, 0, 0, {}, None),
    (300, 200, 100, 0, 0, 3, 5, 7, {}, 256),                  # two blocks, ragged last
    (1000, 520, 333, 1, 1, 0, 1, 0, {}, None),                # 4 blocks of 256, both perms
    (2000, 640, 512, 0, 1, 8, 0, 8,
     dict(bias=True, scale=True, relu=True, residual=True), 256),  # 8 blocks, every operand
    (777, 1001, 640, 1, 0, 5, 3, 1, dict(scale=True, residual=True), 512),
    (513, 300, 1000, 0, 0, 0, 0, 0, dict(bias=True), 4096),  # one block
    (32, 2048, 512, 0, 0, 0, 0, 0, dict(scale=True), None),   # M <= 64: the swapped-operand path
    (64, 1000, 3000, 1, 1, 0, 8, 2, dict(bias=True, residual=True, relu=True), None),
]


@pytest.mark.parametrize("M,N,K,pa,pb,lpa,lpb,lpc,epi,rows", CASES)
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_matches_the_oracle(tg, M, N, K, pa, pb, lpa, lpb, lpc, epi, rows, dtype):
    flags = dict(epi)
    relu = flags.pop("relu", False)
    if flags.get("residual"):
        flags["ldr"] = N + 3
    a_w = K if pa == 0 else M
    b_w = N if pb == 0 else K
    p = synthetic.gemm_problem(M, N, K, dtype, 500 + M + K, permA=pa, permB=pb, lda=a_w + lpa,
                               ldb=b_w + lpb, **flags)
    p["relu"] = relu
    c, rc = run_host(tg, p, N + lpc, block_rows=rows)
    assert rc == tg.TG_OK, tg.tg_status_string(rc)
    st, code = tg.tg_debug_status()
    assert st == tg.TG_OK, hex(code)
    check_close(c, oracle.gemm(p), dtype, what=f"host {M}x{N}x{K}")
    check_padding(c, N)


def test_on_a_side_stream_and_workspace_reuse(tg):
    import torch
    s = torch.cuda.Stream()
    for seed in (1, 2):
        p = synthetic.gemm_problem(700, 300, 200, F16, seed, residual=True, bias=True)
        c, rc = run_host(tg, p, 300, stream=s)
        assert rc == tg.TG_OK
        check_close(c, oracle.gemm(p), F16, what=f"side stream seed {seed}")


def test_headline_shape_equals_the_device_resident_call_within_tolerance(tg):
    # 4096^3 in four 1024-row blocks against the whole-matrix device call
    import torch
    M = N = K = 4096
    p = synthetic.gemm_problem(M, N, K, F16, 1002)
    c, rc = run_host(tg, p, N)
    assert rc == tg.TG_OK
    A = torch.from_numpy(p["A"].view(np.int16)).cuda()
    B = torch.from_numpy(p["B"].view(np.int16)).cuda()
    C = torch.empty((M, N), dtype=torch.int16, device="cuda")
    need = tg.tg_gemm_workspace_size(M, N, K, F16)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
    assert tg.tg_gemm_ws(M, N, K, A, K, 0, B, N, 0, C, N, F16, None, ws, need) == tg.TG_OK
    ref = C.cpu().numpy().view(np.uint16)
    got = c.view(np.float16).astype(np.float64)
    want = ref.view(np.float16).astype(np.float64)
    assert np.all(np.abs(got - want) <= 1e-2 * np.maximum(1.0, np.abs(want)))
    for r0, r1 in ((0, 2), (511, 513), (4094, 4096)):  # across block boundaries
        check_close(c, oracle.gemm(p, rows=(r0, r1)), F16, rows=slice(r0, r1),
                    what=f"host 4096 rows {r0}..{r1}")


def test_argument_checks(tg):
    import torch
    M, N, K = 256, 256, 64
    hA = torch.zeros((M, K), dtype=torch.int16).pin_memory()
    hB = torch.zeros((K, N), dtype=torch.int16).pin_memory()
    hC = torch.zeros((M, N), dtype=torch.int16).pin_memory()
    need = tg.tg_gemm_host_workspace_size(M, N, K, F16)
    ws = torch.zeros(need + 512, dtype=torch.uint8, device="cuda")
    call = lambda A=hA, B=hB, C=hC, w=ws, nb=need, epi=None, lda=K: tg.tg_gemm_host(
        M, N, K, A, lda, 0, B, N, 0, C, N, F16, epi, w, nb)
    assert call() == tg.TG_OK
    torch.cuda.synchronize()
    assert call(A=torch.zeros((M, K), dtype=torch.int16)) == tg.TG_ERR_POINTER  # pageable
    assert call(A=torch.zeros((M, K), dtype=torch.int16, device="cuda")) == tg.TG_ERR_POINTER
    assert call(w=torch.zeros(need, dtype=torch.uint8).pin_memory()) == tg.TG_ERR_POINTER
    assert call(nb=need - 1) == tg.TG_ERR_BUFFER
    assert call(w=ws.data_ptr() + 16) == tg.TG_ERR_ALIGN
    assert call(A=hA.data_ptr() + 1) == tg.TG_ERR_ALIGN
    assert call(lda=K - 1) == tg.TG_ERR_STRIDE
    assert call(C=hA) == tg.TG_ERR_OVERLAP
    assert call(w=None) == tg.TG_ERR_INVALID_ARG
    bad = tg.tg_epilogue(None, None, 2, None, 0)
    assert call(epi=bad) == tg.TG_ERR_INVALID_ARG
    torch.cuda.synchronize()
