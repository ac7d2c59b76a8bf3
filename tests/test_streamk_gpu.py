"""tg_gemm_ws: tail tiles shared out in K-ranges ("stream-K") with a caller
workspace.  Parity with the oracle on every element, reproducible bits, the
workspace left zeroed, and its checks."""
import os

import numpy as np
import pytest

import oracle
import synthetic
from synthetic import F16, BF16
from helpers import SENTINEL, check_close, check_padding, dev, host_bits

pytestmark = pytest.mark.gpu


def run_ws(tg, p, force, ldc=None, ws_extra=0, ws=None):
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
    os.environ["TG_FORCE_CONFIG"] = force
    try:
        cfg = tg.parse_config(tg.tg_query_config_ws(M, N, K, p["dtype"], p["permA"], p["permB"], epi))
        nbytes = tg.tg_gemm_workspace_size(M, N, K, p["dtype"], p["permA"], p["permB"], epi)
        assert nbytes == cfg["ws_bytes"]
        if ws is None:
            ws = torch.zeros(nbytes + ws_extra + 256, dtype=torch.uint8, device="cuda")
        rc = tg.tg_gemm_ws(M, N, K, A, p["lda"], p["permA"], B, p["ldb"], p["permB"], C, ldc,
                           p["dtype"], epi, ws, ws.numel())
    finally:
        if old is None:
            del os.environ["TG_FORCE_CONFIG"]
        else:
            os.environ["TG_FORCE_CONFIG"] = old
    torch.cuda.synchronize()
    return host_bits(C), rc, cfg, ws


CASES = [
    # (M, N, K, dtype, force, epilogue)
    (640, 256, 640, F16, "pair=0,bn=128,grid=4,sk=1", {}),
    (700, 300, 1000, BF16, "pair=0,bn=128,grid=4,sk=1", dict(bias=True, scale=True, residual=True, relu=True)),
    (1000, 520, 1200, F16, "pair=1,bn=256,grid=10,sk=1", {}),
    (1000, 520, 1200, BF16, "pair=1,bn=256,grid=10,sk=1", dict(bias=True, residual=True)),
    (600, 700, 900, F16, "pair=1,bn=128,grid=8,sk=1", dict(scale=True, relu=True)),
    (520, 300, 2000, F16, "pair=0,bn=256,grid=8,sk=1", {}),            # no whole-tile waves at all
    (32, 1000, 2048, BF16, "pair=0,bn=32,swap=1,grid=16,sk=1", dict(scale=True)),
    (200, 900, 3000, F16, "pair=0,bn=64,grid=12,sk=1", dict(bias=True)),
    # column bias held per lane, in 224-wide tiles over several tile columns (odd ones too)
    (1000, 712, 2048, F16, "pair=1,bn=224,grid=10,sk=1", dict(bias=True)),
]


@pytest.mark.parametrize("M,N,K,dtype,force,epi", CASES)
@pytest.mark.parametrize("perm", [(0, 0), (1, 1)])
def test_stream_k_parity(tg, M, N, K, dtype, force, epi, perm):
    flags = dict(epi)
    relu = flags.pop("relu", False)
    up8 = lambda x: -(-x // 8) * 8  # row strides in whole 16-byte units
    lda = up8(K if perm[0] == 0 else M)
    ldb = up8(N if perm[1] == 0 else K)
    if flags.get("residual"):
        flags["ldr"] = up8(N)
    p = synthetic.gemm_problem(M, N, K, dtype, 91 + M + K, permA=perm[0], permB=perm[1],
                               lda=lda, ldb=ldb, **flags)
    p["relu"] = relu
    c, rc, cfg, ws = run_ws(tg, p, force, ldc=-(-N // 8) * 8 + 8)
    assert rc == tg.TG_OK, tg.tg_status_string(rc)
    assert cfg["sk_tiles"] > 0, cfg  # the case exercises the split
    st, code = tg.tg_debug_status()
    assert st == tg.TG_OK, hex(code)
    check_close(c, oracle.gemm(p), dtype, what=force)
    check_padding(c, N)
    # counters are back to zero, so the same workspace serves the next call
    workers = cfg["grid"] // 2 if cfg["pair"] else cfg["grid"]
    counters = ws[: workers * 2 * 4].view(dtype=__import__("torch").int32)
    assert int(counters.abs().sum().item()) == 0
    c2, rc2, _, _ = run_ws(tg, p, force, ldc=-(-N // 8) * 8 + 8, ws=ws)
    assert rc2 == tg.TG_OK and np.array_equal(c, c2)  # reproducible bits


def test_stream_k_matches_whole_tiles_closely(tg):
    p = synthetic.gemm_problem(1000, 520, 1200, F16, 5)
    c_sk, rc, cfg, _ = run_ws(tg, p, "pair=1,bn=256,grid=10,sk=1")
    assert rc == tg.TG_OK and cfg["sk_tiles"] > 0
    from helpers import run_gemm, decode
    c_dp, rc = run_gemm(tg, p, force="pair=1,bn=256,grid=10,sk=1")
    assert rc == tg.TG_OK
    a, b = decode(c_sk, F16), decode(c_dp, F16)
    # both round the same fp32 sum computed in a different association
    assert np.max(np.abs(a - b) / np.maximum(1, np.abs(b))) <= 2e-3


def test_workspace_checks(tg):
    import torch
    p = synthetic.gemm_problem(640, 256, 640, F16, 3)
    A, B = dev(p["A"]), dev(p["B"])
    C = torch.empty((640, 256), dtype=torch.int16, device="cuda")
    old = os.environ.get("TG_FORCE_CONFIG")
    os.environ["TG_FORCE_CONFIG"] = "pair=0,bn=128,grid=4,sk=1"
    try:
        need = tg.tg_gemm_workspace_size(640, 256, 640, F16)
        assert need > 0
        ws = torch.zeros(need + 512, dtype=torch.uint8, device="cuda")
        call = lambda w, n: tg.tg_gemm_ws(640, 256, 640, A, 640, 0, B, 256, 0, C, 256, F16, None, w, n)
        assert call(ws, need - 1) == tg.TG_ERR_BUFFER
        assert call(ws.data_ptr() + 16, need) == tg.TG_ERR_ALIGN
        assert call(C, need) in (tg.TG_ERR_OVERLAP, tg.TG_ERR_BUFFER)
        host = torch.zeros(need + 256, dtype=torch.uint8).pin_memory()
        assert call(host, need) == tg.TG_ERR_POINTER
        assert call(None, 0) == tg.TG_OK  # no workspace: whole tiles
        assert call(ws, need) == tg.TG_OK
        torch.cuda.synchronize()
    finally:
        if old is None:
            del os.environ["TG_FORCE_CONFIG"]
        else:
            os.environ["TG_FORCE_CONFIG"] = old
