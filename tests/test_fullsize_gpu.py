"""Parity at the full sizes of the benchmark workloads, element by element
against the fp64 oracle, in the very launches the bench times.

For each GEMM workload the oracle computes every output element once; then
* the bench's own call (bench.DeviceProblem: tg_gemm_ws with the default
  stream-K workspace, C with ldc = N) runs twice in a row -- the second call
  reuses the workspace the first one left -- and every element of C is
  compared, and
* tg_gemm (whole tiles, no workspace) runs on a C padded with sentinels, and
  every element plus the untouched padding is checked.
The tolerance is |gpu - oracle| <= 1e-2 * max(1, |oracle|) for every element,
the standard of the execution tests "against matrix multiplication" in
pbelevich.github.io "My Triton From Scratch Part 16: Register Tiles",
section "Tests cover the mapping as a contract".  The two pointwise programs
the bench times are checked the same way.
"""
import numpy as np
import pytest

import bench
import oracle
from helpers import SENTINEL, check_close, check_padding, dev, host_bits

pytestmark = pytest.mark.gpu

# the headline and every other GEMM workload the bench times
GEMM_WORKLOADS = ["fp16_4096"] + list(bench.OTHER_WORKLOADS)


def _status_ok(tg):
    st, code = tg.tg_debug_status()
    assert st == tg.TG_OK, hex(code)


@pytest.mark.parametrize("key", GEMM_WORKLOADS)
def test_benched_launch_matches_oracle_everywhere(tg, key):
    import torch
    p = bench.make_problem(bench.workload_specs()[key])
    M, N, K, dtype = p["M"], p["N"], p["K"], p["dtype"]
    ref = oracle.gemm(p)  # every row; the oracle spreads rows over all host cores

    # the bench's launch, twice in a row on one workspace
    dp = bench.DeviceProblem(tg, p, stream_k=True)
    stream = torch.cuda.Stream()
    for call in ("first", "second"):
        dp.C.fill_(SENTINEL)
        dp.call(stream)
        torch.cuda.synchronize()
        _status_ok(tg)
        check_close(host_bits(dp.C), ref, dtype, what=f"{key} ({dp.config}), {call} call")
    del dp

    # tg_gemm: whole tiles, C padded with sentinels that must survive
    ldc = N + 8
    A, B = dev(p["A"]), dev(p["B"])
    bias = dev(p["bias"]) if p["bias"] is not None else None
    scale = dev(p["scale"]) if p["scale"] is not None else None
    R = dev(p["R"]) if p["R"] is not None else None
    C = torch.full((M, ldc), SENTINEL, dtype=torch.int16, device="cuda")
    epi = tg.make_epilogue(bias, scale, p["relu"], R, p["ldr"])
    tg.gemm(M, N, K, A, p["lda"], p["permA"], B, p["ldb"], p["permB"], C, ldc, dtype, epi)
    torch.cuda.synchronize()
    _status_ok(tg)
    c = host_bits(C)
    check_padding(c, N)
    check_close(c, ref, dtype, what=f"{key} through tg_gemm")


@pytest.mark.parametrize("key", [k for k, _ in bench.POINTWISE_WORKLOADS])
def test_benched_pointwise_matches_oracle_everywhere(tg, key):
    import torch
    pp = bench.make_pointwise(key)
    ref = oracle.pointwise(pp)
    dpw = bench.DevicePointwise(tg, pp)
    dpw.C.fill_(SENTINEL)
    dpw.call(torch.cuda.current_stream())
    torch.cuda.synchronize()
    check_close(host_bits(dpw.C), ref, pp["dtype"], what=key)
