"""Parity at the full sizes of the benchmark workloads, in the launch
configuration the bench uses (the default selector).

The oracle computes sampled rows one by one (first, last, middle and seeded
random rows); every element is additionally checked against an fp32 PyTorch
reference on the GPU and for finiteness, and C's padding must be untouched.
"""
import numpy as np
import pytest

import oracle
import synthetic
from synthetic import F16, BF16
from helpers import SENTINEL, check_close, check_padding, decode, dev, host_bits

pytestmark = pytest.mark.gpu

WORKLOADS = {
    # name: (M, N, K, dtype, seed, kwargs)
    "fp16_4096": (4096, 4096, 4096, F16, 1002, {}),
    "bf16_4096": (4096, 4096, 4096, BF16, 1002, {}),
    "fp16_8192x8192x4096_fused": (8192, 8192, 4096, F16, 1003,
                                  dict(bias=True, scale=True, residual=True, relu=True)),
    "fp16_4000x3000x1000_strided": (4000, 3000, 1000, F16, 1004,
                                    dict(permA=1, ldb=3064, dist="normal", bias=True)),
    "bf16_16384x1024x8192_scale": (16384, 1024, 8192, BF16, 1005, dict(scale=True)),
    "bf16_32x16384x16384_scale": (32, 16384, 16384, BF16, 1005, dict(scale=True)),
}


def torch_reference(p):
    """fp32 reference of the same op with PyTorch on the GPU (a cross-check)."""
    import torch
    f = lambda a: torch.from_numpy(decode(a, p["dtype"]).astype(np.float32)).cuda()
    M, N, K = p["M"], p["N"], p["K"]
    A = f(p["A"])
    A = A[:, :K] if p["permA"] == 0 else A[:, :M].T
    B = f(p["B"])
    B = B[:, :N] if p["permB"] == 0 else B[:, :K].T
    y = A @ B
    if p.get("scale") is not None:
        y = y * f(p["scale"])[:, None]
    if p.get("bias") is not None:
        y = y + f(p["bias"])[None, :]
    if p.get("relu"):
        y = torch.relu(y)
    if p.get("R") is not None:
        y = y + f(p["R"])[:, :N]
    return y


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_workload(tg, name):
    import torch
    M, N, K, dtype, seed, kw = WORKLOADS[name]
    kw = dict(kw)
    relu = kw.pop("relu", False)
    p = synthetic.gemm_problem(M, N, K, dtype, seed, **kw)
    p["relu"] = relu
    ldc = N + 8
    A, B = dev(p["A"]), dev(p["B"])
    bias = dev(p["bias"]) if p["bias"] is not None else None
    scale = dev(p["scale"]) if p["scale"] is not None else None
    R = dev(p["R"]) if p["R"] is not None else None
    C = torch.full((M, ldc), SENTINEL, dtype=torch.int16, device="cuda")
    epi = tg.make_epilogue(bias, scale, relu, R, p["ldr"])
    tg.gemm(M, N, K, A, p["lda"], p["permA"], B, p["ldb"], p["permB"], C, ldc, dtype, epi)
    torch.cuda.synchronize()
    st, code = tg.tg_debug_status()
    assert st == tg.TG_OK, hex(code)
    c = host_bits(C)
    check_padding(c, N)
    got = decode(c[:, :N], dtype)
    assert np.all(np.isfinite(got))

    # every element against the fp32 GPU reference
    ref32 = torch_reference(p).double().cpu().numpy()
    err = np.abs(got - ref32) / np.maximum(1.0, np.abs(ref32))
    assert err.max() <= 1e-2, f"max normalised error vs fp32 reference {err.max()}"

    # sampled rows against the fp64 oracle
    rng = np.random.default_rng(seed)
    rows = sorted(set([0, M - 1, M // 2] + list(rng.integers(0, M, 29))))
    if M <= 64:
        rows = list(range(M))
        ref = oracle.gemm(p)  # one call: the oracle parallelises over rows
    else:
        ref = np.concatenate([oracle.gemm(p, rows=(r, r + 1)) for r in rows])
    check_close(c[rows], ref, dtype, what=name)
