"""tg_pointwise (the named-layout pointwise program) against the pointwise
oracle on every element: broadcasting of scale_m / bias_n, the explicit
permute, ragged and unaligned shapes, bit-exact copies and transposes when
there is no epilogue, C's padding, and the argument checks."""
import numpy as np
import pytest

import oracle
import synthetic
from synthetic import F16, BF16
from helpers import SENTINEL, check_close, check_padding, host_bits

pytestmark = pytest.mark.gpu


def placed(bits, offset):
    import torch
    flat = np.ascontiguousarray(bits).reshape(-1).view(np.int16)
    buf = torch.zeros(flat.size + offset + 8, dtype=torch.int16, device="cuda")
    buf[offset:offset + flat.size] = torch.from_numpy(flat).cuda()
    return buf, buf.data_ptr() + 2 * offset


def run(tg, p, ldc, offs=None):
    import torch
    offs = offs or {}
    M, N = p["M"], p["N"]
    keep, addr = [], {}
    for name in ("X", "bias", "scale", "R"):
        if p.get(name) is None:
            addr[name] = None
            continue
        buf, a = placed(p[name], offs.get(name, 0))
        keep.append(buf)
        addr[name] = a
    c_off = offs.get("C", 0)
    cbuf = torch.full((M * ldc + c_off + 8,), SENTINEL, dtype=torch.int16, device="cuda")
    epi = tg.make_epilogue(addr["bias"], addr["scale"], bool(p.get("relu", False)), addr["R"],
                           p.get("ldr", 0) or 0)
    rc = tg.tg_pointwise(M, N, addr["X"], p["ldx"], p["permX"], cbuf.data_ptr() + 2 * c_off, ldc,
                         p["dtype"], epi)
    torch.cuda.synchronize()
    return host_bits(cbuf)[c_off:c_off + M * ldc].reshape(M, ldc), rc


SHAPES = [(1, 1), (1, 1000), (1000, 1), (33, 65), (333, 517), (2048, 3000)]
EPIS = [{}, dict(bias=True), dict(scale=True), dict(relu=True), dict(residual=True),
        dict(bias=True, scale=True, relu=True, residual=True)]


@pytest.mark.parametrize("M,N", SHAPES)
@pytest.mark.parametrize("permX", [0, 1])
@pytest.mark.parametrize("epi", EPIS)
def test_matches_oracle(tg, M, N, permX, epi):
    dtype = BF16 if (M + N + permX) % 2 else F16
    flags = dict(epi)
    relu = flags.pop("relu", False)
    if flags.get("residual"):
        flags["ldr"] = N + 5
    x_w = N if permX == 0 else M
    p = synthetic.pointwise_problem(M, N, dtype, 100 + M + N, permX=permX, ldx=x_w + 8, **flags)
    p["relu"] = relu
    ldc = N + 8
    c, rc = run(tg, p, ldc)
    assert rc == tg.TG_OK, tg.tg_status_string(rc)
    check_close(c, oracle.pointwise(p), dtype, what=f"{M}x{N} perm {permX} {epi}")
    check_padding(c, N)


@pytest.mark.parametrize("permX", [0, 1])
def test_unaligned_strides_and_pointers(tg, permX):
    M, N = 301, 259
    x_w = N if permX == 0 else M
    p = synthetic.pointwise_problem(M, N, F16, 9, permX=permX, ldx=x_w + 3, bias=True,
                                    scale=True, residual=True, ldr=N + 1)
    p["relu"] = True
    c, rc = run(tg, p, N + 3, offs=dict(X=1, C=3, R=5, bias=1, scale=7))
    assert rc == tg.TG_OK, tg.tg_status_string(rc)
    check_close(c, oracle.pointwise(p), F16, what="unaligned")
    check_padding(c, N)


@pytest.mark.parametrize("permX", [0, 1])
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_without_epilogue_copies_and_transposes_bit_exactly(tg, permX, dtype):
    M, N = 517, 333
    x_w = N if permX == 0 else M
    p = synthetic.pointwise_problem(M, N, dtype, 12, permX=permX, ldx=x_w + 16)
    c, rc = run(tg, p, N)
    assert rc == tg.TG_OK
    want = p["X"][:M, :N] if permX == 0 else p["X"][:N, :M].T
    assert np.array_equal(c, want)


def test_argument_checks(tg):
    import torch
    X = torch.zeros((64, 64), dtype=torch.int16, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.int16, device="cuda")
    assert tg.tg_pointwise(64, 64, X, 64, 0, X, 64, F16) == tg.TG_ERR_OVERLAP  # in place
    assert tg.tg_pointwise(64, 64, X, 63, 0, C, 64, F16) == tg.TG_ERR_STRIDE
    assert tg.tg_pointwise(64, 64, X, 64, 0, C, 63, F16) == tg.TG_ERR_STRIDE
    assert tg.tg_pointwise(64, 64, X.data_ptr() + 1, 64, 0, C, 64, F16) == tg.TG_ERR_ALIGN
    assert tg.tg_pointwise(0, 64, X, 64, 0, C, 64, F16) == tg.TG_ERR_INVALID_ARG
    assert tg.tg_pointwise(64, 64, X, 64, 2, C, 64, F16) == tg.TG_ERR_INVALID_ARG
    assert tg.tg_pointwise(64, 64, X, 64, 0, C, 64, 2) == tg.TG_ERR_DTYPE
    e = tg.make_epilogue(residual=C)  # residual aliases the output
    assert tg.tg_pointwise(64, 64, X, 64, 0, C, 64, F16, e) == tg.TG_ERR_OVERLAP
    host = torch.zeros((64, 64), dtype=torch.int16).pin_memory()
    assert tg.tg_pointwise(64, 64, host, 64, 0, C, 64, F16) == tg.TG_ERR_POINTER
    assert tg.tg_pointwise(64, 64, X, 64, 0, C, 64, F16) == tg.TG_OK
    torch.cuda.synchronize()


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("epi", [{}, dict(bias=True, scale=True, relu=True, residual=True)])
def test_permuted_input_with_aligned_rows(tg, dtype, epi):
    # every row starts on a 16-byte boundary: the 16-byte-vector transpose
    # path, with M and N ragged against its 64 x 64 tiles and 8-wide vectors
    M, N = 1001, 700
    flags = dict(epi)
    relu = flags.pop("relu", False)
    if flags.get("residual"):
        flags["ldr"] = 704
    p = synthetic.pointwise_problem(M, N, dtype, 31, permX=1, ldx=1008, **flags)
    p["relu"] = relu
    c, rc = run(tg, p, 704)
    assert rc == tg.TG_OK
    if not epi:
        assert np.array_equal(c[:, :N], p["X"][:N, :M].T)
    else:
        check_close(c, oracle.pointwise(p), dtype, what="aligned permuted")
    check_padding(c, N)
