"""tg_gemm_ws with operands a tensor map cannot describe: base pointers off the
16-byte grid and row strides that are not whole 16-byte units.  Positive
strides of any size are valid (ninetoothed.org "Named layouts", "Runtime and
compilation"); such operands are staged through the caller's workspace.  The
results must match the oracle on every element, C's padding must survive,
and tg_gemm (no workspace) must keep refusing them."""
import numpy as np
import pytest

import oracle
import synthetic
from synthetic import F16, BF16
from helpers import SENTINEL, check_close, check_padding, host_bits

pytestmark = pytest.mark.gpu


def placed(bits, offset):
    """A device buffer holding `bits` (any shape) starting `offset` elements
    past a 256-byte-aligned allocation; returns (buffer, address)."""
    import torch
    flat = np.ascontiguousarray(bits).reshape(-1).view(np.int16)
    buf = torch.zeros(flat.size + offset + 8, dtype=torch.int16, device="cuda")
    buf[offset:offset + flat.size] = torch.from_numpy(flat).cuda()
    return buf, buf.data_ptr() + 2 * offset


def run_unaligned(tg, p, offs, ldc, use_ws=True, ws_shrink=0):
    """Runs p with each operand placed at offs[name] elements past alignment.
    Returns (C storage [M, ldc] bits, status, workspace bytes)."""
    import torch
    M, N, K = p["M"], p["N"], p["K"]
    keep = []
    addr = {}
    for name in ("A", "B", "bias", "scale", "R"):
        if p.get(name) is None:
            addr[name] = None
            continue
        buf, a = placed(p[name], offs.get(name, 0))
        keep.append(buf)
        addr[name] = a
    c_off = offs.get("C", 0)
    cbuf = torch.full((M * ldc + c_off + 8,), SENTINEL, dtype=torch.int16, device="cuda")
    c_addr = cbuf.data_ptr() + 2 * c_off
    epi = tg.make_epilogue(addr["bias"], addr["scale"], bool(p.get("relu", False)), addr["R"],
                           p.get("ldr", 0) or 0)
    args = (M, N, K, addr["A"], p["lda"], p["permA"], addr["B"], p["ldb"], p["permB"], c_addr,
            ldc, p["dtype"], epi)
    need = tg.tg_gemm_workspace_size_ex(*args)
    if use_ws:
        ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
        rc = tg.tg_gemm_ws(*args, ws, need - ws_shrink)
    else:
        rc = tg.tg_gemm(*args)
    torch.cuda.synchronize()
    c = host_bits(cbuf)[c_off:c_off + M * ldc].reshape(M, ldc)
    return c, rc, need


CASES = [
    # (M, N, K, permA, permB, lda, ldb, ldc, offsets, epilogue)
    (200, 130, 100, 0, 0, 101, 133, 131, dict(A=1, B=3, C=5), {}),
    (333, 517, 1111, 0, 0, 1111, 517, 519, dict(A=0, B=2, C=0), {}),        # odd ld only
    (256, 256, 256, 1, 1, 259, 257, 256, dict(A=7, B=0, C=1), {}),           # permutes, C offset
    (300, 260, 400, 0, 1, 403, 405, 261,
     dict(A=2, B=1, C=3, R=5, bias=1, scale=3), dict(bias=True, scale=True, residual=True, relu=True)),
    (640, 768, 520, 0, 0, 520, 768, 768, dict(R=1), dict(residual=True)),    # only R staged
    (1000, 520, 1200, 0, 0, 1203, 520, 520, dict(A=1), {}),                 # staged A only
]


@pytest.mark.parametrize("M,N,K,pa,pb,lda,ldb,ldc,offs,epi", CASES)
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_unaligned_operands_match_the_oracle(tg, M, N, K, pa, pb, lda, ldb, ldc, offs, epi, dtype):
    flags = dict(epi)
    relu = flags.pop("relu", False)
    if flags.get("residual"):
        flags["ldr"] = N + 3
    p = synthetic.gemm_problem(M, N, K, dtype, 77 + M + K, permA=pa, permB=pb, lda=lda, ldb=ldb,
                               **flags)
    p["relu"] = relu
    c, rc, need = run_unaligned(tg, p, offs, ldc)
    assert rc == tg.TG_OK, tg.tg_status_string(rc)
    assert need > 0
    st, code = tg.tg_debug_status()
    assert st == tg.TG_OK, hex(code)
    check_close(c, oracle.gemm(p), dtype, what=f"{M}x{N}x{K} offs={offs}")
    check_padding(c, N)


def test_unaligned_needs_a_workspace_and_enough_of_it(tg):
    p = synthetic.gemm_problem(200, 130, 100, F16, 5, lda=101, ldb=133)
    _, rc, _ = run_unaligned(tg, p, dict(A=1), 136, use_ws=False)
    assert rc == tg.TG_ERR_ALIGN  # tg_gemm keeps the 16-byte requirement
    _, rc, _ = run_unaligned(tg, p, dict(A=1), 136, ws_shrink=1)
    assert rc == tg.TG_ERR_BUFFER
    _, rc, _ = run_unaligned(tg, p, dict(A=1), 136)
    assert rc == tg.TG_OK


def test_aligned_arguments_need_no_staging(tg):
    import torch
    A = torch.empty((4096, 4096), dtype=torch.int16, device="cuda")
    C = torch.empty((4096, 4096), dtype=torch.int16, device="cuda")
    ex = tg.tg_gemm_workspace_size_ex(4096, 4096, 4096, A, 4096, 0, A, 4096, 0, C, 4096, F16)
    assert ex == tg.tg_gemm_workspace_size(4096, 4096, 4096, F16)


def test_odd_byte_pointer_rejected_even_with_workspace(tg):
    import torch
    A = torch.zeros(64 * 64 + 8, dtype=torch.int16, device="cuda")
    C = torch.zeros(64 * 64, dtype=torch.int16, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    rc = tg.tg_gemm_ws(64, 64, 64, A.data_ptr() + 1, 64, 0, A, 64, 0, C, 64, F16, None, ws,
                       ws.numel())
    assert rc == tg.TG_ERR_ALIGN
