"""The library inside CUDA graphs and under concurrent host threads.

* tg_gemm_ws (stream-K workspace, fused epilogue) captured once into a CUDA
  graph, then replayed after new inputs are written into the same buffers:
  every replay must match the oracle for the inputs of that replay.
* tg_gemm_host captured the same way: its copy streams and side stream fork
  from the capturing stream and join it again, so the whole pipeline (host
  copies, block GEMMs, copy-back) becomes one graph.
* tg_gemm_host called from two host threads at once, each with its own
  stream and workspace: the shared per-device copy streams and events must
  keep every call's results intact.
"""
import threading

import numpy as np
import pytest

import oracle
import synthetic
from synthetic import F16, BF16
from helpers import SENTINEL, check_close, dev, host_bits

pytestmark = pytest.mark.gpu


def test_gemm_ws_replayed_from_a_cuda_graph(tg):
    import torch
    M, N, K = 2560, 2504, 2304  # 100 tiles on 76 CTA pairs: a stream-K tail; ragged N
    p = synthetic.gemm_problem(M, N, K, F16, 71, bias=True, scale=True, residual=True)
    p["relu"] = True
    A, B = dev(p["A"]), dev(p["B"])
    bias, scale, R = dev(p["bias"]), dev(p["scale"]), dev(p["R"])
    epi = tg.make_epilogue(bias, scale, True, R, p["ldr"])
    need = tg.tg_gemm_workspace_size(M, N, K, F16, 0, 0, epi)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
    C = torch.full((M, N), SENTINEL, dtype=torch.int16, device="cuda")
    s = torch.cuda.Stream()
    call = lambda: tg.tg_gemm_ws(M, N, K, A, K, 0, B, N, 0, C, N, F16, epi, ws, need, s)
    with torch.cuda.stream(s):
        assert call() == tg.TG_OK  # first call outside the capture: one-time setup
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rc = call()
    assert rc == tg.TG_OK, tg.tg_status_string(rc)
    for seed in (72, 73):
        q = synthetic.gemm_problem(M, N, K, F16, seed, bias=True, scale=True, residual=True)
        q["relu"] = True
        for name, t in (("A", A), ("B", B), ("bias", bias), ("scale", scale), ("R", R)):
            t.copy_(dev(q[name]))
        C.fill_(SENTINEL)
        g.replay()
        torch.cuda.synchronize()
        got = host_bits(C)
        for r0, r1 in ((0, 3), (1279, 1283), (2557, 2560)):
            check_close(got, oracle.gemm(q, rows=(r0, r1)), F16, rows=slice(r0, r1),
                        what=f"graph replay seed {seed} rows {r0}..{r1}")
    st, code = tg.tg_debug_status()
    assert st == tg.TG_OK, hex(code)


def test_gemm_host_replayed_from_a_cuda_graph(tg):
    import torch
    M, N, K = 1100, 520, 640
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory()
    p = synthetic.gemm_problem(M, N, K, BF16, 81, bias=True)
    hA, hB, hbias = pin(p["A"]), pin(p["B"]), pin(p["bias"])
    hC = torch.full((M, N), SENTINEL, dtype=torch.int16).pin_memory()
    epi = tg.make_epilogue(hbias)
    need = tg.tg_gemm_host_workspace_size(M, N, K, BF16, 0, 0, epi)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    call = lambda: tg.tg_gemm_host(M, N, K, hA, K, 0, hB, N, 0, hC, N, BF16, epi, ws, need, s)
    with torch.cuda.stream(s):
        assert call() == tg.TG_OK
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rc = call()
    assert rc == tg.TG_OK, tg.tg_status_string(rc)
    for seed in (82, 83):
        q = synthetic.gemm_problem(M, N, K, BF16, seed, bias=True)
        hA.copy_(pin(q["A"]))
        hB.copy_(pin(q["B"]))
        hbias.copy_(pin(q["bias"]))
        hC.fill_(SENTINEL)
        g.replay()
        torch.cuda.synchronize()
        got = hC.numpy().view(np.uint16)
        check_close(got, oracle.gemm(q), BF16, what=f"host graph replay seed {seed}")


def test_gemm_host_from_two_threads(tg):
    import torch
    results, errors = {}, []

    def worker(k):
        try:
            M, N, K = 700 + 64 * k, 300, 256
            pin = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory()
            s = torch.cuda.Stream()
            need = tg.tg_gemm_host_workspace_size(M, N, K, F16)
            ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
            out = []
            for it in range(3):
                p = synthetic.gemm_problem(M, N, K, F16, 900 + 10 * k + it)
                hA, hB = pin(p["A"]), pin(p["B"])
                hC = torch.empty((M, N), dtype=torch.int16).pin_memory()
                rc = tg.tg_gemm_host(M, N, K, hA, K, 0, hB, N, 0, hC, N, F16, None, ws, need, s)
                s.synchronize()
                out.append((rc, p, hC.numpy().view(np.uint16).copy()))
            results[k] = out
        except Exception as e:  # reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for k, out in results.items():
        for rc, p, c in out:
            assert rc == tg.TG_OK
            check_close(c, oracle.gemm(p), F16, what=f"thread {k}")
