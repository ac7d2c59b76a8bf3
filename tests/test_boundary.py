"""The C-ABI boundary without a GPU: every symbol the headers declare is
exported, and every argument check fires before any device work (so fake,
never-dereferenced pointers are enough)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

FAKE = 1 << 40          # 16-byte aligned, never dereferenced by the checks
F16, BF16 = 0, 1
N_, T_ = 0, 1


def declared_symbols():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            # header-only inline helpers (for kernels) are not library symbols
            inline = set(re.findall(r"TG_LAYOUT_FN\s+\w+\s+(tg_\w+)\s*\(", src))
            names |= set(re.findall(r"\b(tg_\w+)\s*\(", src)) - inline
    return names


def test_every_declared_symbol_is_exported(tg):
    lib = ctypes.CDLL(tg.LIB_PATH)
    decl = declared_symbols()
    assert len(decl) >= 27
    for name in sorted(decl):
        assert hasattr(lib, name), name
    assert decl <= set(tg.EXPORTED)


def test_status_strings(tg):
    assert tg.tg_status_string(0) == "TG_OK"
    assert tg.tg_status_string(tg.TG_ERR_OVERLAP) == "TG_ERR_OVERLAP"
    assert tg.tg_status_string(999) == "TG_ERR_UNKNOWN"


def call(tg, M=256, N=256, K=256, A=FAKE, lda=None, pa=N_, B=FAKE + (1 << 30), ldb=None, pb=N_,
         C=FAKE + (2 << 30), ldc=None, dtype=F16, epi=None):
    lda = (K if pa == N_ else M) if lda is None else lda
    ldb = (N if pb == N_ else K) if ldb is None else ldb
    ldc = N if ldc is None else ldc
    return tg.tg_gemm(M, N, K, A, lda, pa, B, ldb, pb, C, ldc, dtype, epi)


def test_valid_arguments_reach_device_check(tg):
    import torch
    if torch.cuda.is_available():
        pytest.skip("device present: covered by the GPU tests")
    assert call(tg) == tg.TG_ERR_UNSUPPORTED_DEVICE


@pytest.mark.parametrize("kw,code", [
    (dict(M=0), "TG_ERR_INVALID_ARG"),
    (dict(N=-3), "TG_ERR_INVALID_ARG"),
    (dict(K=0), "TG_ERR_INVALID_ARG"),
    (dict(M=1 << 31), "TG_ERR_INVALID_ARG"),
    (dict(A=0), "TG_ERR_INVALID_ARG"),
    (dict(B=0), "TG_ERR_INVALID_ARG"),
    (dict(C=0), "TG_ERR_INVALID_ARG"),
    (dict(pa=2), "TG_ERR_INVALID_ARG"),
    (dict(pb=-1), "TG_ERR_INVALID_ARG"),
    (dict(dtype=2), "TG_ERR_DTYPE"),
    (dict(lda=255), "TG_ERR_STRIDE"),                  # lda < K
    (dict(pa=T_, M=300, lda=296), "TG_ERR_STRIDE"),     # permuted A: lda < M
    (dict(ldb=0), "TG_ERR_STRIDE"),
    (dict(pb=T_, K=512, ldb=504), "TG_ERR_STRIDE"),     # permuted B: ldb < K
    (dict(ldc=248), "TG_ERR_STRIDE"),                   # ldc < N: rows would overlap
    (dict(A=FAKE + 2), "TG_ERR_ALIGN"),                 # tg_gemm: 16-byte bases only
    (dict(B=FAKE + (1 << 30) + 1), "TG_ERR_ALIGN"),     # an odd byte address: never valid
    (dict(C=FAKE + (2 << 30) + 8), "TG_ERR_ALIGN"),
    (dict(lda=260), "TG_ERR_ALIGN"),                    # 520-byte rows
    (dict(K=250, lda=250), "TG_ERR_ALIGN"),
    (dict(C=FAKE + 64), "TG_ERR_OVERLAP"),              # C inside A
    (dict(B=FAKE + (2 << 30) + 256 * 256 * 2 - 16), "TG_ERR_OVERLAP"),  # B starts in C's last row
])
def test_argument_checks(tg, kw, code):
    assert tg.tg_status_string(call(tg, **kw)) == code


def test_adjacent_buffers_do_not_overlap(tg):
    import torch
    if torch.cuda.is_available():
        pytest.skip("device present")
    # B starts exactly where C's last byte ends
    C = FAKE + (2 << 30)
    assert call(tg, C=C, B=C + 256 * 256 * 2) == tg.TG_ERR_UNSUPPORTED_DEVICE


def test_epilogue_checks(tg):
    C = FAKE + (2 << 30)
    e = tg.make_epilogue(relu=2)
    assert call(tg, epi=e) == tg.TG_ERR_INVALID_ARG
    e = tg.make_epilogue(bias_n=FAKE + (3 << 30) + 2)
    assert call(tg, epi=e) == tg.TG_ERR_ALIGN
    e = tg.make_epilogue(residual=C + 512)                     # residual aliases C
    assert call(tg, epi=e) == tg.TG_ERR_OVERLAP
    e = tg.make_epilogue(residual=FAKE + (3 << 30), ldr=100)   # ldr < N
    assert call(tg, epi=e) == tg.TG_ERR_STRIDE
    e = tg.make_epilogue(scale_m=C + 256 * 256 * 2 - 32)       # scale inside C
    assert call(tg, epi=e) == tg.TG_ERR_OVERLAP


def test_query_config_checks_shape_first(tg):
    with pytest.raises(tg.TileGemmError) as e:
        tg.tg_query_config(0, 16, 16, F16)
    assert e.value.status == tg.TG_ERR_INVALID_ARG
    with pytest.raises(tg.TileGemmError) as e:
        tg.tg_query_config(16, 16, 16, 3)
    assert e.value.status == tg.TG_ERR_DTYPE


def test_debug_configure_checks(tg):
    assert tg.tg_debug_configure(-1, -1) == tg.TG_ERR_INVALID_ARG
    assert tg.tg_debug_configure(0, -2) == tg.TG_ERR_INVALID_ARG
    assert tg.tg_debug_configure(0, -1) == tg.TG_OK


def test_package_fails_loudly_without_library(tmp_path):
    import shutil
    import subprocess
    import sys
    pkg = tmp_path / "tiled_gemm_layouts_gb300"
    pkg.mkdir()
    shutil.copy(os.path.join(ROOT, "tiled_gemm_layouts_gb300", "__init__.py"), pkg / "__init__.py")
    r = subprocess.run([sys.executable, "-c", "import tiled_gemm_layouts_gb300"], cwd=tmp_path,
                       capture_output=True, text=True)
    assert r.returncode != 0 and "libtilegemm.so not found" in r.stderr


def test_workspace_call_accepts_unaligned_operands_before_the_device_check(tg):
    import torch
    if torch.cuda.is_available():
        pytest.skip("device present: covered by tests/test_unaligned_gpu.py")
    ws = FAKE + (3 << 30)
    rc = tg.tg_gemm_ws(256, 256, 250, FAKE + 2, 250, N_, FAKE + (1 << 30), 256, N_,
                       FAKE + (2 << 30) + 6, 257, F16, None, ws, 1 << 24)
    assert rc == tg.TG_ERR_UNSUPPORTED_DEVICE  # the arguments passed every check
    rc = tg.tg_gemm(256, 256, 250, FAKE + 2, 250, N_, FAKE + (1 << 30), 256, N_,
                    FAKE + (2 << 30) + 6, 257, F16, None)
    assert rc == tg.TG_ERR_ALIGN


def test_host_pipeline_checks_shape_before_the_device(tg):
    # tg_gemm_host: sizes, null pointers, enums and dtype are refused before
    # any device query; valid arguments reach the device check
    A, B, C, W = FAKE, FAKE + (1 << 30), FAKE + (2 << 30), FAKE + (3 << 30)
    host = lambda M=256, N=256, K=256, pa=0, pb=0, dt=F16, w=W, epi=None: tg.tg_gemm_host(
        M, N, K, A, K, pa, B, N, pb, C, N, dt, epi, w, 1 << 30)
    assert host(M=0) == tg.TG_ERR_INVALID_ARG
    assert host(K=1 << 31) == tg.TG_ERR_INVALID_ARG
    assert host(w=None) == tg.TG_ERR_INVALID_ARG
    assert host(pa=2) == tg.TG_ERR_INVALID_ARG
    assert host(dt=7) == tg.TG_ERR_DTYPE
    assert host(epi=tg.make_epilogue(relu=3)) == tg.TG_ERR_INVALID_ARG
    assert host() == tg.TG_ERR_UNSUPPORTED_DEVICE
    n = ctypes.c_size_t(0)
    assert tg._lib.tg_gemm_host_workspace_size(256, 256, 256, F16, 0, 0, None, None) == \
        tg.TG_ERR_INVALID_ARG
    assert tg._lib.tg_gemm_host_workspace_size(0, 256, 256, F16, 0, 0, None, ctypes.byref(n)) == \
        tg.TG_ERR_INVALID_ARG
    assert tg._lib.tg_gemm_host_workspace_size(256, 256, 256, F16, 0, 0, None, ctypes.byref(n)) == \
        tg.TG_ERR_UNSUPPORTED_DEVICE
