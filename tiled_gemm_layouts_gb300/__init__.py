"""Python binding of libtilegemm (argument marshalling only).

Every computation runs in the C-ABI library ``libtilegemm.so`` built from
``csrc/`` (``python tiled_gemm_layouts_gb300/build.py``).  If the library is
missing this module raises on import: there is no Python or CPU fallback.

Names follow ``include/tilegemm.h``.  Pointers may be given as integers or as
objects with ``data_ptr()`` (e.g. torch tensors); streams as integers, objects
with ``cuda_stream``, or None (legacy default stream).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# TILEGEMM_LIBRARY selects another build of the same library (e.g. one built
# with different flags); the default is the in-tree build.
LIB_PATH = os.environ.get("TILEGEMM_LIBRARY") or os.path.join(_HERE, "libtilegemm.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libtilegemm.so not found at {LIB_PATH}; build it with "
        "`python tiled_gemm_layouts_gb300/build.py` (needs nvcc for sm_103a)")

_lib = ctypes.CDLL(LIB_PATH)

TG_OK = 0
TG_ERR_INVALID_ARG = 1
TG_ERR_STRIDE = 2
TG_ERR_ALIGN = 3
TG_ERR_OVERLAP = 4
TG_ERR_DTYPE = 5
TG_ERR_UNSUPPORTED_DEVICE = 6
TG_ERR_CUDA = 7
TG_ERR_TIMEOUT = 8
TG_ERR_POINTER = 9
TG_ERR_LAYOUT = 10
TG_ERR_BUFFER = 11

TG_F16, TG_BF16 = 0, 1
TG_OP_N, TG_OP_T = 0, 1

_i64, _int, _vp, _cp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_char_p


class tg_epilogue(ctypes.Structure):
    _fields_ = [("bias_n", _vp), ("scale_m", _vp), ("relu", _int), ("residual", _vp),
                ("ldr", _i64)]


def _sig(name, res, *args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_sig("tg_gemm", _int, _i64, _i64, _i64, _vp, _i64, _int, _vp, _i64, _int, _vp, _i64, _int,
     ctypes.POINTER(tg_epilogue), _vp)
_sig("tg_status_string", _cp, _int)
_sig("tg_query_config", _int, _i64, _i64, _i64, _int, _int, _int, ctypes.POINTER(tg_epilogue),
     ctypes.c_char_p, ctypes.c_size_t)
_sig("tg_query_config_for_sms", _int, _int, _int, _i64, _i64, _i64, _int, _int, _int,
     ctypes.POINTER(tg_epilogue), ctypes.c_char_p, ctypes.c_size_t)
_sig("tg_query_config_ws", _int, _i64, _i64, _i64, _int, _int, _int, ctypes.POINTER(tg_epilogue),
     ctypes.c_char_p, ctypes.c_size_t)
_sig("tg_gemm_ws", _int, _i64, _i64, _i64, _vp, _i64, _int, _vp, _i64, _int, _vp, _i64, _int,
     ctypes.POINTER(tg_epilogue), _vp, ctypes.c_size_t, _vp)
_sig("tg_gemm_workspace_size", _int, _i64, _i64, _i64, _int, _int, _int,
     ctypes.POINTER(tg_epilogue), ctypes.POINTER(ctypes.c_size_t))
_sig("tg_pointwise", _int, _i64, _i64, _vp, _i64, _int, _vp, _i64, _int,
     ctypes.POINTER(tg_epilogue), _vp)
_sig("tg_gemm_workspace_size_ex", _int, _i64, _i64, _i64, _vp, _i64, _int, _vp, _i64, _int, _vp,
     _i64, _int, ctypes.POINTER(tg_epilogue), ctypes.POINTER(ctypes.c_size_t))
_sig("tg_gemm_static_ws", _int, _i64, _i64, _i64, _vp, _i64, _int, _vp, _i64, _int, _vp, _i64,
     _int, ctypes.POINTER(tg_epilogue), _vp)
_sig("tg_gemm_host", _int, _i64, _i64, _i64, _vp, _i64, _int, _vp, _i64, _int, _vp, _i64, _int,
     ctypes.POINTER(tg_epilogue), _vp, ctypes.c_size_t, _vp)
_sig("tg_gemm_host_workspace_size", _int, _i64, _i64, _i64, _int, _int, _int,
     ctypes.POINTER(tg_epilogue), ctypes.POINTER(ctypes.c_size_t))
_sig("tg_debug_status", _int, ctypes.POINTER(_int))
_sig("tg_debug_configure", _int, _i64, _i64)
_sig("tg_probe_swizzle128", _int, _vp, _int, _i64, _vp, _vp, _vp)
_sig("tg_probe_tmem_32x32b", _int, _int, _vp, _vp, _vp)

_PP = ctypes.POINTER(ctypes.c_void_p)
_sig("tg_layout_create", _int, _int, ctypes.POINTER(_cp), ctypes.POINTER(_int), _int,
     ctypes.POINTER(_cp), ctypes.POINTER(_int), ctypes.POINTER(ctypes.c_int32), _PP)
_sig("tg_layout_destroy", None, _vp)
_sig("tg_layout_num_dims", _int, _vp, ctypes.POINTER(_int), ctypes.POINTER(_int))
_sig("tg_layout_in_dim", _int, _vp, _int, ctypes.c_char_p, ctypes.c_size_t, ctypes.POINTER(_int))
_sig("tg_layout_out_dim", _int, _vp, _int, ctypes.c_char_p, ctypes.c_size_t, ctypes.POINTER(_int))
_sig("tg_layout_get_bases", _int, _vp, ctypes.POINTER(ctypes.c_int32), ctypes.c_size_t)
_sig("tg_layout_apply", _int, _vp, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32))
_sig("tg_layout_compose", _int, _vp, _vp, _PP)
_sig("tg_layout_product", _int, _vp, _vp, _PP)
_sig("tg_layout_sublayout", _int, _vp, _int, ctypes.POINTER(_cp), _int, ctypes.POINTER(_cp), _PP)
_sig("tg_layout_transpose_outs", _int, _vp, _int, ctypes.POINTER(_cp), _PP)
_sig("tg_layout_transpose_ins", _int, _vp, _int, ctypes.POINTER(_cp), _PP)
_sig("tg_layout_reshape_ins", _int, _vp, _int, ctypes.POINTER(_cp), ctypes.POINTER(_int), _PP)
_sig("tg_layout_reshape_outs", _int, _vp, _int, ctypes.POINTER(_cp), ctypes.POINTER(_int), _PP)
_sig("tg_layout_divide_left", _int, _vp, _vp, _PP)
_sig("tg_layout_divide_right", _int, _vp, _vp, _PP)
_sig("tg_layout_rank", _int, _vp, ctypes.POINTER(_int))
_sig("tg_layout_is_injective", _int, _vp, ctypes.POINTER(_int))
_sig("tg_layout_is_surjective", _int, _vp, ctypes.POINTER(_int))
_sig("tg_layout_invert_and_compose", _int, _vp, _vp, _PP)
_I2 = ctypes.c_int * 2
_sig("tg_layout_blocked", _int, _I2, _I2, _I2, _I2, _I2, _PP)
_IP = ctypes.POINTER(_int)
_sig("tg_layout_blocked_nd", _int, _int, _IP, _IP, _IP, _IP, _IP, _PP)
_sig("tg_layout_cooperative", _int, _I2, _int, _I2, _PP)


class tg_folded_layout(ctypes.Structure):
    """include/tilegemm_layout_device.h: a layout folded for kernel evaluation."""
    _fields_ = [("n_vars", _int), ("var_bits", _int * 8), ("n_bits", _int),
                ("cols", ctypes.c_uint32 * 32), ("constant", ctypes.c_uint32), ("n_outs", _int),
                ("out_shift", _int * 8), ("out_bits", _int * 8)]


_sig("tg_layout_fold", _int, _vp, _int, ctypes.POINTER(_cp), ctypes.POINTER(ctypes.c_int32),
     ctypes.POINTER(tg_folded_layout))
_sig("tg_layout_folded_apply", _int, ctypes.POINTER(tg_folded_layout),
     ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32))
_sig("tg_probe_folded_layout", _int, ctypes.POINTER(tg_folded_layout), _vp, ctypes.c_size_t, _vp)
_sig("tg_layout_register_tile", _int, _I2, _I2, _PP)
_sig("tg_layout_swizzle128", _int, _int, _int, _PP)
_sig("tg_layout_tmem_32x32b", _int, _int, _PP)

EXPORTED = [
    "tg_gemm", "tg_gemm_ws", "tg_gemm_workspace_size", "tg_gemm_workspace_size_ex",
    "tg_pointwise",
    "tg_gemm_static_ws", "tg_gemm_host", "tg_gemm_host_workspace_size",
    "tg_status_string", "tg_query_config",
    "tg_query_config_ws", "tg_query_config_for_sms",
    "tg_debug_status", "tg_debug_configure",
    "tg_probe_swizzle128", "tg_probe_tmem_32x32b", "tg_probe_folded_layout",
    "tg_layout_create", "tg_layout_destroy",
    "tg_layout_num_dims", "tg_layout_in_dim", "tg_layout_out_dim", "tg_layout_get_bases",
    "tg_layout_apply", "tg_layout_compose", "tg_layout_product", "tg_layout_sublayout",
    "tg_layout_transpose_outs", "tg_layout_transpose_ins", "tg_layout_reshape_ins",
    "tg_layout_reshape_outs", "tg_layout_divide_left", "tg_layout_divide_right",
    "tg_layout_rank", "tg_layout_is_injective",
    "tg_layout_is_surjective", "tg_layout_invert_and_compose", "tg_layout_blocked",
    "tg_layout_blocked_nd", "tg_layout_fold", "tg_layout_folded_apply",
    "tg_layout_cooperative", "tg_layout_register_tile", "tg_layout_swizzle128",
    "tg_layout_tmem_32x32b",
]


class TileGemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {tg_status_string(status)}" if what else tg_status_string(status))


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def tg_status_string(status: int) -> str:
    return _lib.tg_status_string(status).decode()


def make_epilogue(bias_n=None, scale_m=None, relu=False, residual=None, ldr=0):
    """A tg_epilogue, or None when every field is neutral."""
    if bias_n is None and scale_m is None and not relu and residual is None:
        return None
    return tg_epilogue(_addr(bias_n), _addr(scale_m), int(relu), _addr(residual), int(ldr))


def tg_gemm(M, N, K, A, lda, permA, B, ldb, permB, C, ldc, dtype, epi=None, stream=None) -> int:
    """Status of one tg_gemm call (see include/tilegemm.h); never raises."""
    return _lib.tg_gemm(M, N, K, _addr(A), lda, permA, _addr(B), ldb, permB, _addr(C), ldc, dtype,
                        ctypes.byref(epi) if epi is not None else None, _stream(stream))


def gemm(M, N, K, A, lda, permA, B, ldb, permB, C, ldc, dtype, epi=None, stream=None) -> None:
    """tg_gemm that raises TileGemmError on a nonzero status."""
    rc = tg_gemm(M, N, K, A, lda, permA, B, ldb, permB, C, ldc, dtype, epi, stream)
    if rc != TG_OK:
        raise TileGemmError(rc, "tg_gemm")


def tg_gemm_ws(M, N, K, A, lda, permA, B, ldb, permB, C, ldc, dtype, epi, workspace,
               workspace_bytes, stream=None) -> int:
    """Status of one tg_gemm_ws call; never raises."""
    return _lib.tg_gemm_ws(M, N, K, _addr(A), lda, permA, _addr(B), ldb, permB, _addr(C), ldc,
                           dtype, ctypes.byref(epi) if epi is not None else None,
                           _addr(workspace), workspace_bytes, _stream(stream))


def gemm_ws(M, N, K, A, lda, permA, B, ldb, permB, C, ldc, dtype, epi, workspace,
            workspace_bytes, stream=None) -> None:
    rc = tg_gemm_ws(M, N, K, A, lda, permA, B, ldb, permB, C, ldc, dtype, epi, workspace,
                    workspace_bytes, stream)
    if rc != TG_OK:
        raise TileGemmError(rc, "tg_gemm_ws")


def tg_gemm_static_ws(M, N, K, A, lda, permA, B, ldb, permB, C, ldc, dtype, epi=None,
                      stream=None) -> int:
    """Status of one tg_gemm_static_ws call (library-owned static scratch; for
    callers that cannot allocate device memory); never raises."""
    return _lib.tg_gemm_static_ws(M, N, K, _addr(A), lda, permA, _addr(B), ldb, permB, _addr(C),
                                  ldc, dtype, ctypes.byref(epi) if epi is not None else None,
                                  _stream(stream))


def tg_gemm_workspace_size(M, N, K, dtype, permA=TG_OP_N, permB=TG_OP_N, epi=None) -> int:
    n = ctypes.c_size_t(0)
    rc = _lib.tg_gemm_workspace_size(M, N, K, dtype, permA, permB,
                                     ctypes.byref(epi) if epi is not None else None,
                                     ctypes.byref(n))
    if rc != TG_OK:
        raise TileGemmError(rc, "tg_gemm_workspace_size")
    return n.value


def tg_gemm_host(M, N, K, A, lda, permA, B, ldb, permB, C, ldc, dtype, epi, workspace,
                 workspace_bytes, stream=None) -> int:
    """Status of one tg_gemm_host call (A, B, C and the epilogue operands in
    page-locked host memory, `workspace` on the device); never raises."""
    return _lib.tg_gemm_host(M, N, K, _addr(A), lda, permA, _addr(B), ldb, permB, _addr(C), ldc,
                             dtype, ctypes.byref(epi) if epi is not None else None,
                             _addr(workspace), workspace_bytes, _stream(stream))


def gemm_host(M, N, K, A, lda, permA, B, ldb, permB, C, ldc, dtype, epi, workspace,
              workspace_bytes, stream=None) -> None:
    rc = tg_gemm_host(M, N, K, A, lda, permA, B, ldb, permB, C, ldc, dtype, epi, workspace,
                      workspace_bytes, stream)
    if rc != TG_OK:
        raise TileGemmError(rc, "tg_gemm_host")


def tg_gemm_host_workspace_size(M, N, K, dtype, permA=TG_OP_N, permB=TG_OP_N, epi=None) -> int:
    n = ctypes.c_size_t(0)
    rc = _lib.tg_gemm_host_workspace_size(M, N, K, dtype, permA, permB,
                                          ctypes.byref(epi) if epi is not None else None,
                                          ctypes.byref(n))
    if rc != TG_OK:
        raise TileGemmError(rc, "tg_gemm_host_workspace_size")
    return n.value


def tg_pointwise(M, N, X, ldx, permX, C, ldc, dtype, epi=None, stream=None) -> int:
    return _lib.tg_pointwise(M, N, _addr(X), ldx, permX, _addr(C), ldc, dtype,
                             ctypes.byref(epi) if epi is not None else None, _stream(stream))


def tg_gemm_workspace_size_ex(M, N, K, A, lda, permA, B, ldb, permB, C, ldc, dtype,
                              epi=None) -> int:
    n = ctypes.c_size_t(0)
    rc = _lib.tg_gemm_workspace_size_ex(M, N, K, _addr(A), lda, permA, _addr(B), ldb, permB,
                                        _addr(C), ldc, dtype,
                                        ctypes.byref(epi) if epi is not None else None,
                                        ctypes.byref(n))
    if rc != TG_OK:
        raise TileGemmError(rc, "tg_gemm_workspace_size_ex")
    return n.value


def tg_query_config_ws(M, N, K, dtype, permA=TG_OP_N, permB=TG_OP_N, epi=None) -> str:
    buf = ctypes.create_string_buffer(256)
    rc = _lib.tg_query_config_ws(M, N, K, dtype, permA, permB,
                                 ctypes.byref(epi) if epi is not None else None, buf, len(buf))
    if rc != TG_OK:
        raise TileGemmError(rc, "tg_query_config_ws")
    return buf.value.decode()


def tg_query_config(M, N, K, dtype, permA=TG_OP_N, permB=TG_OP_N, epi=None) -> str:
    buf = ctypes.create_string_buffer(256)
    rc = _lib.tg_query_config(M, N, K, dtype, permA, permB,
                              ctypes.byref(epi) if epi is not None else None, buf, len(buf))
    if rc != TG_OK:
        raise TileGemmError(rc, "tg_query_config")
    return buf.value.decode()


def tg_query_config_for_sms(sms, M, N, K, dtype, permA=TG_OP_N, permB=TG_OP_N, epi=None,
                            stream_k=False) -> str:
    buf = ctypes.create_string_buffer(256)
    rc = _lib.tg_query_config_for_sms(sms, int(stream_k), M, N, K, dtype, permA, permB,
                                      ctypes.byref(epi) if epi is not None else None, buf,
                                      len(buf))
    if rc != TG_OK:
        raise TileGemmError(rc, "tg_query_config_for_sms")
    return buf.value.decode()


def parse_config(s: str) -> dict:
    return {k: int(v) for k, v in (kv.split("=") for kv in s.split())}


def tg_debug_status() -> tuple[int, int]:
    """(status, raw device code); synchronises the device and clears the word."""
    d = _int(0)
    rc = _lib.tg_debug_status(ctypes.byref(d))
    return rc, d.value


def tg_debug_configure(timeout_cycles: int = 0, skip_kblock: int = -1) -> int:
    return _lib.tg_debug_configure(timeout_cycles, skip_kblock)


def tg_probe_swizzle128(src, rows, ld, dst, status_dev, stream=None) -> int:
    return _lib.tg_probe_swizzle128(_addr(src), rows, ld, _addr(dst), _addr(status_dev),
                                    _stream(stream))


def tg_probe_tmem_32x32b(bn, dst, status_dev, stream=None) -> int:
    return _lib.tg_probe_tmem_32x32b(bn, _addr(dst), _addr(status_dev), _stream(stream))


# ----------------------------------------------------------------- layouts

def _names(names):
    arr = (_cp * max(1, len(names)))(*[n.encode() for n in names])
    return arr


def _check(rc, what):
    if rc != TG_OK:
        raise TileGemmError(rc, what)


class LinearLayout:
    """Owning wrapper of a ``tg_layout`` handle (GF(2) linear layout)."""

    def __init__(self, handle: int):
        self._h = ctypes.c_void_p(handle)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            _lib.tg_layout_destroy(h)
            self._h = None

    @staticmethod
    def _new(fn, *args, what="layout"):
        out = ctypes.c_void_p()
        _check(fn(*args, ctypes.byref(out)), what)
        return LinearLayout(out.value)

    @classmethod
    def create(cls, in_dims, out_dims, bases):
        """in_dims/out_dims: [(name, log2 size)]; bases: {in name: [coords per bit]}."""
        rows = [tuple(v) for name, b in in_dims for v in bases.get(name, [])]
        nout = len(out_dims)
        flat = (ctypes.c_int32 * max(1, len(rows) * nout))(*[c for r in rows for c in r])
        ib = (_int * max(1, len(in_dims)))(*[b for _, b in in_dims])
        ob = (_int * max(1, len(out_dims)))(*[b for _, b in out_dims])
        return cls._new(_lib.tg_layout_create, len(in_dims), _names([n for n, _ in in_dims]), ib,
                        nout, _names([n for n, _ in out_dims]), ob, flat, what="tg_layout_create")

    # dims and bases
    def _dims(self, fn, n):
        out = []
        for i in range(n):
            buf = ctypes.create_string_buffer(32)
            bits = _int(0)
            _check(fn(self._h, i, buf, 32, ctypes.byref(bits)), "dim")
            out.append((buf.value.decode(), bits.value))
        return out

    @property
    def in_dims(self):
        ni, no = _int(0), _int(0)
        _lib.tg_layout_num_dims(self._h, ctypes.byref(ni), ctypes.byref(no))
        return self._dims(_lib.tg_layout_in_dim, ni.value)

    @property
    def out_dims(self):
        ni, no = _int(0), _int(0)
        _lib.tg_layout_num_dims(self._h, ctypes.byref(ni), ctypes.byref(no))
        return self._dims(_lib.tg_layout_out_dim, no.value)

    @property
    def bases(self) -> dict:
        ins, outs = self.in_dims, self.out_dims
        total = sum(b for _, b in ins)
        buf = (ctypes.c_int32 * max(1, total * len(outs)))()
        _check(_lib.tg_layout_get_bases(self._h, buf, total * len(outs)), "get_bases")
        rows = [tuple(buf[r * len(outs):(r + 1) * len(outs)]) for r in range(total)]
        out, r = {}, 0
        for name, b in ins:
            out[name] = rows[r:r + b]
            r += b
        return out

    def as_tuple(self):
        """(in_dims, out_dims, bases) -- the plain representation."""
        return self.in_dims, self.out_dims, self.bases

    def apply(self, ins: dict) -> tuple:
        names = [n for n, _ in self.in_dims]
        nout = len(self.out_dims)
        arr = (ctypes.c_int32 * max(1, len(names)))(*[ins[n] for n in names])
        out = (ctypes.c_int32 * max(1, nout))()
        _check(_lib.tg_layout_apply(self._h, arr, out), "apply")
        return tuple(out[:nout])

    def fold(self, fixed: dict) -> "FoldedLayout":
        """Folds the inputs in ``fixed`` (name -> value) for kernel evaluation;
        the other input dims stay variable, in the layout's order."""
        names = list(fixed)
        arr_n = (_cp * max(1, len(names)))(*[n.encode() for n in names])
        arr_v = (ctypes.c_int32 * max(1, len(names)))(*[int(fixed[n]) for n in names])
        f = tg_folded_layout()
        _check(_lib.tg_layout_fold(self._h, len(names), arr_n, arr_v, ctypes.byref(f)), "fold")
        var_names = [n for n, _ in self.in_dims if n not in fixed]
        return FoldedLayout(f, var_names, [n for n, _ in self.out_dims])

    def compose(self, outer: "LinearLayout") -> "LinearLayout":
        return self._new(_lib.tg_layout_compose, self._h, outer._h, what="compose")

    def __mul__(self, other: "LinearLayout") -> "LinearLayout":
        return self._new(_lib.tg_layout_product, self._h, other._h, what="product")

    def sublayout(self, in_names, out_names) -> "LinearLayout":
        return self._new(_lib.tg_layout_sublayout, self._h, len(in_names), _names(in_names),
                         len(out_names), _names(out_names), what="sublayout")

    def transpose_outs(self, out_names) -> "LinearLayout":
        return self._new(_lib.tg_layout_transpose_outs, self._h, len(out_names),
                         _names(out_names), what="transpose_outs")

    def transpose_ins(self, in_names) -> "LinearLayout":
        return self._new(_lib.tg_layout_transpose_ins, self._h, len(in_names),
                         _names(in_names), what="transpose_ins")

    def reshape_ins(self, in_dims) -> "LinearLayout":
        """in_dims: [(name, log2 size)] with the same total bits."""
        bits = (_int * max(1, len(in_dims)))(*[b for _, b in in_dims])
        return self._new(_lib.tg_layout_reshape_ins, self._h, len(in_dims),
                         _names([n for n, _ in in_dims]), bits, what="reshape_ins")

    def reshape_outs(self, out_dims) -> "LinearLayout":
        """out_dims: [(name, log2 size)] with the same total bits."""
        bits = (_int * max(1, len(out_dims)))(*[b for _, b in out_dims])
        return self._new(_lib.tg_layout_reshape_outs, self._h, len(out_dims),
                         _names([n for n, _ in out_dims]), bits, what="reshape_outs")

    def divide_left(self, B: "LinearLayout") -> "LinearLayout":
        """C with self = B * C."""
        return self._new(_lib.tg_layout_divide_left, self._h, B._h, what="divide_left")

    def divide_right(self, B: "LinearLayout") -> "LinearLayout":
        """C with self = C * B."""
        return self._new(_lib.tg_layout_divide_right, self._h, B._h, what="divide_right")

    def _int_query(self, fn):
        v = _int(0)
        _check(fn(self._h, ctypes.byref(v)), "query")
        return v.value

    @property
    def rank(self) -> int:
        return self._int_query(_lib.tg_layout_rank)

    @property
    def is_injective(self) -> bool:
        return bool(self._int_query(_lib.tg_layout_is_injective))

    @property
    def is_surjective(self) -> bool:
        return bool(self._int_query(_lib.tg_layout_is_surjective))

    def invert_and_compose(self, S: "LinearLayout") -> "LinearLayout":
        return self._new(_lib.tg_layout_invert_and_compose, self._h, S._h,
                         what="invert_and_compose")

    # constructors
    @classmethod
    def blocked(cls, size_per_thread, threads_per_warp, warps_per_cta, order, shape):
        return cls._new(_lib.tg_layout_blocked, _I2(*size_per_thread), _I2(*threads_per_warp),
                        _I2(*warps_per_cta), _I2(*order), _I2(*shape), what="blocked")

    @classmethod
    def blocked_nd(cls, size_per_thread, threads_per_warp, warps_per_cta, order, shape):
        """Blocked encoding of any rank (every argument has one entry per dim)."""
        rank = len(shape)
        if any(len(x) != rank for x in (size_per_thread, threads_per_warp, warps_per_cta, order)):
            raise TileGemmError(TG_ERR_INVALID_ARG, "blocked_nd")
        arrs = [(_int * rank)(*x) for x in (size_per_thread, threads_per_warp, warps_per_cta,
                                             order, shape)]
        return cls._new(_lib.tg_layout_blocked_nd, rank, *arrs, what="blocked_nd")

    @classmethod
    def cooperative(cls, shape, threads, order):
        return cls._new(_lib.tg_layout_cooperative, _I2(*shape), threads, _I2(*order),
                        what="cooperative")

    @classmethod
    def register_tile(cls, logical, thread_shape):
        return cls._new(_lib.tg_layout_register_tile, _I2(*logical), _I2(*thread_shape),
                        what="register_tile")

    @classmethod
    def swizzle128(cls, rows, elem_bytes=2):
        return cls._new(_lib.tg_layout_swizzle128, rows, elem_bytes, what="swizzle128")

    @classmethod
    def tmem_32x32b(cls, bn):
        return cls._new(_lib.tg_layout_tmem_32x32b, bn, what="tmem_32x32b")


class FoldedLayout:
    """A layout folded by tg_layout_fold: ``raw`` is the plain struct a kernel
    takes; ``apply`` evaluates it on the host with the kernel's functions."""

    def __init__(self, raw: tg_folded_layout, var_names: list, out_names: list):
        self.raw = raw
        self.var_names = var_names
        self.out_names = out_names

    def apply(self, vars: dict) -> tuple:
        arr = (ctypes.c_int32 * max(1, len(self.var_names)))(*[vars[n] for n in self.var_names])
        out = (ctypes.c_int32 * max(1, len(self.out_names)))()
        _check(_lib.tg_layout_folded_apply(ctypes.byref(self.raw), arr, out), "folded_apply")
        return tuple(out[:len(self.out_names)])
