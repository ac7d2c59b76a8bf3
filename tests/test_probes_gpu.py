"""Hardware pins of the layout module (bit-exact):

* the 128-byte swizzle a TMA copy writes into shared memory equals the
  (offset) -> (row, col) layout ``swizzle128`` and the oracle's definition;
* the accumulator readout of tcgen05.ld 32x32b equals the
  (register, lane, warp) -> (m, n) layout ``tmem_32x32b``;
* a layout folded for kernels (tilegemm_layout_device.h) evaluates on the
  device to what the host module and the oracle give, for every variable
  input.
"""
import ctypes

import numpy as np
import pytest

from oracle import layout_oracle as lo

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows", [8, 64, 256])
def test_tma_swizzle128_matches_layout(tg, rows):
    import torch
    ld = 72  # row stride in elements (144 bytes): the tile is not contiguous in global memory
    # element value = its linear position row*64 + col (fits 16 bits)
    src = np.zeros((rows, ld), dtype=np.uint16)
    src[:, :64] = np.arange(rows * 64, dtype=np.uint32).reshape(rows, 64).astype(np.uint16)
    src_d = torch.from_numpy(src.view(np.int16)).cuda()
    dst = torch.zeros(rows * 64, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert tg.tg_probe_swizzle128(src_d, rows, ld, dst, status) == tg.TG_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    dump = dst.cpu().numpy().view(np.uint16).astype(np.int64)
    L = tg.LinearLayout.swizzle128(rows, 2)
    for off in range(rows * 64):
        r, c = L.apply({"offset": off})
        assert dump[off] == r * 64 + c, off
        assert lo.swizzle128_offset(r, c, 2) == 2 * off


@pytest.mark.parametrize("bn", [64, 128, 256])
def test_tmem_readout_matches_layout(tg, bn):
    import torch
    dst = torch.zeros(128 * bn, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert tg.tg_probe_tmem_32x32b(bn, dst, status) == tg.TG_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    vals = dst.cpu().numpy().view(np.float32).reshape(4, 32, bn)
    L = tg.LinearLayout.tmem_32x32b(bn)
    for w in range(4):
        for t in range(32):
            for j in range(bn):
                v = vals[w, t, j]
                m, n = divmod(int(v), 256)
                assert v == 256 * m + n
                assert (m, n) == L.apply({"register": j, "lane": t, "warp": w})
                assert (m, n) == lo.tmem_32x32b_coordinate(w, t, j)


def test_folded_layout_on_the_device(tg):
    import torch
    from test_layout_module import folded_cases
    for L, fixed in folded_cases(tg):
        F = L.fold(fixed)
        r = F.raw
        n = 1 << r.n_bits
        dst = torch.full((n * r.n_outs,), -1, dtype=torch.int32, device="cuda")
        assert tg._lib.tg_probe_folded_layout(ctypes.byref(r), dst.data_ptr(), dst.numel() * 4,
                                              None) == tg.TG_OK
        torch.cuda.synchronize()
        got = dst.cpu().numpy().reshape(n, r.n_outs)
        T = L.as_tuple()
        for c in range(n):
            x, shift = dict(fixed), 0
            for name, b in zip(F.var_names, r.var_bits[:r.n_vars]):
                x[name] = (c >> shift) & ((1 << b) - 1)
                shift += b
            assert tuple(int(v) for v in got[c]) == lo.apply(T, x), (fixed, x)
    # a buffer one element short is refused before any launch
    F = folded_cases(tg)[3][0].fold({"register": 3})
    short = torch.zeros(((1 << F.raw.n_bits) * F.raw.n_outs - 1,), dtype=torch.int32, device="cuda")
    assert tg._lib.tg_probe_folded_layout(ctypes.byref(F.raw), short.data_ptr(), short.numel() * 4,
                                          None) == tg.TG_ERR_BUFFER
