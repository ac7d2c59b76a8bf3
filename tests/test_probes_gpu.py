"""Hardware pins of the layout module (bit-exact):

* the 128-byte swizzle a TMA copy writes into shared memory equals the
  (offset) -> (row, col) layout ``swizzle128`` and the oracle's definition;
* the accumulator readout of tcgen05.ld 32x32b equals the
  (register, lane, warp) -> (m, n) layout ``tmem_32x32b``.
"""
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
