"""Pins for the layout oracle (no GPU): the pages' printed worked examples and
the algebraic facts a GF(2)-linear map must satisfy, checked by enumeration."""
import itertools
import math

import numpy as np
import pytest

from oracle import layout_oracle as lo
from conftest import load_golden


def golden_layout(g):
    return ([tuple(d) for d in g["in_dims"]], [tuple(d) for d in g["out_dims"]],
            {k: [tuple(v) for v in vs] for k, vs in g["bases"].items()})


def test_lane_warp_example_printed_values():
    g = load_golden("linear_layout_lane_warp.json")
    L = golden_layout(g)
    for ev in g["evaluations"]:
        assert lo.apply(L, ev["in"]) == tuple(ev["out"])
    # closed form stated on the page: (lane, lane XOR warp)
    for x in lo.all_inputs(L):
        assert lo.apply(L, x) == (x["lane"], x["lane"] ^ x["warp"])


def test_blocked_example_printed_values():
    g = load_golden("blocked_32x32.json")
    spt, tpw, wpc, order, shape = (g[k] for k in ("size_per_thread", "threads_per_warp",
                                                  "warps_per_cta", "order", "shape"))
    # the integer ownership formula reproduces the printed bases ...
    for i, b in enumerate(g["bases"]["register"]):
        assert lo.blocked_coordinate(spt, tpw, wpc, order, shape, 1 << i, 0, 0) == tuple(b)
    for i, b in enumerate(g["bases"]["lane"]):
        assert lo.blocked_coordinate(spt, tpw, wpc, order, shape, 0, 1 << i, 0) == tuple(b)
    for i, b in enumerate(g["bases"]["warp"]):
        assert lo.blocked_coordinate(spt, tpw, wpc, order, shape, 0, 0, 1 << i) == tuple(b)
    # ... the printed evaluation, and full coverage
    ev = g["evaluations"][0]["in"]
    assert lo.blocked_coordinate(spt, tpw, wpc, order, shape, ev["register"], ev["lane"],
                                 ev["warp"]) == tuple(g["evaluations"][0]["out"])
    seen = {lo.blocked_coordinate(spt, tpw, wpc, order, shape, r, l, w)
            for r in range(8) for l in range(32) for w in range(4)}
    assert len(seen) == g["coverage"] == 32 * 32
    # and the printed bases, applied as a GF(2) map, agree with the integer formula
    L = ([("register", 3), ("lane", 5), ("warp", 2)], [("dim0", 5), ("dim1", 5)],
         {k: [tuple(v) for v in vs] for k, vs in g["bases"].items()})
    for x in lo.all_inputs(L):
        assert lo.apply(L, x) == lo.blocked_coordinate(spt, tpw, wpc, order, shape,
                                                       x["register"], x["lane"], x["warp"])
    assert lo.is_injective(L) and lo.is_surjective(L)


def test_cooperative_examples():
    g = load_golden("cooperative_tiles.json")
    for case in g["cases"]:
        shape = tuple(case["shape"])
        assert lo.cooperative_iterations(shape, g["threads"]) == case["iterations"]
        for v in case["visits"]:
            got = [lo.cooperative_coordinate(shape, g["threads"], tuple(g["order"]), v["thread"], it)
                   for it in range(case["iterations"])]
            assert got == [tuple(c) for c in v["coords"]]
        # every element exactly once
        cover = [lo.cooperative_coordinate(shape, g["threads"], tuple(g["order"]), t, it)
                 for t in range(g["threads"]) for it in range(case["iterations"])]
        assert sorted(cover) == sorted(itertools.product(*map(range, shape)))


def test_cooperative_tail_lanes():
    # 48 elements over 32 threads: second iteration has 16 active lanes
    act = [lo.cooperative_coordinate((3, 16), 32, (1, 0), t, 1) is not None for t in range(32)]
    assert sum(act) == 16 and all(act[:16]) and not any(act[16:])


def test_register_tile_examples():
    g = load_golden("register_tiles.json")
    for case in g["cases"]:
        lg, ts = tuple(case["logical"]), tuple(case["thread_shape"])
        assert lo.register_shape(lg, ts) == tuple(case["register_shape"])
        assert math.prod(lo.register_shape(lg, ts)) == case["registers_per_thread"]
        for own in case["owns"]:
            assert lo.register_tile_coordinate(lg, ts, tuple(case["thread"]),
                                               tuple(own["register"])) == tuple(own["logical"])
        # exact cover
        rs = lo.register_shape(lg, ts)
        cover = [lo.register_tile_coordinate(lg, ts, th, r)
                 for th in itertools.product(*map(range, ts))
                 for r in itertools.product(*map(range, rs))]
        assert sorted(cover) == sorted(itertools.product(*map(range, lg)))


def test_thread_prologue_row_major():
    # Part 12: for a (4, 8) thread shape, tile_i = t / 8, tile_j = t % 8
    assert lo.thread_coordinate(11, (4, 8)) == (1, 3)
    assert lo.thread_coordinate(31, (4, 8)) == (3, 7)


def _random_layout(rng, in_bits, out_bits, zero_prob=0.15):
    ins = [(f"i{j}", b) for j, b in enumerate(in_bits)]
    outs = [(f"o{j}", b) for j, b in enumerate(out_bits)]
    bases = {}
    for name, b in ins:
        vs = []
        for _ in range(b):
            if rng.random() < zero_prob:
                vs.append(tuple(0 for _ in outs))
            else:
                vs.append(tuple(int(rng.integers(0, 1 << ob)) for _, ob in outs))
        bases[name] = vs
    return ins, outs, bases


@pytest.mark.parametrize("seed", range(20))
def test_linearity_and_zero(seed):
    rng = np.random.default_rng(seed)
    L = _random_layout(rng, [int(rng.integers(0, 4)) for _ in range(2)], [3, 2])
    xs = list(lo.all_inputs(L))
    zero = {n: 0 for n, _ in L[0]}
    assert lo.apply(L, zero) == (0, 0)
    for x in xs[:16]:
        for y in xs[:16]:
            xy = {n: x[n] ^ y[n] for n in x}
            assert lo.apply(L, xy) == tuple(a ^ b for a, b in zip(lo.apply(L, x), lo.apply(L, y)))


def test_zero_basis_broadcasts():
    L = ([("lane", 2), ("warp", 1)], [("x", 2)], {"lane": [(1,), (2,)], "warp": [(0,)]})
    for lane in range(4):
        assert lo.apply(L, {"lane": lane, "warp": 0}) == lo.apply(L, {"lane": lane, "warp": 1})
    assert not lo.is_injective(L) and lo.is_surjective(L)
    assert lo.rank_by_enumeration(L) == 2


def test_swizzle128_definition_properties():
    # each 8-row atom is a permutation of its 1024 bytes; chunk 0 of row r moves to chunk r%8
    offs = {lo.swizzle128_offset(r, c, 2) for r in range(8) for c in range(64)}
    assert offs == set(range(0, 1024, 2))
    for r in range(16):
        assert lo.swizzle128_offset(r, 0, 2) == r * 128 + (r % 8) * 16
        assert lo.swizzle128_offset(r, 8 * (r % 8), 2) == r * 128  # chunk r%8 lands at 0
    # the XOR is bit-linear: offset(r, c) ^ offset(r', c') = offset(r^r', c^c') (r, c within a power-of-two box)
    for r, c, r2, c2 in [(3, 5, 6, 17), (7, 63, 1, 1), (12, 40, 5, 9)]:
        assert lo.swizzle128_offset(r, c, 2) ^ lo.swizzle128_offset(r2, c2, 2) == \
            lo.swizzle128_offset(r ^ r2, c ^ c2, 2)


def test_tmem_32x32b_definition():
    # warps 4..7 cover the same lane quadrants as warps 0..3
    assert lo.tmem_32x32b_coordinate(6, 5, 7) == (69, 7)
    assert lo.tmem_32x32b_coordinate(2, 5, 7, 32) == (69, 39)
    rows = {lo.tmem_32x32b_coordinate(w, t, 0)[0] for w in range(4) for t in range(32)}
    assert rows == set(range(128))


def test_blocked_rank3_with_a_unit_dim_reproduces_the_printed_example():
    # the rank-generic owner rule, pinned to the page's rank-2 example: a
    # leading dim of size 1 changes no coordinate of the other two
    g = load_golden("blocked_32x32.json")
    spt, tpw, wpc, order, shape = (g["size_per_thread"], g["threads_per_warp"],
                                   g["warps_per_cta"], g["order"], g["shape"])
    for r in range(8):
        for l in range(32):
            for w in range(4):
                c2 = lo.blocked_coordinate(spt, tpw, wpc, order, shape, r, l, w)
                c3 = lo.blocked_coordinate([1] + spt, [1] + tpw, [1] + wpc,
                                           [o + 1 for o in order] + [0], [1] + shape, r, l, w)
                assert c3 == (0,) + c2


@pytest.mark.parametrize("spt,tpw,wpc,order", [
    ([2, 1, 4], [2, 4, 4], [1, 2, 2], [2, 0, 1]),
    ([1, 2, 1, 2], [2, 2, 4, 2], [2, 1, 2, 1], [1, 3, 0, 2]),
])
def test_blocked_rank_n_is_a_bijection_on_one_cta_tile(spt, tpw, wpc, order):
    # shape == CTA tile: every element has exactly one owner
    shape = [s * t * w for s, t, w in zip(spt, tpw, wpc)]
    regs = int(np.prod(spt))
    lanes, warps = int(np.prod(tpw)), int(np.prod(wpc))
    seen = {lo.blocked_coordinate(spt, tpw, wpc, order, shape, r, l, w)
            for r in range(regs) for l in range(lanes) for w in range(warps)}
    assert len(seen) == int(np.prod(shape)) == regs * lanes * warps
    assert all(all(0 <= c[d] < shape[d] for d in range(len(shape))) for c in seen)


def test_blocked_rank_n_permuting_dims_permutes_coordinates():
    # relabelling dims (order relabelled to match) relabels each coordinate
    spt, tpw, wpc, order, shape = [2, 1, 4], [2, 4, 4], [1, 2, 2], [2, 0, 1], [8, 16, 64]
    perm = [1, 2, 0]  # new dim i is old dim perm[i]
    inv = [perm.index(d) for d in range(3)]
    P = lambda v: [v[perm[i]] for i in range(3)]
    for r in range(16):
        for l in range(32):
            for w in range(4):
                a = lo.blocked_coordinate(spt, tpw, wpc, order, shape, r, l, w)
                b = lo.blocked_coordinate(P(spt), P(tpw), P(wpc), [inv[d] for d in order],
                                          P(shape), r, l, w)
                assert b == tuple(P(a))
