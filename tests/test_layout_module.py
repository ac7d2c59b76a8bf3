"""The product's GF(2) layout module (C++, through the C ABI) against the layout
oracle: the pages' printed examples, the pages' ownership rules written as
integer formulas, and brute-force enumeration of every input.  No GPU."""
import itertools

import numpy as np
import pytest

from oracle import layout_oracle as lo
from conftest import load_golden


def tuple_of(L):
    return L.as_tuple()


def same_table(L, ref_fn):
    """L.apply(x) == ref_fn(x) for every input x."""
    T = tuple_of(L)
    for x in lo.all_inputs(T):
        assert L.apply(x) == ref_fn(x), x


def test_create_and_apply_page_example(tg):
    g = load_golden("linear_layout_lane_warp.json")
    L = tg.LinearLayout.create([tuple(d) for d in g["in_dims"]], [tuple(d) for d in g["out_dims"]],
                               g["bases"])
    for ev in g["evaluations"]:
        assert L.apply(ev["in"]) == tuple(ev["out"])
    same_table(L, lambda x: (x["lane"], x["lane"] ^ x["warp"]))
    assert L.in_dims == [("lane", 2), ("warp", 2)]
    assert L.out_dims == [("row", 2), ("col", 2)]


def test_blocked_constructor_matches_page(tg):
    g = load_golden("blocked_32x32.json")
    L = tg.LinearLayout.blocked(g["size_per_thread"], g["threads_per_warp"], g["warps_per_cta"],
                                g["order"], g["shape"])
    assert L.bases == {k: [tuple(v) for v in vs] for k, vs in g["bases"].items()}
    ev = g["evaluations"][0]
    assert L.apply(ev["in"]) == tuple(ev["out"])
    assert L.is_injective and L.is_surjective and L.rank == 10


@pytest.mark.parametrize("spt,tpw,wpc,order,shape", [
    ([1, 1], [1, 32], [4, 1], [1, 0], [32, 32]),
    ([2, 4], [4, 8], [2, 2], [1, 0], [64, 128]),
    ([1, 8], [8, 4], [1, 4], [0, 1], [16, 256]),
    ([4, 1], [2, 16], [2, 2], [0, 1], [8, 64]),     # CTA tile wider than dim0: broadcast
    ([1, 2], [32, 1], [1, 1], [1, 0], [16, 4]),     # lanes beyond the shape broadcast
])
def test_blocked_constructor_matches_integer_rule(tg, spt, tpw, wpc, order, shape):
    L = tg.LinearLayout.blocked(spt, tpw, wpc, order, shape)
    same_table(L, lambda x: lo.blocked_coordinate(spt, tpw, wpc, order, shape, x["register"],
                                                  x["lane"], x["warp"]))


@pytest.mark.parametrize("shape,threads,order", [
    ((4, 16), 32, (1, 0)), ((16, 8), 32, (1, 0)), ((64, 64), 256, (1, 0)),
    ((8, 32), 64, (0, 1)), ((32, 32), 32, (1, 0)),
])
def test_cooperative_constructor(tg, shape, threads, order):
    L = tg.LinearLayout.cooperative(shape, threads, order)
    same_table(L, lambda x: lo.cooperative_coordinate(shape, threads, order, x["thread"],
                                                      x["iteration"]))
    assert L.is_injective and L.is_surjective


def test_cooperative_page_examples(tg):
    g = load_golden("cooperative_tiles.json")
    for case in g["cases"]:
        L = tg.LinearLayout.cooperative(case["shape"], g["threads"], g["order"])
        for v in case["visits"]:
            got = [L.apply({"thread": v["thread"], "iteration": it}) for it in range(case["iterations"])]
            assert got == [tuple(c) for c in v["coords"]]


@pytest.mark.parametrize("logical,thread_shape", [((8, 8), (4, 8)), ((16, 16), (4, 8)),
                                                  ((64, 32), (8, 4)), ((4, 8), (4, 8))])
def test_register_tile_constructor(tg, logical, thread_shape):
    L = tg.LinearLayout.register_tile(logical, thread_shape)
    rs = lo.register_shape(logical, thread_shape)

    def ref(x):
        th = lo.thread_coordinate(x["thread"], thread_shape)
        r = (x["register"] // rs[1], x["register"] % rs[1])
        return lo.register_tile_coordinate(logical, thread_shape, th, r)
    same_table(L, ref)


def test_register_tile_page_examples(tg):
    g = load_golden("register_tiles.json")
    for case in g["cases"]:
        L = tg.LinearLayout.register_tile(case["logical"], case["thread_shape"])
        ts = case["thread_shape"]
        rs = case["register_shape"]
        t = case["thread"][0] * ts[1] + case["thread"][1]
        for own in case["owns"]:
            r = own["register"][0] * rs[1] + own["register"][1]
            assert L.apply({"register": r, "thread": t}) == tuple(own["logical"])


@pytest.mark.parametrize("rows", [8, 64, 128, 256])
def test_swizzle128_constructor(tg, rows):
    L = tg.LinearLayout.swizzle128(rows, 2)
    inv = {}
    for r in range(rows):
        for c in range(64):
            inv[lo.swizzle128_offset(r, c, 2) // 2] = (r, c)
    same_table(L, lambda x: inv[x["offset"]])
    assert L.is_injective and L.is_surjective


@pytest.mark.parametrize("bn", [32, 64, 128, 256])
def test_tmem_constructor(tg, bn):
    L = tg.LinearLayout.tmem_32x32b(bn)
    same_table(L, lambda x: lo.tmem_32x32b_coordinate(x["warp"], x["lane"], x["register"]))
    assert L.is_injective and L.is_surjective


# --- algebra against brute force ------------------------------------------

def random_layout(tg, rng, in_bits, out_bits, zero_prob=0.15, names=("a", "b", "c")):
    ins = [(names[i], b) for i, b in enumerate(in_bits)]
    outs = [(f"o{i}", b) for i, b in enumerate(out_bits)]
    bases = {}
    for name, b in ins:
        bases[name] = [tuple(0 if rng.random() < zero_prob else int(rng.integers(0, 1 << ob))
                             for _, ob in outs) for _ in range(b)]
    return tg.LinearLayout.create(ins, outs, bases)


@pytest.mark.parametrize("seed", range(25))
def test_apply_rank_injective_surjective(tg, seed):
    rng = np.random.default_rng(seed)
    L = random_layout(tg, rng, [int(rng.integers(0, 5)) for _ in range(3)],
                      [int(rng.integers(1, 4)) for _ in range(2)])
    T = tuple_of(L)
    same_table(L, lambda x: lo.apply(T, x))
    assert L.rank == lo.rank_by_enumeration(T)
    assert L.is_injective == lo.is_injective(T)
    assert L.is_surjective == lo.is_surjective(T)


@pytest.mark.parametrize("seed", range(15))
def test_compose_is_function_composition(tg, seed):
    rng = np.random.default_rng(1000 + seed)
    inner = random_layout(tg, rng, [int(rng.integers(0, 4)) for _ in range(2)], [3, 2])
    outer_in = [("o0", 3), ("o1", 2)]
    outer = tg.LinearLayout.create(outer_in, [("x", 4), ("y", 3)],
                                   {n: [(int(rng.integers(0, 16)), int(rng.integers(0, 8)))
                                        for _ in range(b)] for n, b in outer_in})
    C = inner.compose(outer)
    Ti, To = tuple_of(inner), tuple_of(outer)
    same_table(C, lambda x: lo.apply(To, dict(zip(["o0", "o1"], lo.apply(Ti, x)))))


@pytest.mark.parametrize("seed", range(10))
def test_product_rule(tg, seed):
    rng = np.random.default_rng(2000 + seed)
    # a: (a, b) -> (o0, o1); f: (b, c) -> (o1, o2): shares input dim b and output dim o1
    A = random_layout(tg, rng, [2, 2], [2, 3], names=("a", "b"))
    ins = [("b", 1), ("c", 2)]
    outs = [("o1", 2), ("o2", 2)]
    B = tg.LinearLayout.create(ins, outs, {n: [(int(rng.integers(0, 4)), int(rng.integers(0, 4)))
                                               for _ in range(b)] for n, b in ins})
    P = A * B
    assert P.in_dims == [("a", 2), ("b", 3), ("c", 2)]
    assert P.out_dims == [("o0", 2), ("o1", 5), ("o2", 2)]
    TA, TB = tuple_of(A), tuple_of(B)

    def ref(x):
        xa = {"a": x["a"], "b": x["b"] & 3}
        xb = {"b": x["b"] >> 2, "c": x["c"]}
        o0, o1a = lo.apply(TA, xa)
        o1b, o2 = lo.apply(TB, xb)
        return (o0, o1a | (o1b << 3), o2)
    same_table(P, ref)


@pytest.mark.parametrize("seed", range(20))
def test_invert_and_compose_is_a_right_inverse(tg, seed):
    rng = np.random.default_rng(3000 + seed)
    # S: shared offset (+ a broadcast dim) -> (row, col), surjective; R: (reg, lane) -> (row, col)
    while True:
        S = random_layout(tg, rng, [5, int(rng.integers(0, 3))], [3, 2], zero_prob=0.1,
                          names=("offset", "bcast"))
        if S.is_surjective:
            break
    R = random_layout(tg, rng, [int(rng.integers(0, 4)), int(rng.integers(0, 4))], [3, 2],
                      names=("reg", "lane"))
    X = R.invert_and_compose(S)
    assert X.in_dims == R.in_dims and X.out_dims == S.in_dims
    TS, TR = tuple_of(S), tuple_of(R)
    for x in lo.all_inputs(TR):
        assert lo.apply(TS, dict(zip([n for n, _ in TS[0]], X.apply(x)))) == lo.apply(TR, x)


def test_invert_and_compose_swizzle_gives_store_offsets(tg):
    # register tile -> tensor coords, then through the inverse swizzle: the
    # shared offset where the epilogue thread must store each value.
    S = tg.LinearLayout.swizzle128(128, 2).transpose_outs(["row", "col"])
    R = tg.LinearLayout.tmem_32x32b(64).sublayout(["register", "lane", "warp"], ["m", "n"])
    R = tg.LinearLayout.create(R.in_dims, [("row", 7), ("col", 6)], R.bases)
    X = R.invert_and_compose(S)
    for x in [{"register": 5, "lane": 3, "warp": 2}, {"register": 63, "lane": 31, "warp": 3}]:
        m, n = R.apply(x)
        assert X.apply(x) == (lo.swizzle128_offset(m, n, 2) // 2,)


def test_invert_and_compose_rejects_outside_image(tg):
    S = tg.LinearLayout.create([("offset", 2)], [("row", 2), ("col", 1)],
                               {"offset": [(1, 0), (2, 0)]})  # never reaches col=1
    R = tg.LinearLayout.create([("lane", 1)], [("row", 2), ("col", 1)], {"lane": [(0, 1)]})
    with pytest.raises(tg.TileGemmError):
        R.invert_and_compose(S)


def test_sublayout_and_transpose(tg):
    L = tg.LinearLayout.blocked([1, 1], [1, 32], [4, 1], [1, 0], [32, 32])
    s = L.sublayout(["lane"], ["dim1"])
    assert s.bases == {"lane": [(1,), (2,), (4,), (8,), (16,)]}
    t = L.transpose_outs(["dim1", "dim0"])
    assert t.apply({"register": 5, "lane": 3, "warp": 2}) == (3, 22)


def test_invariant_violations_rejected(tg):
    with pytest.raises(tg.TileGemmError):  # coordinate does not fit the out dim
        tg.LinearLayout.create([("a", 1)], [("x", 2)], {"a": [(4,)]})
    with pytest.raises(tg.TileGemmError):  # duplicate names
        tg.LinearLayout.create([("a", 1), ("a", 1)], [("x", 2)], {"a": [(1,), (2,)]})
    with pytest.raises(tg.TileGemmError):  # not a power of two
        tg.LinearLayout.blocked([1, 1], [1, 32], [3, 1], [1, 0], [32, 32])
    with pytest.raises(tg.TileGemmError):
        tg.LinearLayout.cooperative((4, 16), 128, (1, 0))  # more threads than elements
    a = tg.LinearLayout.create([("a", 1)], [("x", 2)], {"a": [(1,)]})
    with pytest.raises(tg.TileGemmError):  # out dims of inner != in dims of outer
        a.compose(a)
