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


@pytest.mark.parametrize("spt,tpw,wpc,order,shape", [
    ([1], [32], [4], [0], [512]),                                      # rank 1, repetitions
    ([1, 1, 1], [1, 1, 32], [1, 4, 1], [2, 1, 0], [1, 32, 32]),        # a unit dim before 2-D
    ([2, 1, 4], [2, 4, 4], [1, 2, 2], [2, 0, 1], [8, 16, 64]),
    ([1, 2, 2], [4, 2, 4], [2, 2, 1], [0, 2, 1], [4, 32, 16]),         # dim0 tile wider: broadcast
    ([1, 1, 2, 2], [2, 2, 2, 4], [1, 2, 1, 2], [3, 2, 1, 0], [4, 8, 8, 32]),
])
def test_blocked_nd_matches_integer_rule(tg, spt, tpw, wpc, order, shape):
    L = tg.LinearLayout.blocked_nd(spt, tpw, wpc, order, shape)
    assert L.out_dims == [(f"dim{d}", int(np.log2(shape[d]))) for d in range(len(shape))]
    same_table(L, lambda x: lo.blocked_coordinate(spt, tpw, wpc, order, shape, x["register"],
                                                  x["lane"], x["warp"]))


def test_blocked_nd_rank2_is_the_rank2_constructor(tg):
    args = ([2, 4], [4, 8], [2, 2], [1, 0], [64, 128])
    assert tg.LinearLayout.blocked_nd(*args).bases == tg.LinearLayout.blocked(*args).bases


def test_blocked_nd_checks(tg):
    bad = [
        ([1, 1, 1], [1, 1, 32], [1, 4, 1], [2, 2, 0], [1, 32, 32]),   # order not a permutation
        ([1, 1, 1], [1, 1, 32], [1, 4, 1], [2, 1, 3], [1, 32, 32]),   # order out of range
        ([1, 1, 1], [1, 1, 24], [1, 4, 1], [2, 1, 0], [1, 32, 32]),   # not a power of two
    ]
    for args in bad:
        with pytest.raises(tg.TileGemmError) as e:
            tg.LinearLayout.blocked_nd(*args)
        assert e.value.status == tg.TG_ERR_LAYOUT
    with pytest.raises(tg.TileGemmError) as e:
        tg.LinearLayout.blocked_nd([1] * 9, [1] * 9, [1] * 9, list(range(9)), [2] * 9)
    assert e.value.status == tg.TG_ERR_INVALID_ARG
    with pytest.raises(tg.TileGemmError):
        tg.LinearLayout.blocked_nd([1, 1], [1], [1, 1], [1, 0], [2, 2])  # ragged arguments


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


# --- transposeIns, reshapeIns / reshapeOuts, divideLeft / divideRight ------
# (Triton LinearLayout, "Combining layouts".  The page only names them; the
# readings taken are stated in include/tilegemm.h.  Each test checks the
# result by evaluating every input with the layout oracle.)

def flat(dims, values):
    """Flattened index of a dims-ordered coordinate, first dim least significant."""
    v, shift = 0, 0
    for (_, b), x in zip(dims, values):
        v |= x << shift
        shift += b
    return v


def split(dims, f):
    out, shift = [], 0
    for _, b in dims:
        out.append((f >> shift) & ((1 << b) - 1))
        shift += b
    return out


@pytest.mark.parametrize("seed", range(10))
def test_transpose_ins_keeps_the_map(tg, seed):
    rng = np.random.default_rng(4000 + seed)
    L = random_layout(tg, rng, [int(rng.integers(0, 4)) for _ in range(3)], [3, 2])
    order = [("a", "b", "c"), ("c", "a", "b"), ("b", "c", "a")][seed % 3]
    T = L.transpose_ins(list(order))
    assert [n for n, _ in T.in_dims] == list(order)
    assert dict(T.in_dims) == dict(L.in_dims) and T.out_dims == L.out_dims
    TL = tuple_of(L)
    same_table(T, lambda x: lo.apply(TL, x))
    with pytest.raises(tg.TileGemmError):
        L.transpose_ins(["a", "b"])  # must name every dim


@pytest.mark.parametrize("seed", range(10))
def test_reshape_ins_keeps_the_flattened_index(tg, seed):
    rng = np.random.default_rng(5000 + seed)
    bits = [int(rng.integers(1, 4)) for _ in range(3)]
    L = random_layout(tg, rng, bits, [3, 3])
    total = sum(bits)
    cut = int(rng.integers(0, total + 1))
    new = [("p", cut), ("q", total - cut)]
    R = L.reshape_ins(new)
    assert R.in_dims == new and R.out_dims == L.out_dims
    TL, TR = tuple_of(L), tuple_of(R)
    for f in range(1 << total):
        old_x = dict(zip([n for n, _ in TL[0]], split(TL[0], f)))
        new_x = dict(zip([n for n, _ in TR[0]], split(TR[0], f)))
        assert R.apply(new_x) == lo.apply(TL, old_x), f
    with pytest.raises(tg.TileGemmError):
        L.reshape_ins([("p", total + 1)])


@pytest.mark.parametrize("seed", range(10))
def test_reshape_outs_keeps_the_flattened_coordinate(tg, seed):
    rng = np.random.default_rng(6000 + seed)
    L = random_layout(tg, rng, [2, 3], [2, 3, 2], names=("a", "b"))
    new = [("flat", 7)] if seed % 2 else [("lo", 4), ("hi", 3)]
    R = L.reshape_outs(new)
    assert R.out_dims == new and R.in_dims == L.in_dims
    TL = tuple_of(L)
    for x in lo.all_inputs(TL):
        assert flat(new, R.apply(x)) == flat(TL[1], lo.apply(TL, x))
    with pytest.raises(tg.TileGemmError):
        L.reshape_outs([("flat", 6)])


def product_by_rule(TB, TC, x, A_dims):
    """(B * C)(x) written out from the product rule: for a dim both factors
    have, B owns the low input bits and the low output bits."""
    in_b, in_c = dict(TB[0]), dict(TC[0])
    xb = {n: x[n] & ((1 << b) - 1) for n, b in in_b.items()}
    xc = {n: x[n] >> in_b.get(n, 0) for n in in_c}
    ob = dict(zip([n for n, _ in TB[1]], lo.apply(TB, xb)))
    oc = dict(zip([n for n, _ in TC[1]], lo.apply(TC, xc)))
    out_b = dict(TB[1])
    return tuple(ob.get(n, 0) | (oc.get(n, 0) << out_b.get(n, 0)) for n, _ in A_dims)


@pytest.mark.parametrize("seed", range(12))
def test_divide_left_and_right_invert_the_product(tg, seed):
    rng = np.random.default_rng(7000 + seed)
    # B: (a, b) -> (o0, o1); C: (b, c) -> (o1, o2), sharing input b and output o1
    B = random_layout(tg, rng, [int(rng.integers(0, 3)), int(rng.integers(1, 3))], [2, 2],
                      names=("a", "b"))
    cin = [("b", int(rng.integers(0, 3))), ("c", int(rng.integers(1, 3)))]
    cout = [("o1", 2), ("o2", 2)]
    C = tg.LinearLayout.create(cin, cout, {n: [tuple(int(rng.integers(0, 4)) for _ in cout)
                                               for _ in range(b)] for n, b in cin})
    # left: A = B * C
    A = B * C
    TB, TC, TA = tuple_of(B), tuple_of(C), tuple_of(A)
    for x in lo.all_inputs(TA):  # the product itself, by the rule
        assert lo.apply(TA, x) == product_by_rule(TB, TC, x, TA[1])
    Cl = A.divide_left(B)
    assert [n for n, _ in Cl.in_dims] == [n for n, _ in A.in_dims]
    TCl = tuple_of(Cl)
    for x in lo.all_inputs(TA):
        assert lo.apply(TA, x) == product_by_rule(TB, TCl, x, TA[1])
    # right: A2 = C * B, divided by B on the right gives back C's map
    A2 = C * B
    Cr = A2.divide_right(B)
    TA2, TCr = tuple_of(A2), tuple_of(Cr)
    for x in lo.all_inputs(TA2):
        assert lo.apply(TA2, x) == product_by_rule(TCr, TB, x, TA2[1])


def test_divide_rejects_a_non_factor(tg):
    B = tg.LinearLayout.create([("lane", 1)], [("x", 1)], {"lane": [(1,)]})
    A = tg.LinearLayout.create([("lane", 2)], [("x", 2)], {"lane": [(2,), (1,)]})
    with pytest.raises(tg.TileGemmError):  # A's low lane bit does not map as B's does
        A.divide_left(B)
    ok = tg.LinearLayout.create([("lane", 2)], [("x", 2)], {"lane": [(1,), (2,)]})
    assert ok.divide_left(B).bases == {"lane": [(1,)]}
    assert ok.divide_right(B).bases == {"lane": [(1,)]}
    big = tg.LinearLayout.create([("lane", 3)], [("x", 1)], {"lane": [(1,), (0,), (0,)]})
    with pytest.raises(tg.TileGemmError):  # B needs more output bits than A has left
        tg.LinearLayout.create([("lane", 1)], [("x", 1)], {"lane": [(1,)]}).divide_left(big)


def folded_cases(tg):
    g = load_golden("linear_layout_lane_warp.json")
    page = tg.LinearLayout.create([tuple(d) for d in g["in_dims"]],
                                  [tuple(d) for d in g["out_dims"]], g["bases"])
    blocked = tg.LinearLayout.blocked([2, 4], [4, 8], [2, 2], [1, 0], [64, 128])
    tmem = tg.LinearLayout.tmem_32x32b(256)
    swz = tg.LinearLayout.swizzle128(64, 2)
    nd = tg.LinearLayout.blocked_nd([1, 2, 2], [4, 2, 4], [2, 2, 1], [0, 2, 1], [4, 32, 16])
    return [
        (page, {}), (page, {"warp": 2}), (page, {"lane": 3, "warp": 1}),
        # the page's example: register 3 folded, lane and warp variable
        (blocked, {"register": 3}), (blocked, {"warp": 2}), (blocked, {}),
        (tmem, {"register": 17}), (tmem, {"warp": 3, "lane": 5}),
        (swz, {}), (nd, {"register": 5, "warp": 1}),
    ]


def test_folded_layout_matches_apply_on_every_input(tg):
    for L, fixed in folded_cases(tg):
        F = L.fold(fixed)
        T = tuple_of(L)
        for x in lo.all_inputs(T):
            if any(x[n] != v for n, v in fixed.items()):
                continue
            want = lo.apply(T, x)
            assert F.apply({n: x[n] for n in F.var_names}) == want, (fixed, x)
            assert L.apply(x) == want


def test_folded_layout_structure(tg):
    # constant part = the layout applied to the fixed inputs alone; one packed
    # column per variable bit; outputs packed low to high in layout order
    L = tg.LinearLayout.blocked([2, 4], [4, 8], [2, 2], [1, 0], [64, 128])
    F = L.fold({"register": 3})
    r = F.raw
    assert r.n_vars == 2 and list(r.var_bits[:2]) == [5, 2] and r.n_bits == 7
    assert r.n_outs == 2 and list(r.out_shift[:2]) == [0, 6] and list(r.out_bits[:2]) == [6, 7]
    c = L.apply({"register": 3, "lane": 0, "warp": 0})
    assert r.constant == c[0] | (c[1] << 6)
    lane_bases = L.bases["lane"]
    for i, (d0, d1) in enumerate(lane_bases):
        assert r.cols[i] == d0 | (d1 << 6)


def test_fold_checks(tg):
    L = tg.LinearLayout.blocked([2, 4], [4, 8], [2, 2], [1, 0], [64, 128])
    for fixed in ({"nope": 0}, {"lane": 32}, {"lane": -1}):
        with pytest.raises(tg.TileGemmError) as e:
            L.fold(fixed)
        assert e.value.status == tg.TG_ERR_LAYOUT
    F = L.fold({})
    with pytest.raises(tg.TileGemmError) as e:
        F.apply({"register": 64, "lane": 0, "warp": 0})  # register has 5 bits
    assert e.value.status == tg.TG_ERR_INVALID_ARG
    # more than 32 variable input bits cannot be packed into one word
    big = tg.LinearLayout.create([("a", 20), ("b", 20)], [("x", 20), ("y", 20)],
                                 {"a": [(1 << i, 0) for i in range(20)],
                                  "b": [(0, 1 << i) for i in range(20)]})
    with pytest.raises(tg.TileGemmError) as e:
        big.fold({})
    assert e.value.status == tg.TG_ERR_LAYOUT
    with pytest.raises(tg.TileGemmError) as e:
        big.fold({"a": 5})  # 20 variable bits fit, but the outputs need 40
    assert e.value.status == tg.TG_ERR_LAYOUT
