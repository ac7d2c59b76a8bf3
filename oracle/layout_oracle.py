"""Layout oracle -- test infrastructure only (see ``oracle/__init__.py``).

Everything here is evaluated by brute force or by the pages' ownership rules
written out with ordinary integer arithmetic, so the product's GF(2) layout
module (C++) can be checked against it bit for bit.

A layout is given as ``(in_dims, out_dims, bases)``:
  * ``in_dims``:  list of ``(name, size_log2)``, in order;
  * ``out_dims``: list of ``(name, size_log2)``, in order;
  * ``bases``:    dict ``name -> list`` of ``size_log2`` basis vectors, each a
    tuple with one coordinate per output dim.
This is the representation of retepy.com "Triton LinearLayout", section
"Basis-vector representation": one basis per input bit, one coordinate per
output dimension.
"""
from __future__ import annotations

import itertools
import math


def apply(layout, ins: dict) -> tuple:
    """Triton LinearLayout, section "LinearLayout::apply": for every output
    coordinate, XOR together the basis vectors of the set input bits."""
    in_dims, out_dims, bases = layout
    out = []
    for o, _ in enumerate(out_dims):
        v = 0
        for name, nbits in in_dims:
            x = ins[name]
            for i in range(nbits):
                if (x >> i) & 1:
                    v ^= bases[name][i][o]
        out.append(v)
    return tuple(out)


def all_inputs(layout):
    """Every input tuple, first input dim varying fastest."""
    in_dims = layout[0]
    ranges = [range(1 << b) for _, b in in_dims]
    for combo in itertools.product(*reversed(ranges)):
        yield {name: v for (name, _), v in zip(in_dims, reversed(combo))}


def table(layout) -> list:
    return [apply(layout, x) for x in all_inputs(layout)]


def image_size(layout) -> int:
    return len(set(table(layout)))


def rank_by_enumeration(layout) -> int:
    """The image of a GF(2)-linear map is a subspace, so |image| = 2^rank."""
    n = image_size(layout)
    r = int(math.log2(n))
    assert 1 << r == n, "image size of a linear map must be a power of two"
    return r


def is_injective(layout) -> bool:
    t = table(layout)
    return len(set(t)) == len(t)


def is_surjective(layout) -> bool:
    total = sum(b for _, b in layout[1])
    return image_size(layout) == 1 << total


def out_as_dict(layout, out: tuple) -> dict:
    return {name: v for (name, _), v in zip(layout[1], out)}


# ---------------------------------------------------------------------------
# Ownership rules of the pages, as plain integer formulas
# ---------------------------------------------------------------------------

def thread_coordinate(t: int, thread_shape: tuple) -> tuple:
    """pbelevich.github.io Part 12, "One shape was doing too many jobs": the
    generated prologue decodes the linear thread id row-major,
    tile_i = t / cols, tile_j = t % cols."""
    cols = thread_shape[1]
    return (t // cols, t % cols)


def cooperative_coordinate(shape: tuple, threads: int, order: tuple, t: int, it: int):
    """Part 12, "Cooperative tile layouts": thread t at iteration it visits
    linear index t + it * threads; the coordinate is peeled axis by axis in
    ``order`` (fastest axis first).  Returns None for an inactive tail lane."""
    size = math.prod(shape)
    linear = t + it * threads
    if linear >= size:
        return None
    coord = [0] * len(shape)
    rem = linear
    for axis in order:
        coord[axis] = rem % shape[axis]
        rem //= shape[axis]
    return tuple(coord)


def cooperative_iterations(shape: tuple, threads: int) -> int:
    return -(-math.prod(shape) // threads)


def register_tile_coordinate(logical: tuple, thread_shape: tuple, thread: tuple,
                             register: tuple) -> tuple:
    """pbelevich.github.io Part 16, "A strided ownership rule":
    logical = thread + register * thread_shape, per axis."""
    return tuple(th + r * ts for th, r, ts in zip(thread, register, thread_shape))


def register_shape(logical: tuple, thread_shape: tuple) -> tuple:
    """Part 16, "Describing the mapping": elementwise quotient."""
    return tuple(l // t for l, t in zip(logical, thread_shape))


def blocked_coordinate(spt, tpw, wpc, order, shape, reg: int, lane: int, warp: int) -> tuple:
    """Owner -> element of a Triton blocked encoding, in integer arithmetic.

    Along each dim d the CTA tile is spt[d] * tpw[d] * wpc[d] elements and is
    repeated rep[d] = shape[d] / tile[d] times.  Lane and warp ids are split
    over the dims in ``order`` (minor dim first).  The register id holds first
    the per-thread elements (spt, dims in ``order``), then the repetitions
    (dims in ``order``).  Element coordinate:
        x[d] = rep_idx[d]*tile[d] + warp_idx[d]*spt[d]*tpw[d] + lane_idx[d]*spt[d] + elem_idx[d]
    (retepy.com "Triton LinearLayout", "Blocked-layout example").
    """
    rank = len(shape)
    tile = [spt[d] * tpw[d] * wpc[d] for d in range(rank)]
    rep = [max(1, shape[d] // tile[d]) for d in range(rank)]

    def split(x, sizes):
        out = [0] * rank
        for d in order:
            out[d] = x % sizes[d]
            x //= sizes[d]
        return out, x

    lane_idx, _ = split(lane, tpw)
    warp_idx, _ = split(warp, wpc)
    elem_idx, rest = split(reg, spt)
    rep_idx, _ = split(rest, rep)
    return tuple((rep_idx[d] * tile[d] + warp_idx[d] * spt[d] * tpw[d]
                  + lane_idx[d] * spt[d] + elem_idx[d]) % shape[d] for d in range(rank))


def swizzle128_offset(row: int, col: int, elem_bytes: int) -> int:
    """Byte offset of element (row, col) of a tile with 128-byte rows stored
    with the 128-byte XOR swizzle: the 16-byte chunk index inside each
    128-byte row is XORed with (row mod 8), so one 1024-byte atom of 8 rows
    touches every bank once per chunk column."""
    byte = col * elem_bytes
    assert 0 <= byte < 128
    chunk = (byte >> 4) ^ (row & 7)
    return row * 128 + (chunk << 4) + (byte & 15)


def tmem_32x32b_coordinate(warp: int, lane: int, reg: int, col_base: int = 0) -> tuple:
    """Accumulator element that thread ``lane`` of warp ``warp`` receives in
    register ``reg`` of a tcgen05.ld of shape 32x32b: the warp reads TMEM lanes
    32*(warp % 4) .. +31, thread t gets lane 32*(warp%4)+t, and register j
    holds column col_base + j.  For an M=128 single-CTA accumulator TMEM lane
    is the tile row and the column is the tile column."""
    return (32 * (warp % 4) + lane, col_base + reg)
