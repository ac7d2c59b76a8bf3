"""The tile selector's host logic (no GPU): deterministic choices for the
benchmark workloads and structural invariants for arbitrary shapes."""
import math
import os

import numpy as np
import pytest

F16, BF16 = 0, 1


def cfg(tg, *args, sms=152):
    return tg.parse_config(tg.tg_query_config_for_sms(sms, *args))


def test_benchmark_workload_choices(tg):
    # dense square and large GEMMs run on CTA pairs with the widest tile
    c = cfg(tg, 4096, 4096, 4096, F16, 0, 0)
    assert (c["swap"], c["pair"], c["bm"], c["bn"], c["grid"]) == (0, 1, 256, 256, 152)
    c = cfg(tg, 8192, 8192, 4096, F16, 0, 0)
    assert (c["pair"], c["bn"], c["tiles"]) == (1, 256, 1024)
    # 16384 x 1024 x 8192: 4 tile columns, so raster groups of 19 tile rows
    # (76 tiles: one wave of CTA pairs)
    c = cfg(tg, 16384, 1024, 8192, BF16, 0, 0)
    assert (c["pair"], c["bn"], c["group_m"]) == (1, 256, 19)
    # K = 1000 (16 K-blocks) is too shallow for stream-K: both 256 x 256 (192
    # tiles) and 256 x 224 (224 tiles) take three whole waves and stage 256
    # B columns per tile; the narrower one computes fewer columns
    c = cfg(tg, 4000, 3000, 1000, F16, 1, 0)
    assert (c["pair"], c["bm"], c["bn"], c["tiles"], c["sk_tiles"]) == (1, 256, 224, 224, 0)
    # M = 32 cannot fill the accumulator lanes: operands swap, one 32-wide column
    c = cfg(tg, 32, 16384, 16384, BF16, 0, 0)
    assert (c["swap"], c["pair"], c["bn"], c["tiles"], c["grid"]) == (1, 0, 32, 128, 128)


def test_deterministic(tg):
    a = tg.tg_query_config_for_sms(152, 3000, 5000, 700, F16, 1, 0)
    b = tg.tg_query_config_for_sms(152, 3000, 5000, 700, F16, 1, 0)
    assert a == b


@pytest.mark.parametrize("seed", range(40))
def test_invariants(tg, seed):
    rng = np.random.default_rng(seed)
    M, N, K = (int(x) for x in rng.integers(1, 20000, 3))
    pa, pb = (int(x) for x in rng.integers(0, 2, 2))
    sms = int(rng.choice([8, 64, 148, 152]))
    c = cfg(tg, M, N, K, F16, pa, pb, sms=sms)
    assert c["bm"] == (256 if c["pair"] else 128)
    Mk, Nk = (N, M) if c["swap"] else (M, N)
    assert c["tiles"] == math.ceil(Mk / c["bm"]) * math.ceil(Nk / c["bn"])
    slots = sms // 2 if c["pair"] else sms
    assert 1 <= c["grid"] <= (2 * slots if c["pair"] else slots)
    if c["pair"]:
        assert c["grid"] % 2 == 0 and c["grid"] // 2 <= c["tiles"]
    else:
        assert c["grid"] <= c["tiles"]
    # raster groups: 16 tile rows, widened to a whole wave when there are few
    # tile columns, never more rows than the problem has
    tiles_m, tiles_n = math.ceil(Mk / c["bm"]), math.ceil(Nk / c["bn"])
    workers = c["grid"] // 2 if c["pair"] else c["grid"]
    assert c["stages"] >= 4 and 1 <= c["group_m"] <= tiles_m
    assert c["group_m"] == min(tiles_m, 16 if tiles_n * 16 >= workers else -(-workers // tiles_n))
    q_mn = (pa == 1) if c["swap"] else (pb == 0)
    assert not (c["bn"] == 32 and q_mn)
    assert c["swap"] == (1 if (M <= 64 and N > M) else 0)


def test_force_override(tg, monkeypatch):
    monkeypatch.setenv("TG_FORCE_CONFIG", "pair=0,bn=192,group_m=2,grid=40")
    c = cfg(tg, 4096, 4096, 4096, F16, 0, 0)
    assert (c["pair"], c["bn"], c["group_m"], c["grid"]) == (0, 192, 2, 40)
    monkeypatch.setenv("TG_FORCE_CONFIG", "pair=1,bn=64")  # not compiled for pairs
    c = cfg(tg, 4096, 4096, 4096, F16, 0, 0)
    assert c["bn"] in (32, 64, 128, 192, 224, 256) and c["stages"] > 0
    monkeypatch.setenv("TG_FORCE_CONFIG", "bn=32")  # MN-major B cannot use 32-wide tiles
    c = cfg(tg, 4096, 4096, 4096, F16, 0, 0)
    assert c["bn"] != 32


def test_rejects_bad_shape(tg):
    with pytest.raises(tg.TileGemmError):
        tg.tg_query_config_for_sms(152, 0, 1, 1, F16)
    with pytest.raises(tg.TileGemmError):
        tg.tg_query_config_for_sms(1, 16, 16, 16, F16)


def test_stream_k_split(tg):
    # 256 pair tiles over 76 clusters: 2 whole waves, then 76 + 28 tiles dealt out in K-ranges
    c = cfg_sk(tg, 4096, 4096, 4096, F16, 0, 0)
    assert (c["pair"], c["bn"], c["grid"], c["tiles"], c["sk_tiles"]) == (1, 256, 152, 256, 104)
    assert c["sk_cmax"] == 2
    counters = -(-(76 * 2 * 4) // 256) * 256
    assert c["ws_bytes"] == counters + 76 * 2 * 256 * 256 * 4
    # whole waves: nothing to split
    c = cfg_sk(tg, 256 * 76 // 4, 1024, 4096, F16, 0, 0)  # 19 x 4 = 76 tiles
    assert c["sk_tiles"] == 0 and c["ws_bytes"] == 0
    # fewer tiles than workers, full waves or shallow K: whole tiles only
    assert cfg_sk(tg, 32, 16384, 16384, BF16, 0, 0)["sk_tiles"] == 0
    assert cfg_sk(tg, 2048, 2048, 4096, F16, 0, 0)["sk_tiles"] == 0   # 64 pair tiles, 76 clusters
    assert cfg_sk(tg, 8192, 8192, 4096, F16, 0, 0)["sk_tiles"] == 0   # 13.5 waves: 96 % full
    assert cfg_sk(tg, 4000, 3000, 1000, F16, 1, 0)["sk_tiles"] == 0   # 16 K-blocks
    # without a workspace the same shapes keep whole tiles
    assert cfg(tg, 4096, 4096, 4096, F16, 0, 0)["sk_tiles"] == 0


def cfg_sk(tg, *args, sms=152):
    return tg.parse_config(tg.tg_query_config_for_sms(sms, *args, stream_k=True))


@pytest.mark.parametrize("seed", range(30))
def test_stream_k_invariants(tg, seed):
    rng = np.random.default_rng(1000 + seed)
    M, N, K = (int(x) for x in rng.integers(1, 30000, 3))
    sms = int(rng.choice([8, 64, 148, 152]))
    c = cfg_sk(tg, M, N, K, BF16, 0, 1, sms=sms)
    workers = c["grid"] // 2 if c["pair"] else c["grid"]
    kb = -(-K // 64)
    if c["sk_tiles"]:
        assert c["sk_tiles"] <= c["tiles"] and c["tiles"] > workers and kb >= 32
        assert c["tiles"] % workers != 0
        assert c["sk_tiles"] * kb >= 2 * workers
        shortest = c["sk_tiles"] * kb // workers
        # a tile's K-range never meets more ranges than there are slots
        assert c["sk_cmax"] >= (kb - 1) // shortest + 2 or c["sk_cmax"] == workers
        assert c["ws_bytes"] >= workers * c["sk_cmax"] * c["bm"] * c["bn"] * 4
    else:
        assert c["ws_bytes"] == 0


def simulate_items(workers, dp_tiles, sk_tiles, kb):
    """The kernel's work split, restated: whole tiles w, w+workers, ... below
    dp_tiles and equal contiguous ranges of the sk_tiles*kb iterations, in the
    kernel's order: every whole tile but the last, the range, the last one."""
    iters = sk_tiles * kb
    items = {}
    for w in range(workers):
        whole = [(t, 0, kb) for t in range(w, dp_tiles, workers)]
        pieces = []
        it, end = iters * w // workers, iters * (w + 1) // workers
        while it < end:
            ts = it // kb
            k0 = it - ts * kb
            k1 = min(kb, k0 + (end - it))
            pieces.append((dp_tiles + ts, k0, k1))
            it += k1 - k0
        items[w] = whole[:-1] + pieces + whole[-1:]
    return items


@pytest.mark.parametrize("seed", range(30))
def test_stream_k_schedule_covers_every_k_block_once(tg, seed):
    rng = np.random.default_rng(2000 + seed)
    M, N, K = (int(x) for x in rng.integers(1, 20000, 3))
    sms = int(rng.choice([8, 16, 64, 152]))
    c = cfg_sk(tg, M, N, K, F16, 1, 0, sms=sms)
    workers = c["grid"] // 2 if c["pair"] else c["grid"]
    kb = -(-K // 64)
    dp = c["tiles"] - c["sk_tiles"]
    items = simulate_items(workers, dp, c["sk_tiles"], kb)
    seen = {}
    owners = {}
    for w, its in items.items():
        for t, k0, k1 in its:
            assert 0 <= k0 < k1 <= kb and 0 <= t < c["tiles"]
            for k in range(k0, k1):
                assert (t, k) not in seen
                seen[(t, k)] = w
            owners.setdefault(t, []).append(w)
    assert len(seen) == c["tiles"] * kb
    for w, its in items.items():  # a worker holding whole tiles ends on one
        if any(k1 - k0 == kb and t < dp for t, k0, k1 in its):
            assert its[-1][0] < dp
    first_owners = set()
    for t, ws in owners.items():
        assert ws == sorted(ws) and ws == list(range(ws[0], ws[0] + len(ws)))
        if len(ws) > 1:  # a split tile: its slots and counter are indexed by the first owner
            assert len(ws) <= c["sk_cmax"]
            assert ws[0] not in first_owners
            first_owners.add(ws[0])
