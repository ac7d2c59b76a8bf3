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
    assert c["stages"] >= 4 and 1 <= c["group_m"] <= 8
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
