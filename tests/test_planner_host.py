"""The split planner (oscar_decode_plan_splits, host arithmetic only) against
the split counts that sweeps on GB300 (152 SMs, 4 decode CTAs per SM for
INT2) measured best, with L2 flushed between
repetitions.  The counts are the kernel's tuning, not the method's
arithmetic: a change of the planner's cost model that moves one of them
must come with a new sweep.
"""
import ctypes

import pytest

from int2_kv_cache_02_gb300 import _build


@pytest.fixture(scope="module")
def plan():
    lib = ctypes.CDLL(_build.build()["liboscar.so"])
    f = lib.oscar_decode_plan_splits
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_longlong, ctypes.c_longlong, ctypes.c_int, ctypes.c_int]
    return f


# (rows = B * Hkv, 32-token blocks, CTAs per SM) -> measured-best split count
MEASURED = {
    "batch 48 x 128K, 32/8 heads": ((384, 4092, 4), 13),   # 11-17 swept; even counts slower
    "batch 48 x 128K after 1280 steps": ((384, 4132, 4), 13),
    "batch 8 x 32K, 32/8 heads": ((64, 1024, 4), 9),       # 3-10 swept
    "batch 1 x 128K, 32/8 heads": ((8, 4096, 4), 37),      # 18-113 swept
    "batch 16 x 64K, 32/4 heads": ((64, 2048, 4), 9),      # 6-12 swept
    "batch 1 x 1K, 1/1 heads": ((1, 31, 4), 3),            # 1-8 swept (3 and 5 best)
    "batch 1 x 16K, 32/8 heads": ((8, 508, 4), 37),        # 4-50 swept (16 and 37 best)
    "batch 8 x 4K, 32/8 heads": ((64, 124, 4), 3),         # 1-6 swept (3 and 6 best)
}


@pytest.mark.parametrize("name", sorted(MEASURED))
def test_planned_count_is_the_measured_best(plan, name):
    args, want = MEASURED[name]
    assert plan(*args, 152) == want


def test_counts_stay_in_range(plan):
    for rows in (1, 3, 8, 64, 384, 4096, 65536):
        for nblk in (1, 2, 31, 32, 100, 1024, 4096, 32768):
            for cps in (1, 3, 4):
                s = plan(rows, nblk, cps, 152)
                assert 1 <= s <= 512, (rows, nblk, cps, s)
                # every warp of a split keeps at least 2 blocks (one wave) or
                # 16 (more waves), unless the row is too short for 2 splits
                assert s == 1 or nblk // s >= 4 * 2, (rows, nblk, cps, s)


def test_degenerate_arguments_give_one_split(plan):
    assert plan(0, 100, 4, 152) == 1
    assert plan(8, 0, 4, 152) == 1
    assert plan(8, 100, 4, 0) == 1
    assert plan(-1, -1, -1, -1) == 1


def test_even_winner_gives_way_to_an_odd_neighbour_on_many_waves(plan):
    # many waves: batch 48 x 128K plans an odd count; the same rows with one
    # wave are not subject to the rule
    assert plan(384, 4092, 4, 152) % 2 == 1
