"""The split planner (oscar_decode_plan_splits, host arithmetic only) against
sweeps of the split count on GB300 (152 SMs, 4 decode CTAs per SM for INT2),
with L2 flushed between repetitions where the shape fits in it.  The counts are the kernel's tuning, not the method's
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


# (rows = B * Hkv, 32-token blocks, CTAs per SM) -> (planned count, decode us
# at that count, fastest swept count and its us), from sweeps of the split
# count on GB300 with the INT2 kernel; L2 flushed for the shapes that fit in
# it.  The planner's model was fitted to these sweeps.
MEASURED = {
    "batch 48 x 128K, 32/8 heads": ((384, 4092, 4), 11, 970.0, 13, 969.0),
    "batch 48 x 112K": ((384, 3584, 4), 11, 853.0, 13, 852.6),
    "batch 48 x 96K": ((384, 3072, 4), 11, 736.0, 11, 736.0),
    "batch 48 x 80K": ((384, 2560, 4), 11, 618.7, 9, 618.1),
    "batch 48 x 64K": ((384, 2048, 4), 11, 501.8, 9, 500.4),
    "batch 48 x 32K": ((384, 1024, 4), 3, 270.5, 7, 264.7),
    "batch 48 x 16K": ((384, 512, 4), 3, 144.4, 5, 143.4),
    "batch 32 x 32K": ((256, 1024, 4), 7, 181.9, 7, 181.9),
    "batch 24 x 128K": ((192, 4096, 4), 19, 498.6, 15, 494.6),
    "batch 16 x 64K, 32/8 heads": ((128, 2048, 4), 14, 180.0, 13, 178.1),
    "batch 12 x 128K": ((96, 4096, 4), 19, 257.1, 19, 257.1),
    "batch 8 x 128K": ((64, 4096, 4), 19, 177.5, 19, 177.5),
    "batch 8 x 32K, 32/8 heads": ((64, 1020, 4), 9, 54.9, 9, 54.9),
    "batch 16 x 64K, 32/4 heads (8-head groups)": ((64, 2044, 4), 19, 140.7, 19, 140.7),
    "batch 4 x 64K": ((32, 2048, 4), 19, 54.8, 19, 54.8),
    "batch 2 x 128K": ((16, 4096, 4), 37, 54.8, 37, 54.8),
    "batch 1 x 128K, 32/8 heads": ((8, 4092, 4), 37, 34.8, 37, 34.8),
    "batch 1 x 16K, 32/8 heads": ((8, 512, 4), 37, 14.6, 37, 14.6),
    "batch 1 x 4K, 32/8 heads": ((8, 128, 4), 16, 10.4, 8, 10.4),
}
# planned counts pinned from earlier sweeps of the same kernel
EARLIER = {
    "batch 1 x 1K, 1/1 heads": ((1, 31, 4), 3),        # 1-8 swept (3 and 5 best)
    "batch 8 x 4K, 32/8 heads": ((64, 124, 4), 6),     # 1-6 swept (3 and 6 best)
    "batch 48 x 128K after 1280 steps": ((384, 4132, 4), 11),
}


@pytest.mark.parametrize("name", sorted(MEASURED))
def test_planned_count_is_near_the_measured_best(plan, name):
    args, want, us, _, best_us = MEASURED[name]
    assert plan(*args, 152) == want
    assert us <= 1.025 * best_us          # the sweep: within 2.5 % of the fastest count


@pytest.mark.parametrize("name", sorted(EARLIER))
def test_planned_count_of_earlier_sweeps(plan, name):
    args, want = EARLIER[name]
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
