"""Oracle pins: the split-KV planners (CPU only)."""

import numpy as np
import pytest

from oracle import plan as op
from oracle_pins import load_golden


def test_dynamic_plan_hand_example():
    g = load_golden("plan_hand_example.json")["dynamic"]
    items, cta_ptr, seg_ptr, home_end, pool = op.plan_dynamic(g["seq_lens"], g["num_ctas"],
                                                              g["min_tiles"])
    assert [list(i) for i in items] == g["items"]
    assert cta_ptr == g["cta_ptr"]
    assert seg_ptr == g["seg_ptr"]
    assert home_end == cta_ptr[1:] and pool == [], "no pool without pool chunks"


def test_dynamic_plan_with_pool_hand_example():
    g = load_golden("plan_hand_example.json")["dynamic_pool"]
    items, cta_ptr, seg_ptr, home_end, pool = op.plan_dynamic(
        g["seq_lens"], g["num_ctas"], g["min_tiles"], g["pool_chunks"])
    assert [list(i) for i in items] == g["items"]
    assert cta_ptr == g["cta_ptr"] and seg_ptr == g["seg_ptr"]
    assert home_end == g["home_end"] and pool == g["pool"]


def test_static_plan_hand_example():
    g = load_golden("plan_hand_example.json")["static"]
    items, cta_ptr, seg_ptr, num_ctas = op.plan_static(g["seq_lens"], g["splits"])
    assert [list(i) for i in items] == g["items"]
    assert num_ctas == g["num_ctas"]
    assert seg_ptr == g["seg_ptr"]
    assert cta_ptr == [min(c, len(items)) for c in range(num_ctas + 1)]


def _length_mixes(rng):
    yield [1, 63, 64, 300]
    yield [4096] * 32
    yield [131072] + [4096] * 31
    yield [0, 5, 0, 64 * 7 + 1]
    yield [0, 0, 0]
    yield list(rng.integers(1, 5000, size=50))
    yield list(np.exp(rng.uniform(np.log(128), np.log(262144), 64)).astype(int))


@pytest.mark.parametrize("J,kmin", [(0, 1), (1, 1), (6, 1), (4, 2), (4, 16)])
@pytest.mark.parametrize("C", [1, 7, 152, 304, 1000])
def test_dynamic_plan_covers_and_balances(C, J, kmin):
    rng = np.random.default_rng(C)
    for lens in _length_mixes(rng):
        for min_tiles in (1, 4):
            items, cta_ptr, seg_ptr, home_end, pool = op.plan_dynamic(lens, C, min_tiles, J, kmin)
            n = op.check_coverage(lens, items, cta_ptr, seg_ptr, home_end, pool)
            B = len(lens)
            assert n <= C * (1 + J) + 8 * B, "capacity bound"
            T = 8 * sum(op.num_tiles(L) for L in lens)
            q = max(min_tiles, -(-T // C)) if T else min_tiles
            ns = [op.num_tiles(L) for L in lens]
            if ns and ns[0] > 0 and len(set(ns)) == 1 and 8 * B <= C:
                q = max(q, ns[0])             # equal lengths: whole segments
            per_cta = [sum(items[i][3] - items[i][2] for i in range(cta_ptr[c], cta_ptr[c + 1]))
                       for c in range(C)]
            assert sum(per_cta) == T
            # every unit gets exactly q tiles except the tail ones
            full = T // q
            assert per_cta[:full] == [q] * full
            assert all(x == 0 for x in per_cta[full + 1:])


@pytest.mark.parametrize("S", [1, 2, 3, 64])
def test_static_plan_covers(S):
    rng = np.random.default_rng(S)
    for lens in _length_mixes(rng):
        items, cta_ptr, seg_ptr, C = op.plan_static(lens, S)
        op.check_coverage(lens, items, cta_ptr, seg_ptr)
        assert len(items) <= C
        # every segment's chunks differ in size by at most one chunk remainder
        for s in range(len(lens) * 8):
            sizes = [items[i][3] - items[i][2] for i in range(seg_ptr[s], seg_ptr[s + 1])]
            assert len(sizes) <= S
            if sizes:
                assert all(x == sizes[0] for x in sizes[:-1]) and sizes[-1] <= sizes[0]


def test_tiles_of_ragged_lengths():
    assert [op.num_tiles(L) for L in (0, 1, 63, 64, 65, 128, 129)] == [0, 1, 1, 1, 2, 2, 3]


def test_pool_min_chunk_hand_example():
    """seq_lens [700], C = 2, J = 2: P = 5 pooled tiles in chunks of 3.  With
    the smallest worthwhile chunk at 3 the pool stays (the golden plan); at 4
    the chunks are too short and the plan is the plain one."""
    g = load_golden("plan_hand_example.json")
    with_pool = op.plan_dynamic([700], 2, 1, 2, 3)
    assert [list(i) for i in with_pool[0]] == g["dynamic_pool"]["items"]
    assert with_pool[4] == g["dynamic_pool"]["pool"]
    items, cta_ptr, seg_ptr, home_end, pool = op.plan_dynamic([700], 2, 1, 2, 4)
    plain = op.plan_dynamic([700], 2, 1, 0)
    assert items == plain[0] and cta_ptr == plain[1] and pool == [] and home_end == cta_ptr[1:]
    # by hand: q = 44, so the plain plan cuts segment 3 ([33,44)) and 7 only at 44
    assert items[3] == (0, 3, 0, 11) and len(items) == 8


def test_equal_lengths_get_whole_segments():
    """Equal lengths with no more segments than units: every segment is one
    item and unit c runs segment c (the proportional quota would have split
    each of them); one tile more anywhere restores the proportional split."""
    lens = [4096] * 32                                   # 256 segments of 64 tiles
    items, cta_ptr, seg_ptr, home_end, pool = op.plan_dynamic(lens, 304)
    assert len(items) == 256 and seg_ptr == list(range(257))
    assert cta_ptr == list(range(257)) + [256] * 48
    assert all(it[2] == 0 and it[3] == 64 for it in items)
    op.check_coverage(lens, items, cta_ptr, seg_ptr, home_end, pool)
    # more segments than units, or one unequal length: the plain quota (54)
    items2, cta2, _, _, _ = op.plan_dynamic(lens, 200)
    assert cta2[1] - cta2[0] >= 1 and any(it[3] - it[2] < 64 for it in items2)
    items3, _, _, _, _ = op.plan_dynamic([4096] * 31 + [4097], 304)
    assert any(it[3] - it[2] < 64 for it in items3)
