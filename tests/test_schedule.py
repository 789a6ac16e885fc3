"""Pins of the oracle's tile-grid and program-order arithmetic (CPU only)."""
import itertools

import pytest

from oracle import schedule


def test_program_order_4x4(golden):
    g = golden("program_order_4x4.txt")
    assert schedule.order_layout(4, 4, None) == g["ROW_MAJOR"]
    assert schedule.order_layout(4, 4, 2) == g["GROUP_MAJOR_G2"]


def test_grid_cases(golden):
    for row in golden("grid_cases.txt")["CASES"]:
        M, K, N, bm, bn, bk, gm, gn, kr, prods, mr, mc, mk = row
        assert schedule.grid_2d(M, N, bm, bn) == (gm, gn)
        if kr is not None:
            assert schedule.k_rounds(K, bk) == kr
        if prods is not None:
            assert gm * gn * schedule.k_rounds(K, bk) == prods
        if mr is not None:
            assert schedule.out_of_range(M, bm) == mr
        if mc is not None:
            assert schedule.out_of_range(N, bn) == mc
        if mk is not None:
            assert schedule.out_of_range(K, bk) == mk
    assert schedule.grid_2d(1023, 1023, 64, 64)[0] * schedule.grid_2d(1023, 1023, 64, 64)[1] == 256


@pytest.mark.parametrize("bm,bn,g", list(itertools.product([1, 2, 3, 5, 8, 13], [1, 3, 4, 7], [1, 2, 3, 8])))
def test_group_major_is_a_bijection(bm, bn, g):
    seen = set()
    for pid in range(bm * bn):
        r, c = schedule.group_major_tile(pid, bm, bn, g)
        assert 0 <= r < bm and 0 <= c < bn
        seen.add((r, c))
    assert len(seen) == bm * bn


def test_group_major_partial_last_group():
    """5 tile rows, GROUP 2: strips {0,1}, {2,3}, {4} (the min() of Step 4)."""
    lay = schedule.order_layout(5, 3, 2)
    assert [lay[r][0] for r in range(5)] == [0, 1, 6, 7, 12]
    assert lay[4] == [12, 13, 14]


def test_group_one_is_column_major_within_strip_of_one_row():
    """GROUP 1 degenerates to row-major order."""
    assert schedule.order_layout(3, 4, 1) == schedule.order_layout(3, 4, None)
