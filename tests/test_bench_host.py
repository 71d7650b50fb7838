"""Host-side plan logic of bench.py (no GPU): the chunk plans of the end-to-end rounds."""
import pytest

import bench


@pytest.mark.parametrize("S", [1, 2, 3, 5, 16, 17, 64])
@pytest.mark.parametrize("split", ["pairs", "ramp", ""])
def test_chunk_plans_cover_every_sequence_once(split, S):
    sizes = bench.e2e_chunk_sizes(split, S, 4)
    assert sum(sizes) == S and min(sizes) >= 1


def test_pairs_plan():
    assert bench.e2e_chunk_sizes("pairs", 16) == [1, 1, 2, 2, 2, 2, 2, 2, 2]
    assert bench.e2e_chunk_sizes("pairs", 5) == [1, 1, 2, 1]
    assert bench.e2e_chunk_sizes("pairs", 1) == [1]


def test_ramp_plan_folds_a_small_tail():
    assert bench.e2e_chunk_sizes("ramp", 16) == [1, 1, 2, 3, 4, 5]
    # 1, 1, 2, 3, 4, 5, 1 -> the last 1 folds into the 5
    assert bench.e2e_chunk_sizes("ramp", 17) == [1, 1, 2, 3, 4, 6]


def test_explicit_and_equal_plans():
    assert bench.e2e_chunk_sizes("4,4,4,4", 16) == [4, 4, 4, 4]
    assert bench.e2e_chunk_sizes("", 16, 4) == [4, 4, 4, 4]
    assert bench.e2e_chunk_sizes("", 15, 4) == [15]  # not a multiple: one chunk
    with pytest.raises(SystemExit):
        bench.e2e_chunk_sizes("4,4,4", 16)
    with pytest.raises(SystemExit):
        bench.e2e_chunk_sizes("0,16", 16)
