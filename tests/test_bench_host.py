"""Host-side logic of the bench: the end-to-end leg's row chunks."""
import pytest

import bench


@pytest.mark.parametrize("R", [1, 3, 7, 128, 1000])
@pytest.mark.parametrize("weights", [None, "", "3,3,2,1", "1", "5,4,2,1", "1,1,1,1,1,1,1,1,1"])
def test_chunk_bounds_cover_the_rows(R, weights):
    b = bench._chunk_bounds(R, 4, weights)
    assert b[0][0] == 0 and b[-1][1] == R
    assert all(lo < hi for lo, hi in b)
    assert all(b[k][1] == b[k + 1][0] for k in range(len(b) - 1))
    n_w = len([x for x in weights.split(",")]) if weights else min(4, R)
    assert len(b) == min(n_w, R)


def test_chunk_bounds_follow_the_weights():
    assert [hi - lo for lo, hi in bench._chunk_bounds(128, 4, "3,3,2,1")] == [43, 42, 29, 14]
    assert [hi - lo for lo, hi in bench._chunk_bounds(128, 4, None)] == [32] * 4
    assert [hi - lo for lo, hi in bench._chunk_bounds(9, 2, "1,2")] == [3, 6]
    with pytest.raises(ValueError):
        bench._chunk_bounds(8, 4, "1,0,1")
