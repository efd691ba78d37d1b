"""The comparison helpers of the GPU parity tests, on the CPU: the per-row
error and the choice of segment-edge rows that the sampled tests add."""
import numpy as np
import pytest

from _parity import check_rows, edge_tokens, row_rel_l2, segment_edge_rows


def test_row_rel_l2_per_row_and_zero_rows():
    b = np.array([[3.0, 4.0], [0.0, 0.0], [1.0, 0.0]])
    a = np.array([[3.0, 4.5], [0.0, 0.0], [1.0, 0.0]])
    e = row_rel_l2(a, b)
    assert e[0] == pytest.approx(0.1) and e[1] == 0.0 and e[2] == 0.0
    a[1, 0] = 1e-30  # a zero reference row must be matched exactly
    assert np.isinf(row_rel_l2(a, b)[1])


def test_check_rows_catches_one_bad_row_the_whole_matrix_norm_hides():
    rng = np.random.default_rng(0)
    b = rng.standard_normal((4096, 64))
    a = b * (1 + 1e-3 * rng.standard_normal(b.shape))
    a[4000] *= 1.2  # one row 20 % off
    whole = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert whole < 1e-2  # the whole-matrix bound would pass
    with pytest.raises(AssertionError, match="row 4000"):
        check_rows("out", a, b, 1e-2)


def test_segment_edge_rows_hand_example():
    # expert 0: 300 rows [0, 300); expert 1: empty; expert 2: 40 rows [300, 340)
    rows = set(segment_edge_rows([0, 300, 300, 340], head=2, tail=4).tolist())
    want = {0, 1, 296, 297, 298, 299,           # expert 0: head, tail
            256, 288,                           # last 128-row tile starts at 256: groups at 256, 288
            300, 301, 336, 337, 338, 339,       # expert 2: head, tail
            }
    # expert 0's last 256-row tile starts at 256 as well; expert 2's tiles start at 300
    want |= {256, 288, 300, 332}
    assert rows == want


def test_edge_tokens_maps_rows_back_to_tokens():
    # 6 tokens, top-2 over 3 experts; offsets from counts [4, 5, 3]
    idx = np.array([[0, 1], [1, 2], [0, 1], [2, 1], [0, 1], [0, 2]])
    pos = np.array([[0, 0], [1, 0], [1, 2], [1, 3], [2, 4], [3, 2]])
    offsets = np.array([0, 4, 9, 12])
    toks = edge_tokens(idx, pos, offsets, head=1, tail=1)
    # first/last rows: expert 0 rows 0 (t0) and 3 (t5); expert 1 rows 4 (t0 r1) and 8 (t4 r1);
    # expert 2 rows 9 (t1 r1) and 11 (t5 r1); plus 32-row group starts = the segment starts
    assert toks == [0, 1, 4, 5]
    pos2 = pos.copy()
    pos2[0, 0] = -1  # a dropped assignment never selects its token
    pos2[0, 1] = -1
    assert 0 not in edge_tokens(idx, pos2, offsets, head=1, tail=1)
