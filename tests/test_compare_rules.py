"""The parity comparators themselves (CPU): the selection rule must reject a GPU selection
that drops a forced block (sink block 0, the query's local block) even when the block kept in
its place scores higher, or that breaks the list layout (ids ascending, then -1 padding), and
accept a near-tie swap of two non-forced blocks."""
import numpy as np
import pytest

from _compare import check_selection


def _case():
    # one row, one group, 6 blocks: 4 causal (local block 3), k 3
    s = np.full((1, 1, 6), -np.inf)
    s[0, 0, :4] = [1.0, 5.0, 5.0, 0.5]
    ids_ref = np.array([[[0, 1, 3]]], dtype=np.int32)
    return s, ids_ref


def test_same_selection_passes():
    s, ids_ref = _case()
    assert check_selection(ids_ref.copy(), ids_ref, s) == 0


def test_near_tie_swap_passes():
    s, ids_ref = _case()
    # blocks 1 and 2 tie exactly: keeping 2 instead of 1 is a near-tie swap
    assert check_selection(np.array([[[0, 2, 3]]], dtype=np.int32), ids_ref, s) == 1


@pytest.mark.parametrize("gpu,what", [([0, 1, 2], "local block"), ([1, 2, 3], "sink block 0")])
def test_dropped_forced_block_fails(gpu, what):
    s, ids_ref = _case()
    with pytest.raises(AssertionError, match=what):
        check_selection(np.array([gpu], dtype=np.int32)[None], ids_ref, s)


def test_clear_loss_fails():
    s, ids_ref = _case()
    s[0, 0, 2] = 4.0  # block 2 now clearly below block 1
    with pytest.raises(AssertionError, match="chose block 2"):
        check_selection(np.array([[[0, 2, 3]]], dtype=np.int32), ids_ref, s)


def _padded_case():
    # one row, one group, 3 causal blocks (local block 2) and k 4: one slot of padding
    s = np.full((1, 1, 6), -np.inf)
    s[0, 0, :3] = [1.0, 2.0, 0.5]
    return s, np.array([[[0, 1, 2, -1]]], dtype=np.int32)


@pytest.mark.parametrize("gpu", [[0, -1, 1, 2],    # padding inside the list
                                 [0, 1, 2, -2],    # padding other than -1
                                 [0, 2, 1, -1],    # ids not ascending
                                 [0, 1, 1, 2]])    # a repeated id in place of the padding
def test_broken_list_layout_fails(gpu):
    s, ids_ref = _padded_case()
    with pytest.raises(AssertionError):
        check_selection(np.array([gpu], dtype=np.int32)[None], ids_ref, s)
