"""Pins for the CP layout oracle (CPU only): the ranks' local streams
partition the tokens, each rank holds the same number of tokens of every
segment, and a small case written out by hand from the load-balanced rule
(rank r holds chunks r and 2*cp-1-r of each segment)."""
import numpy as np
import pytest

from oracle import cp_local_mask, cp_local_to_global


@pytest.mark.parametrize("cp", [1, 2, 4, 8])
def test_ranks_partition_the_tokens(cp):
    rng = np.random.default_rng(cp)
    lens = rng.integers(1, 9, size=7) * 2 * cp
    offs = np.concatenate([[0], np.cumsum(lens)])
    T = int(offs[-1])
    allg = np.concatenate([cp_local_to_global(offs, cp, r) for r in range(cp)])
    assert sorted(allg.tolist()) == list(range(T))
    for r in range(cp):
        loc = cp_local_to_global(offs, cp, r)
        assert len(loc) == T // cp
        # the rank's share of each segment is L / cp tokens
        seg = np.searchsorted(offs, loc, side="right") - 1
        np.testing.assert_array_equal(np.bincount(seg, minlength=len(lens)), lens // cp)


def test_hand_written_case():
    # two segments: [0, 8) and [8, 16); cp = 2 -> chunks of 2 tokens
    offs = [0, 8, 16]
    assert cp_local_to_global(offs, 2, 0).tolist() == [0, 1, 6, 7, 8, 9, 14, 15]
    assert cp_local_to_global(offs, 2, 1).tolist() == [2, 3, 4, 5, 10, 11, 12, 13]
    mask = np.arange(16) % 3 == 0
    assert cp_local_mask(mask, offs, 2, 1).tolist() == [False, True, False, False,
                                                        False, False, True, False]
    assert cp_local_to_global(offs, 1, 0).tolist() == list(range(16))


def test_rejects_segments_not_divisible():
    with pytest.raises(ValueError):
        cp_local_to_global([0, 6], 2, 0)
