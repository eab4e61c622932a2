"""The fp64 oracle against its pins (CPU only).

Every pin in ``_pins.py`` checks the oracle against something other than
itself: 60-digit brute force on tiny inputs, integer cases that numpy's
integer matmul computes exactly, closed forms (one token, two tokens, equal
keys, zero scale, a dominant key), invariants (rows sum to one, permutation,
shift, linearity, split == unsplit) and the page's shape table.
"""
import pytest

import _pins  # noqa: E402  (tests/ is on sys.path via pytest rootdir insertion)


@pytest.mark.parametrize("pin", _pins.PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_bad_arguments_rejected(orc):
    import numpy as np

    q = np.zeros((1, 3, 128), np.uint16)
    k = np.zeros((1, 2, 4, 128), np.uint16)  # 3 query heads over 2 KV heads: not a GQA layout
    with pytest.raises(ValueError):
        orc.attention(q, k, k, np.array([4], np.int32), 1.0)
    k = np.zeros((1, 1, 4, 128), np.uint16)
    with pytest.raises(ValueError):
        orc.attention(q, k, k, np.array([5], np.int32), 1.0)  # longer than the cache


def test_threads_reported(orc):
    assert orc.num_threads() >= 1
