"""Pins of the oracle's zero-copy (ptrExchange) state machines."""
import numpy as np
import pytest

import oracle
from oracle import (Deadlock, ProtocolViolation, System, ZeroCopyChannel, ZeroCopyReceiver,
                    ZeroCopySender, explore)


def _bytes(n, seed=0):
    return np.random.default_rng(seed).integers(0, 256, n, dtype=np.uint8)


@pytest.mark.parametrize("n", [1, 16, 100, 4096, 10000])
@pytest.mark.parametrize("nchan", [1, 4])
def test_zero_copy_identity_and_slots_untouched(n, nchan):
    src = _bytes(n, n)
    dst, chans, _ = oracle.zero_copy_transfer(src, nchan, 2, 512, seed=n)
    assert np.array_equal(dst, src)
    for c in chans:
        assert (c.slots == 0xA5).all()
        assert c.ptr_exchange is None and c.head == c.tail


def test_zero_copy_repeated_operations():
    chans = None
    for i in range(4):
        src = _bytes(3000 + 17 * i, i)
        dst, chans, _ = oracle.zero_copy_transfer(src, 2, 2, 256, seed=i, chans=chans)
        assert np.array_equal(dst, src)


def _zc_system(n, nslots, chunk):
    c = ZeroCopyChannel(nslots, chunk)
    src = np.arange(1, n + 1, dtype=np.uint8)
    dst = np.zeros(n, np.uint8)
    return lambda: System([ZeroCopySender(c, src, 0, n), ZeroCopyReceiver(c, dst, 0, n)], [c], [dst])


def _zc_final(s):
    d = s.buffers[0]
    assert np.array_equal(d, np.arange(1, len(d) + 1, dtype=np.uint8))


@pytest.mark.parametrize("nslots,n", [(1, 1), (1, 4), (2, 4), (2, 6)])
def test_zero_copy_exhaustive(nslots, n):
    assert explore(_zc_system(n, nslots, 2), _zc_final) > 1


def test_zero_copy_not_cleared_is_caught():
    # the first op leaves its address in ptrExchange; in the next op the
    # receiver can never post and the sender consumes the stale address
    c = ZeroCopyChannel(2, 2)
    src, dst = np.arange(1, 5, dtype=np.uint8), np.zeros(4, np.uint8)
    oracle.run(System([ZeroCopySender(c, src, 0, 4, fault="no_clear"), ZeroCopyReceiver(c, dst, 0, 4)], [c], [dst]))
    assert np.array_equal(dst, src) and c.ptr_exchange is not None
    dst2 = np.zeros(4, np.uint8)
    with pytest.raises((ProtocolViolation, Deadlock)):
        oracle.run(System([ZeroCopySender(c, src, 0, 4), ZeroCopyReceiver(c, dst2, 0, 4)], [c], [dst2]), seed=3)
