"""Pins of the oracle's receiver-driven credit FIFO (posts and completions)."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import Deadlock, PostedChannel, PostedReceiver, PostedSender, ProtocolViolation, System, explore

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bytes(n, seed=0):
    return np.random.default_rng(seed).integers(0, 256, n, dtype=np.uint8)


@pytest.mark.parametrize("n", [1, 16, 1000, 4096, 10007])
@pytest.mark.parametrize("nchan,nslots", [(1, 1), (3, 2), (4, 8)])
def test_posted_identity(n, nchan, nslots):
    src = _bytes(n, n)
    dst, chans, _ = oracle.posted_transfer(src, nchan, nslots, 512, seed=n + nslots)
    assert np.array_equal(dst, src)
    for c in chans:
        assert c.posted == c.completed and c.max_outstanding <= c.N


def test_posted_repeated_operations():
    chans = None
    for i in range(4):
        src = _bytes(2000 + 37 * i, i)
        dst, chans, _ = oracle.posted_transfer(src, 2, 2, 256, seed=i, chans=chans)
        assert np.array_equal(dst, src)


def test_first_post_index_golden():
    g = json.load(open(os.path.join(GOLD, "counters_init.json")))
    c = PostedChannel(4, 16)
    dst = np.zeros(16, np.uint8)
    r = PostedReceiver(c, dst, 0, 16)
    r.fire(("post",))
    assert c.posts[0].idx == g["first_posted_index"] and c.completed == g["initial_head"]


def _system(n, nslots, chunk, send_fault=None, recv_fault=None):
    c = PostedChannel(nslots, chunk)
    src = np.arange(1, n + 1, dtype=np.uint8)
    dst = np.zeros(n, np.uint8)
    return lambda: System([PostedSender(c, src, 0, n, fault=send_fault),
                           PostedReceiver(c, dst, 0, n, fault=recv_fault)], [c], [dst])


def _final(s):
    d = s.buffers[0]
    assert np.array_equal(d, np.arange(1, len(d) + 1, dtype=np.uint8))


@pytest.mark.parametrize("nslots,n", [(1, 2), (1, 6), (2, 6), (2, 8)])
def test_posted_exhaustive(nslots, n):
    assert explore(_system(n, nslots, 2), _final) > 1


def test_overposting_receiver_is_caught():
    with pytest.raises(ProtocolViolation):
        explore(_system(8, 1, 2, recv_fault="overpost"), _final)


def test_sender_ignoring_the_index_is_caught():
    # a stale post from the previous operation sits in the slot
    c = PostedChannel(2, 2)
    src = np.arange(1, 5, dtype=np.uint8)
    d1 = np.zeros(4, np.uint8)
    oracle.run(System([PostedSender(c, src, 0, 4), PostedReceiver(c, d1, 0, 4)], [c], [d1]))
    d2 = np.zeros(4, np.uint8)
    with pytest.raises((ProtocolViolation, Deadlock)):
        oracle.run(System([PostedSender(c, src, 0, 4, fault="ignore_idx"), PostedReceiver(c, d2, 0, 4)], [c], [d2]),
                   seed=1)
