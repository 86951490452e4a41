"""Pins of the oracle's receiver-driven credit FIFO: posts {addr, size, idx}
written by the receiver, completions {idx, size} written by the sender, in
copy mode (posts name staging slots) and direct mode (posts name dst)."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import Deadlock, PostedChannel, PostedReceiver, PostedSender, ProtocolViolation, System, explore

GOLD = os.path.join(os.path.dirname(__file__), "golden")
MODES = [False, True]


def _bytes(n, seed=0):
    return np.random.default_rng(seed).integers(0, 256, n, dtype=np.uint8)


@pytest.mark.parametrize("direct", MODES)
@pytest.mark.parametrize("n", [1, 16, 1000, 4096, 10007])
@pytest.mark.parametrize("nchan,nslots", [(1, 1), (3, 2), (4, 8)])
def test_posted_identity(n, nchan, nslots, direct):
    src = _bytes(n, n)
    dst, chans, _ = oracle.posted_transfer(src, nchan, nslots, 512, seed=n + nslots, direct=direct)
    assert np.array_equal(dst, src)
    for c in chans:
        assert c.posted == c.completed and c.max_outstanding <= c.N


@pytest.mark.parametrize("direct", MODES)
def test_posted_repeated_operations(direct):
    chans = None
    for i in range(4):
        src = _bytes(2000 + 37 * i, i)
        dst, chans, _ = oracle.posted_transfer(src, 2, 2, 256, seed=i, chans=chans, direct=direct)
        assert np.array_equal(dst, src)
    # 4 operations over channels of ceil(len/2) bytes, 256-byte chunks
    assert chans[0].completed == sum(-(-(((2000 + 37 * i + 1) // 2 + 15) // 16 * 16) // 256) for i in range(4))


def test_copy_mode_lands_in_the_slots():
    # copy mode writes the payload through the staging slots; direct mode never touches them
    src = _bytes(3 * 256, 5)
    _, chans, _ = oracle.posted_transfer(src, 1, 4, 256)
    assert np.array_equal(chans[0].slots[:3 * 256], src)
    _, chans, _ = oracle.posted_transfer(src, 1, 4, 256, direct=True)
    assert not chans[0].slots.any()


def test_first_post_index_golden():
    g = json.load(open(os.path.join(GOLD, "counters_init.json")))
    c = PostedChannel(4, 16)
    dst = np.zeros(16, np.uint8)
    r = PostedReceiver(c, dst, 0, 16)
    r.fire(("post",))
    assert c.posts[0].idx == g["first_posted_index"] and c.completed == g["initial_head"]


def _system(n, nslots, chunk, direct=False, send_fault=None, recv_fault=None):
    c = PostedChannel(nslots, chunk)
    src = np.arange(1, n + 1, dtype=np.uint8)
    dst = np.zeros(n, np.uint8)
    return lambda: System([PostedSender(c, src, 0, n, fault=send_fault),
                           PostedReceiver(c, dst, 0, n, direct=direct, fault=recv_fault)], [c], [dst])


def _final(s):
    d = s.buffers[0]
    if not np.array_equal(d, np.arange(1, len(d) + 1, dtype=np.uint8)):
        raise ProtocolViolation("wrong bytes delivered")


@pytest.mark.parametrize("direct", MODES)
@pytest.mark.parametrize("nslots,n", [(1, 2), (1, 6), (2, 6), (2, 8)])
def test_posted_exhaustive(nslots, n, direct):
    # every interleaving of 1-4 chunks of 2 bytes: invariants hold, bytes arrive
    assert explore(_system(n, nslots, 2, direct), _final) > 1


@pytest.mark.parametrize("direct", MODES)
def test_overposting_receiver_is_caught(direct):
    with pytest.raises(ProtocolViolation):
        explore(_system(8, 1, 2, direct, recv_fault="overpost"), _final)


def test_freeing_a_slot_before_copying_it_out_is_caught():
    # the sender may then overwrite the staging slot before its bytes reach dst
    with pytest.raises(ProtocolViolation):
        explore(_system(6, 1, 2, recv_fault="early_free"), _final)


@pytest.mark.parametrize("direct", MODES)
def test_sender_ignoring_the_index_is_caught(direct):
    # entries of the previous operation are still in the FIFO
    c = PostedChannel(2, 2)
    src = np.arange(1, 5, dtype=np.uint8)
    d1 = np.zeros(4, np.uint8)
    oracle.run(System([PostedSender(c, src, 0, 4), PostedReceiver(c, d1, 0, 4, direct=direct)], [c], [d1]))
    d2 = np.zeros(4, np.uint8)
    with pytest.raises((ProtocolViolation, Deadlock)):
        oracle.run(System([PostedSender(c, src, 0, 4, fault="ignore_idx"),
                           PostedReceiver(c, d2, 0, 4, direct=direct)], [c], [d2]), seed=1)


def test_oversized_chunk_is_caught():
    # a post smaller than the chunk: the sender must refuse it
    c = PostedChannel(2, 4)
    src = np.arange(1, 9, dtype=np.uint8)
    dst = np.zeros(8, np.uint8)
    r = PostedReceiver(c, dst, 0, 8, direct=True)
    r.fire(("post",))
    c.posts[0].size = 2
    s = PostedSender(c, src, 0, 8)
    s.fire(0)
    with pytest.raises(ProtocolViolation):
        s.fire(0)
