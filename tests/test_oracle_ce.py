"""Pins of the oracle's proxy (copy-engine) mode: the sender kernel fills its
send ring, host proxy hops copy each slot-step to the next ring and publish
its tail after the copy, the receiver kernel drains the last ring and returns
head ("NCCL transport data transfer (二)", CE mode and shm useMemcpy mode)."""
import numpy as np
import pytest

import oracle
from oracle import CEFifo, CEProxy, CEReceiver, CESender, Deadlock, ProtocolViolation, System, explore


def _bytes(n, seed=0):
    return np.random.default_rng(seed).integers(0, 256, n, dtype=np.uint8)


@pytest.mark.parametrize("hops", [1, 2])
@pytest.mark.parametrize("n", [1, 16, 1000, 4096, 10007])
@pytest.mark.parametrize("nchan,nslots", [(1, 1), (3, 2), (4, 8)])
def test_ce_identity(n, nchan, nslots, hops):
    src = _bytes(n, n + hops)
    dst, fifos, _ = oracle.ce_transfer(src, nchan, nslots, 512, hops=hops, seed=n + nslots)
    assert np.array_equal(dst, src)
    for f in fifos:
        assert len(set(f.tails + [f.head])) == 1 and f.max_occupancy <= f.N


@pytest.mark.parametrize("hops", [1, 2])
def test_ce_counters_continue(hops):
    fifos = None
    for i in range(3):
        src = _bytes(3000 + 777 * i, i)
        dst, fifos, _ = oracle.ce_transfer(src, 2, 2, 256, hops=hops, seed=i, fifos=fifos)
        assert np.array_equal(dst, src)
    # channel 0 moved ceil(q / 256) steps per operation, q = round_up(ceil(n / 2), 16)
    want = sum(-(-(((3000 + 777 * i + 1) // 2 + 15) // 16 * 16) // 256) for i in range(3))
    assert fifos[0].head == want


def test_every_ring_holds_the_last_steps():
    # after a transfer each ring's slot k holds the last step that went
    # through it: the same bytes in every ring of the chain
    src = _bytes(5 * 64, 3)
    _, fifos, _ = oracle.ce_transfer(src, 1, 4, 64, hops=2)
    f = fifos[0]
    for r in f.rings:
        assert np.array_equal(r.slots[0], src[256:320])
        assert np.array_equal(r.slots[1:4].reshape(-1), src[64:256])


def _system(n, nslots, hops, send_fault=None, proxy_fault=None, recv_fault=None):
    f = CEFifo(nslots, 2, hops)
    src = np.arange(1, n + 1, dtype=np.uint8)
    dst = np.zeros(n, np.uint8)
    steps = -(-n // 2)
    return lambda: System([CESender(f, src, 0, n, fault=send_fault)] +
                          [CEProxy(f, h, steps, fault=proxy_fault if h == 0 else None) for h in range(hops)] +
                          [CEReceiver(f, dst, 0, n, fault=recv_fault)], [f], [dst])


def _final(s):
    d = s.buffers[0]
    if not np.array_equal(d, np.arange(1, len(d) + 1, dtype=np.uint8)):
        raise ProtocolViolation("wrong bytes delivered")


@pytest.mark.parametrize("nslots,n,hops", [(1, 2, 1), (1, 6, 1), (2, 6, 1), (2, 8, 1), (1, 4, 2), (2, 6, 2)])
def test_ce_exhaustive(nslots, n, hops):
    assert explore(_system(n, nslots, hops), _final) > 1


@pytest.mark.parametrize("kw", [dict(send_fault="skip_credit"), dict(proxy_fault="tail_before_copy"),
                                dict(recv_fault="head_before_copy")])
@pytest.mark.parametrize("hops", [1, 2])
def test_planted_mistakes_are_caught(kw, hops):
    with pytest.raises((ProtocolViolation, Deadlock)):
        explore(_system(6, 1, hops, **kw), _final)


def test_bad_size_word_is_refused():
    f = CEFifo(2, 4, 1)
    src = np.arange(1, 5, dtype=np.uint8)
    s = CESender(f, src, 0, 4)
    for _ in range(3):
        s.fire(0)
    f.size[0] = 9          # larger than a slot
    p = CEProxy(f, 0, 1)
    p.fire(0)
    with pytest.raises(ProtocolViolation):
        p.fire(0)
