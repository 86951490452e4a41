"""Pins of the oracle's SIMPLE FIFO state machines and channel partition."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import (Deadlock, ProtocolViolation, SimpleFifo, SimpleReceiver, SimpleSender, System,
                    channel_byte_ranges, explore, slot_steps)

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bytes(n, seed=0):
    return np.random.default_rng(seed).integers(0, 256, n, dtype=np.uint8)


@pytest.mark.parametrize("n", [0, 1, 15, 16, 17, 4095, 4096, 4097, 65536 + 3])
@pytest.mark.parametrize("nchan", [1, 3, 8])
def test_simple_identity(n, nchan):
    src = _bytes(n, n)
    dst, fifos, _ = oracle.simple_transfer(src, nchan, 2, 1024, seed=n + nchan)
    assert np.array_equal(dst, src)
    for f in fifos:
        assert f.head == f.tail
        assert f.max_occupancy <= f.N


def test_simple_result_independent_of_interleaving():
    src = _bytes(20000, 7)
    outs = [oracle.simple_transfer(src, 2, 3, 1000, seed=s)[0] for s in range(6)]
    for o in outs:
        assert np.array_equal(o, src)


def test_simple_occupancy_reaches_depth():
    # with a slow receiver some schedules fill the whole FIFO, never more
    src = _bytes(64 * 40, 1)
    seen = set()
    for s in range(20):
        _, fifos, _ = oracle.simple_transfer(src, 1, 4, 64, seed=s)
        seen.add(fifos[0].max_occupancy)
    assert max(seen) == 4


def test_counters_continue_across_operations():
    src1, src2 = _bytes(5000, 1), _bytes(7001, 2)
    d1, fifos, _ = oracle.simple_transfer(src1, 2, 2, 512, seed=1)
    steps1 = [f.tail for f in fifos]
    d2, fifos, _ = oracle.simple_transfer(src2, 2, 2, 512, seed=2, fifos=fifos)
    assert np.array_equal(d1, src1) and np.array_equal(d2, src2)
    for (lo, hi), f, s1 in zip(channel_byte_ranges(len(src2), 2), fifos, steps1):
        assert f.tail == f.head == s1 + len(slot_steps(hi - lo, 512))


def _simple_system(n, nslots, slot_bytes, send_fault=None, recv_fault=None):
    src = np.arange(1, n + 1, dtype=np.uint8)
    dst = np.zeros(n, np.uint8)
    f = SimpleFifo(nslots, slot_bytes)
    return lambda: System([SimpleSender(f, src, 0, n, fault=send_fault),
                           SimpleReceiver(f, dst, 0, n, fault=recv_fault)], [f], [dst])


def _final_identity(s):
    dst = s.buffers[0]
    assert np.array_equal(dst, np.arange(1, len(dst) + 1, dtype=np.uint8))


@pytest.mark.parametrize("nslots", [1, 2])
@pytest.mark.parametrize("n", [1, 2, 3, 5, 8])
def test_simple_exhaustive(nslots, n):
    # slot of 2 bytes: up to 4 slot-steps; every interleaving keeps the
    # invariants and ends with dst == src
    nstates = explore(_simple_system(n, nslots, 2), _final_identity)
    assert nstates > 1


@pytest.mark.parametrize("fault", ["skip_credit", "tail_before_fill"])
def test_planted_sender_mistakes_are_caught(fault):
    with pytest.raises(ProtocolViolation):
        explore(_simple_system(8, 1, 2, send_fault=fault), _final_identity)


@pytest.mark.parametrize("fault", ["head_before_copy", "skip_tail_wait"])
def test_planted_receiver_mistakes_are_caught(fault):
    with pytest.raises(ProtocolViolation):
        explore(_simple_system(8, 2, 2, recv_fault=fault), _final_identity)


def test_dropped_tail_is_a_deadlock():
    with pytest.raises(Deadlock):
        oracle.run(_simple_system(8, 2, 2, send_fault="skip_tail")(), seed=0)


def test_channel_partition_rule():
    for n in [0, 1, 17, 1000, 1 << 20, (1 << 20) + 5]:
        for c in [1, 2, 3, 16]:
            r = channel_byte_ranges(n, c)
            assert len(r) == c
            assert r[0][0] == 0 and r[-1][1] == n
            for (a, b), (a2, _) in zip(r, r[1:]):
                assert b == a2 and b >= a and (a % 16 == 0 or a == b == n)
    # the bandwidth workloads: 1 GiB over 16 channels of 512 KiB slots, and
    # 256 MiB over 8 channels of 1 MiB slots
    r = channel_byte_ranges(1 << 30, 16)
    assert all(hi - lo == 64 << 20 for lo, hi in r)
    assert len(slot_steps(64 << 20, 512 << 10)) == 128
    r = channel_byte_ranges(256 << 20, 8)
    assert all(hi - lo == 32 << 20 for lo, hi in r)
    assert len(slot_steps(32 << 20, 1 << 20)) == 32


def test_geometry_golden():
    g = json.load(open(os.path.join(GOLD, "geometry.json")))
    assert g["simple_buffer_bytes"] // g["nccl_steps"] == g["step_bytes"]
    # the oracle runs the pages' geometry unchanged: 8 slots of 512 KiB
    src = _bytes(3 * g["simple_buffer_bytes"] + 11, 3)
    dst, fifos, _ = oracle.simple_transfer(src, 1, g["nccl_steps"], g["step_bytes"], seed=4)
    assert np.array_equal(dst, src)
    assert fifos[0].tail == len(slot_steps(len(src), g["step_bytes"]))


def test_counter_initial_values_golden():
    g = json.load(open(os.path.join(GOLD, "counters_init.json")))
    f = SimpleFifo(8, 64)
    assert f.head == g["initial_head"] and f.tail == g["initial_head"]
    assert all(s == g["size_word_init"] for s in f.size)
