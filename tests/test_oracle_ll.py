"""Pins of the oracle's LL state machines (16-byte lines with two inline flags)."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import LLFifo, LLReceiver, LLSender, ProtocolViolation, System, explore, ll_flag

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _words(n, seed=1):
    return np.random.default_rng(seed).integers(0, 1 << 32, n, dtype=np.uint32)


@pytest.mark.parametrize("nbytes", [8, 16, 24, 64, 1000, 4096])
@pytest.mark.parametrize("nchan", [1, 2])
def test_ll_identity(nbytes, nchan):
    w = _words(nbytes // 4, nbytes)
    out, fifos, _ = oracle.ll_transfer(w, nchan, 2, 64, seed=nbytes)
    assert np.array_equal(out, w)
    for f in fifos:
        assert f.max_occupancy <= f.N


def test_ll_size_sweep_through_one_fifo():
    # the sweep 8 B ... 2 KiB through one FIFO: stale lines of earlier
    # messages (older flags) must never be accepted
    fifos = None
    for k in range(3, 12):
        w = _words((1 << k) // 4, k)
        out, fifos, _ = oracle.ll_transfer(w, 1, 4, 64, seed=k, fifos=fifos)
        assert np.array_equal(out, w)


def test_ll_flag_reading():
    g = json.load(open(os.path.join(GOLD, "counters_init.json")))
    # the first entry after a zero head carries index 1: zeroed memory never
    # reads as a posted line
    assert ll_flag(g["initial_head"]) == g["first_posted_index"]
    assert ll_flag(0xFFFFFFFF) == 0 and ll_flag(5) == 6


def _ll_system(nlines, nslots, lines_per_slot, send_fault=None, recv_fault=None, window=2):
    w = np.arange(1, 2 * nlines + 1, dtype=np.uint32)
    out = np.zeros_like(w)
    f = LLFifo(nslots, 16 * lines_per_slot)
    return lambda: System([LLSender(f, w, 0, len(w), window=window, fault=send_fault),
                           LLReceiver(f, out, 0, len(w), fault=recv_fault)], [f], [out])


def _ll_final(s):
    out = s.buffers[0]
    assert np.array_equal(out, np.arange(1, len(out) + 1, dtype=np.uint32))


@pytest.mark.parametrize("nslots,lps,nlines", [(1, 1, 1), (1, 1, 3), (2, 1, 4), (1, 2, 4), (2, 2, 4)])
def test_ll_exhaustive(nslots, lps, nlines):
    # every interleaving of 8-byte half-line visibility, with torn lines
    assert explore(_ll_system(nlines, nslots, lps), _ll_final) > 1


def test_ll_one_flag_receiver_is_caught():
    with pytest.raises(ProtocolViolation):
        explore(_ll_system(2, 1, 1, recv_fault="one_flag"), _ll_final)


def test_ll_early_credit_is_caught():
    with pytest.raises(ProtocolViolation):
        explore(_ll_system(3, 1, 2, recv_fault="head_early"), _ll_final)


def test_ll_skipped_credit_is_caught():
    with pytest.raises(ProtocolViolation):
        explore(_ll_system(3, 1, 1, send_fault="skip_credit"), _ll_final)


def test_ll_flags_wrap_at_32_bits():
    # step counters are 64-bit, flags (step + 1) mod 2^32: a run that starts
    # with every slot used once below the wrap crosses it intact, and the
    # step whose flag is 0 reads its own lines, not the zeroed memory
    N, S = 4, 64
    B = (1 << 32) - 2 * N - 3
    words = np.random.default_rng(7).integers(0, 2 ** 32, 1000, dtype=np.uint32)
    out, fifos, _ = oracle.ll_transfer(words, 2, N, S, seed=4, fifos=[LLFifo(N, S, step0=B) for _ in range(2)])
    assert np.array_equal(out, words)
    assert ll_flag((1 << 32) - 1) == 0 and all(f.head > (1 << 32) for f in fifos)


def test_ll_zero_flag_on_unwritten_slot_is_caught():
    # an unreachable start: the very first use of a slot expects flag 0, which
    # zeroed memory matches; the checker must refuse the stale lines
    N, S = 1, 16
    f = LLFifo(N, S, step0=(1 << 32) - 1)
    words = np.arange(1, 5, dtype=np.uint32)
    out = np.zeros_like(words)
    with pytest.raises(ProtocolViolation):
        explore(lambda: System([LLSender(f, words, 0, 4), LLReceiver(f, out, 0, 4)], [f], [out]),
                lambda s: None)
