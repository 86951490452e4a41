"""Pins of the oracle's LL128 state machines (128-byte lines: 15 payload
words and a flag word in the last 8 bytes)."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import LL128Fifo, LL128Receiver, LL128Sender, ProtocolViolation, System, explore, ll128_flag, run

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bytes(n, seed):
    return np.random.default_rng(seed).integers(0, 256, n, dtype=np.uint8)


@pytest.mark.parametrize("nbytes", [8, 112, 120, 128, 240, 248, 1000, 3840, 4096, 40000])
@pytest.mark.parametrize("nchan", [1, 3])
def test_ll128_identity(nbytes, nchan):
    src = _bytes(nbytes, nbytes)
    out, fifos, _ = oracle.ll128_transfer(src, nchan, 2, 256, seed=nbytes)
    assert np.array_equal(out.view(np.uint8), src)
    for f in fifos:
        assert f.max_occupancy <= f.N


def test_ll128_size_sweep_through_one_fifo():
    # 8 B ... 32 KiB through one FIFO of 3 x 2 lines: stale lines of earlier
    # messages (older flags, older payload) must never be read
    fifos = None
    for k in range(3, 16):
        src = _bytes(1 << k, k)
        out, fifos, _ = oracle.ll128_transfer(src, 1, 3, 256, seed=k, fifos=fifos, batch=3)
        assert np.array_equal(out.view(np.uint8), src)


def test_ll128_rejects_partial_words_and_partial_lines():
    with pytest.raises(ValueError):
        oracle.ll128_transfer(_bytes(12, 0), 1, 2, 256)
    with pytest.raises(ValueError):
        LL128Fifo(2, 192)


def test_ll128_flag_reading():
    g = json.load(open(os.path.join(GOLD, "counters_init.json")))
    assert ll128_flag(g["initial_head"]) == g["first_posted_index"]
    # a whole 8-byte flag word: no wrap at 2^32, unlike LL's 4-byte flags
    assert ll128_flag(0xFFFFFFFF) == 1 << 32 and ll128_flag(5) == 6


def test_ll128_slot_layout():
    # After a transfer, every slot holds the lines of the last step that used
    # it, laid out by the format's definition: line i of step s carries
    # payload words 15*(s*L + i) ... + 14 (zeros past the end) and s + 1 in
    # word 15.  Built here with a plain loop over steps.
    N, S = 2, 256
    L = S // 128
    nwords = 7 * 15 * L + 11                       # 7 full steps and a short one
    words = np.arange(1, nwords + 1, dtype=np.uint64) * np.uint64(0x9E3779B97F4A7C15)
    out, fifos, _ = oracle.ll128_transfer(words.view(np.uint8), 1, N, S, seed=3)
    assert np.array_equal(out, words)
    want = np.zeros((N, L, 16), np.uint64)
    nsteps = -(-nwords // (15 * L))
    for s in range(nsteps):
        for i in range(L):
            g0 = (s * L + i) * 15
            if g0 >= nwords:
                break
            for j in range(15):
                want[s % N, i, j] = words[g0 + j] if g0 + j < nwords else 0
            want[s % N, i, 15] = s + 1
    assert np.array_equal(fifos[0].lines, want)
    assert fifos[0].head == nsteps


def _ll128_system(nlines, nslots, lines_per_slot, batch=2, send_fault=None, recv_fault=None, window=2,
                  piece_words=8):
    nw = 15 * nlines - 4                           # the last line is short
    w = np.arange(1, nw + 1, dtype=np.uint64)
    out = np.zeros_like(w)
    f = LL128Fifo(nslots, 128 * lines_per_slot)
    return lambda: System([LL128Sender(f, w, 0, nw, batch=batch, window=window, piece_words=piece_words,
                                       fault=send_fault),
                           LL128Receiver(f, out, 0, nw, fault=recv_fault)], [f], [out])


def _ll128_final(s):
    out = s.buffers[0]
    assert np.array_equal(out, np.arange(1, len(out) + 1, dtype=np.uint64))


@pytest.mark.parametrize("nslots,lps,nlines,batch", [(1, 1, 1, 1), (1, 1, 3, 1), (2, 1, 3, 1), (1, 2, 4, 2),
                                                     (2, 2, 4, 2), (1, 3, 3, 3)])
def test_ll128_exhaustive(nslots, lps, nlines, batch):
    # every interleaving of payload-piece and flag visibility with the batch
    # fence, for 2-piece lines
    assert explore(_ll128_system(nlines, nslots, lps, batch=batch), _ll128_final) > 1


def test_ll128_exhaustive_fine_grained():
    # two lines in two slots, each line's payload visible in 8 pieces of at
    # most 2 words, in any order
    assert explore(_ll128_system(2, 2, 1, batch=1, window=2, piece_words=2), _ll128_final) > 1000


def test_ll128_flag_without_fence_is_caught():
    with pytest.raises(ProtocolViolation):
        explore(_ll128_system(2, 1, 1, send_fault="flag_with_data"), _ll128_final)


def test_ll128_payload_loaded_before_flag_is_caught():
    with pytest.raises(ProtocolViolation):
        explore(_ll128_system(2, 1, 1, recv_fault="data_before_flag"), _ll128_final)


def test_ll128_early_credit_is_caught():
    with pytest.raises(ProtocolViolation):
        explore(_ll128_system(3, 1, 2, recv_fault="head_early"), _ll128_final)


def test_ll128_skipped_credit_is_caught():
    with pytest.raises(ProtocolViolation):
        explore(_ll128_system(3, 1, 1, send_fault="skip_credit"), _ll128_final)


@pytest.mark.parametrize("seed", range(4))
def test_ll128_result_independent_of_interleaving(seed):
    src = _bytes(5000, 42)
    out, _, _ = oracle.ll128_transfer(src, 2, 2, 384, seed=seed, batch=1 + seed % 3, piece_words=1 + seed)
    assert np.array_equal(out.view(np.uint8), src)


# sender and receiver sides cut into different numbers of lanes (receiver
# lanes with a head each; a sender lane waits for every receiver lane its
# lines meet): the credit rule keeps every line from being overwritten before
# the receiver lane that owns it has read it, whatever the interleaving

def _lane_system(nlines, nslots, lines_per_slot, lanes, rlanes, fault=None, batch=1):
    words = np.arange(1, nlines * 15 + 1, dtype=np.uint64)

    def make():
        f = oracle.LL128LaneFifo(nslots, lines_per_slot * 128, rlanes)
        out = np.zeros_like(words)
        actors = [oracle.LL128LaneSender(f, words, 0, len(words), lanes, g, batch=batch, fault=fault)
                  for g in range(lanes)]
        actors += [oracle.LL128LaneReceiver(f, out, 0, len(words), r) for r in range(rlanes)]
        return System(actors, [f], [out])

    def final(s):
        assert np.array_equal(s.buffers[0], words)
    return make, final


@pytest.mark.parametrize("nlines,nslots,lps,lanes,rlanes", [
    (4, 1, 2, 1, 2), (4, 1, 2, 2, 1), (6, 1, 3, 1, 3), (6, 1, 3, 3, 2), (6, 1, 3, 2, 2), (6, 2, 3, 2, 3),
    (6, 2, 3, 3, 1), (9, 2, 3, 2, 2)])
def test_ll128_lanes_exhaustive(nlines, nslots, lps, lanes, rlanes):
    make, final = _lane_system(nlines, nslots, lps, lanes, rlanes)
    assert explore(make, final) > 10


@pytest.mark.parametrize("cfg", [(4, 1, 2, 1, 2), (6, 1, 3, 1, 3), (6, 1, 3, 2, 3)])
def test_ll128_lane_credit_from_one_receiver_lane_is_caught(cfg):
    # a sender lane whose lines meet two receiver lanes but that waits only
    # for the first overwrites the second's lines in some interleaving
    make, final = _lane_system(*cfg, fault="one_lane_credit")
    with pytest.raises(ProtocolViolation):
        explore(make, final)


@pytest.mark.parametrize("seed", range(6))
def test_ll128_lanes_random_interleavings(seed):
    # 8 lines a slot, 3 slots, 5 + 3 / 3 + 5 / 8 + 1 lanes, several steps
    lanes, rlanes = [(5, 3), (3, 5), (8, 1)][seed % 3]
    make, final = _lane_system(8 * 5 + 3, 3, 8, lanes, rlanes, batch=1 + seed % 2)
    s = make()
    run(s, seed=seed)
    final(s)
