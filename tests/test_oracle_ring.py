"""Pins of the oracle's virtual ring allreduce.

The fp32 result is pinned against exact rational arithmetic with every
partial sum rounded to fp32 by an independent round-to-nearest-even
(`_f32_round`, written from the IEEE 754 definition), in an order derived by
walking the schedule's dataflow symbolically (`_chain_order`), not from the
oracle's closed form.  int32 is pinned against an int64 sum, fp32 against the
fp64 sum within (P-1) * 2**-24 * sum|x|, and P = 2 against x0 + x1.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import (explore, ring_channel_ranges, ring_chunk_elems, ring_next, ring_order_sum,
                    ring_prev, ring_rounds, ring_schedule, ring_system)
from oracle.ring import ring_chunks

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _f32_round(q: Fraction) -> Fraction:
    """Nearest fp32 value to the exact rational q, ties to even (normal range)."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    assert e > -126, "subnormal partial sum: outside the pinned range"
    ulp = Fraction(2) ** (e - 23)
    return sign * round(a / ulp) * ulp      # round() on a Fraction is half-to-even


def _chain_order(P):
    """For each chunk k, the ranks in the order their copies enter its sum,
    found by running the schedule's dataflow: rank r's i-th send is rank
    r+1's i-th receive."""
    scheds = [ring_schedule(r, P) for r in range(P)]
    pc = [0] * P
    sent = [[] for _ in range(P)]          # (chunk, contributors) carried by each send of rank r
    nrecv = [0] * P
    final = {}
    progress = True
    while progress:
        progress = False
        for r in range(P):
            if pc[r] == len(scheds[r]):
                continue
            kind, k = scheds[r][pc[r]]
            got = None
            if kind != "send":
                prev = (r - 1) % P
                if nrecv[r] >= len(sent[prev]):
                    continue
                got = sent[prev][nrecv[r]]
                nrecv[r] += 1
                assert got[0] == k, "neighbours disagree on the chunk"
            if kind == "send":
                val = (k, (r,))
            elif kind in ("recvReduceSend", "recvReduceCopySend"):
                val = (k, got[1] + (r,))
            else:
                val = got
            if kind == "recvReduceCopySend":
                final[k] = val[1]
            if kind != "recv":
                sent[r].append(val)
            pc[r] += 1
            progress = True
    assert all(pc[r] == len(scheds[r]) for r in range(P)), "schedule deadlocks"
    return final


def test_chain_order_matches_definition():
    for P in range(2, 9):
        order = _chain_order(P)
        for k in range(P):
            assert order[k] == tuple((k + j) % P for j in range(1, P + 1))


def _inputs(P, n, seed=10, dtype="f32"):
    if dtype == "f32":
        return [np.random.default_rng(seed + r).uniform(-1, 1, n).astype(np.float32) for r in range(P)]
    return [np.random.default_rng(seed + r).integers(-1000, 1001, n, dtype=np.int32) for r in range(P)]


@pytest.mark.parametrize("P", [2, 3, 4])
@pytest.mark.parametrize("n,nch,nslots,slot", [(8, 1, 2, 16), (40, 2, 2, 16), (64, 1, 4, 32), (63, 3, 2, 16)])
def test_fp32_ring_sum_exact_rational(P, n, nch, nslots, slot):
    xs = _inputs(P, n, seed=100 + P + n)
    got = ring_order_sum(xs, nch, nslots, slot)
    order = _chain_order(P)
    for lo, hi, k in ring_chunks(n, 4, P, nch, nslots, slot):
        for i in range(lo, hi):
            acc = Fraction(float(xs[order[k][0]][i]))
            for r in order[k][1:]:
                acc = _f32_round(acc + Fraction(float(xs[r][i])))
            assert Fraction(float(got[i])) == acc, (i, k)


def test_fp32_order_matters_and_is_pinned():
    # a chain starting at rank k instead of k+1 gives different bits on this
    # input, so the exact pin above would catch a shifted schedule
    P, n = 4, 256
    xs = _inputs(P, n, seed=3)
    got = ring_order_sum(xs, 1, 2, 64)
    shifted = np.empty_like(got)
    for lo, hi, k in ring_chunks(n, 4, P, 1, 2, 64):
        acc = xs[k % P][lo:hi].copy()
        for j in range(1, P):
            acc = acc + xs[(k + j) % P][lo:hi]
        shifted[lo:hi] = acc
    assert not np.array_equal(got, shifted)


def test_int32_ring_sum_matches_int64():
    for P in (2, 3, 8):
        xs = _inputs(P, 5000, dtype="i32")
        got = ring_order_sum(xs, 3, 4, 64)
        ref = np.sum(np.stack(xs).astype(np.int64), axis=0)
        assert np.array_equal(got, ref.astype(np.int32))
    # wrapping: values near the int32 limits
    xs = [np.full(64, 2 ** 31 - 1, np.int32) for _ in range(3)]
    got = ring_order_sum(xs, 1, 2, 64)
    want = np.full(64, 3 * (2 ** 31 - 1), np.int64).astype(np.int32)
    assert np.array_equal(got, want) and int(want[0]) == 2 ** 31 - 3


def test_fp32_ring_sum_error_bound():
    for P in (2, 5, 8):
        xs = _inputs(P, 20000, seed=7 * P)
        got = ring_order_sum(xs, 4, 8, 512).astype(np.float64)
        stack = np.stack(xs).astype(np.float64)
        exact = stack.sum(axis=0)
        bound = (P - 1) * 2.0 ** -24 * np.abs(stack).sum(axis=0)
        assert np.all(np.abs(got - exact) <= bound)


def test_two_ranks_is_plain_sum():
    xs = _inputs(2, 3000, seed=1)
    got = ring_order_sum(xs, 2, 4, 128)
    assert np.array_equal(got, xs[0] + xs[1]) and np.array_equal(got, xs[1] + xs[0])


@pytest.mark.parametrize("P,n,nch,nslots,slot", [
    (2, 100, 1, 2, 16), (3, 257, 2, 2, 32), (4, 1000, 3, 4, 64), (8, 4099, 2, 8, 64), (5, 7, 4, 3, 16)])
@pytest.mark.parametrize("dtype", ["f32", "i32"])
def test_ring_state_machines_match_definition(P, n, nch, nslots, slot, dtype):
    xs = _inputs(P, n, seed=n, dtype=dtype)
    ref = ring_order_sum(xs, nch, nslots, slot)
    for seed in (0, 1):
        outs, _ = oracle.ring_allreduce(xs, nch, nslots, slot, seed=seed)
        for o in outs:
            assert np.array_equal(o, ref)


@pytest.mark.parametrize("P,n", [(2, 8), (3, 12)])
def test_ring_exhaustive(P, n):
    xs = _inputs(P, n, seed=5)
    ref = ring_order_sum(xs, 1, 2, 16)

    def make():
        outs = [np.zeros_like(x) for x in xs]
        return ring_system(xs, outs, 1, 2, 16)

    def final(s):
        for o in s.buffers:
            assert np.array_equal(o, ref)

    assert explore(make, final) > 1


def test_ring_needs_two_slots():
    with pytest.raises(ValueError):
        ring_chunk_elems(1, 64, 4)


def test_ring_neighbours_golden():
    g = json.load(open(os.path.join(GOLD, "ring_neighbours.json")))
    assert ring_prev(g["rank"], g["nranks"]) == g["recvpeer"]
    assert ring_next(g["rank"], g["nranks"]) == g["sendpeer"]


def test_schedule_structure():
    for P in range(2, 10):
        for r in range(P):
            s = ring_schedule(r, P)
            assert len(s) == 2 * P - 1
            # every chunk is finished (reduce-copied) by exactly one rank: chunk r at rank r
            assert [k for kind, k in s if kind == "recvReduceCopySend"] == [r]
            # the input of every chunk is read exactly once
            reads = [k for kind, k in s if kind in ("send", "recvReduceSend", "recvReduceCopySend")]
            assert sorted(reads) == list(range(P))
            # every chunk is written to the output exactly once
            outs = [k for kind, k in s if kind in ("recvReduceCopySend", "recvCopySend", "recv")]
            assert sorted(outs) == list(range(P))


def test_ring_partition():
    # 256 MiB fp32 per rank, 8 channels, 8 slots of 512 KiB: 32 MiB per channel,
    # chunks of 4 slots (2 MiB), 2 rounds of 8 chunks
    ranges = ring_channel_ranges(1 << 26, 4, 8)
    assert all(hi - lo == 1 << 23 for lo, hi in ranges)
    ce = ring_chunk_elems(8, 512 << 10, 4)
    assert ce == 1 << 19
    rounds = ring_rounds(1 << 23, 8, ce, 4)
    assert len(rounds) == 2 and all(hi - lo == ce for rnd in rounds for lo, hi in rnd)
    # a ragged channel: chunks cover it exactly, 16-byte aligned
    rounds = ring_rounds(1001, 3, 64, 4)
    flat = [c for rnd in rounds for c in rnd]
    assert flat[0][0] == 0 and flat[-1][1] == 1001
    for (a, b), (a2, _) in zip(flat, flat[1:]):
        assert b == a2 and (a % 4 == 0 or a == b)
