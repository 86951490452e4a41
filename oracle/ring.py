"""Virtual ring allreduce over P ranks (CPU oracle; test infrastructure only).

Ring topology: rank r receives from r-1 and sends to r+1 ("NCCL transport
setup", 具体说明: with 8 ranks rank 0's recvpeer is 7 and its sendpeer is 1).
Each rank owns, per channel, the SIMPLE FIFO its predecessor writes into (the
receiver owns the buffers and tail: "NCCL transport setup", shmTransport,
默认情况数据buff是recv侧分配的).  The pages name ring allreduce but do not
spell out its schedule; the textbook reduce-scatter + allgather schedule is
used (see `partition.ring_schedule`), built from the fused steps send,
recvReduceSend, recvReduceCopySend, recvCopySend and recv.

Two views are given:
* `ring_order_sum` — the plain definition of the result: element i of chunk k
  is ((x[k+1] + x[k+2]) + ...) + x[k], rank indices mod P, accumulated
  left to right in the element type (fp32 round-to-nearest-even, int32
  wrapping), because chunk k starts at rank k+1 and ends at rank k;
* `ring_system` — the ranks as FIFO state machines, for `fifo.run`/`explore`.
"""
from __future__ import annotations

import numpy as np

from .fifo import Actor, SimpleFifo, System
from .partition import (RECV, RECV_COPY_SEND, RECV_REDUCE_COPY_SEND, RECV_REDUCE_SEND, SEND,
                        ring_channel_ranges, ring_chunk_elems, ring_rounds, ring_schedule)

_HAS_RECV = {RECV_REDUCE_SEND, RECV_REDUCE_COPY_SEND, RECV_COPY_SEND, RECV}
_HAS_SEND = {SEND, RECV_REDUCE_SEND, RECV_REDUCE_COPY_SEND, RECV_COPY_SEND}
_REDUCES = {RECV_REDUCE_SEND, RECV_REDUCE_COPY_SEND}
_WRITES_OUT = {RECV_REDUCE_COPY_SEND, RECV_COPY_SEND, RECV}


def _add(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Elementwise a + b in the element type: IEEE fp32 or wrapping int32."""
    if a.dtype == np.float32:
        return np.add(a, b, dtype=np.float32)
    if a.dtype == np.int32:
        return np.add(a, b, dtype=np.int32)      # numpy int32 arrays wrap
    raise TypeError(a.dtype)


def ring_chunks(count: int, esize: int, nranks: int, nchannels: int, nslots: int, slot_bytes: int):
    """All (lo, hi, k) absolute element ranges: chunk index k within its round."""
    out = []
    ce = ring_chunk_elems(nslots, slot_bytes, esize)
    for (clo, chi) in ring_channel_ranges(count, esize, nchannels):
        for rnd in ring_rounds(chi - clo, nranks, ce, esize):
            for k, (lo, hi) in enumerate(rnd):
                out.append((clo + lo, clo + hi, k))
    return out


def ring_order_sum(inputs: list[np.ndarray], nchannels: int, nslots: int, slot_bytes: int) -> np.ndarray:
    """The allreduce result every rank ends with (definition, no FIFOs)."""
    P = len(inputs)
    x0 = inputs[0]
    out = np.empty_like(x0)
    for lo, hi, k in ring_chunks(len(x0), x0.itemsize, P, nchannels, nslots, slot_bytes):
        acc = inputs[(k + 1) % P][lo:hi].copy()
        for j in range(2, P + 1):
            acc = _add(acc, inputs[(k + j) % P][lo:hi])
        out[lo:hi] = acc
    return out


class RingAgent(Actor):
    """One rank on one channel: receives from its own FIFO (written by rank
    r-1) and sends into rank r+1's FIFO, one slot-step at a time.

    Events per slot-step: wait (tail of own FIFO > rstep for steps that
    receive; sstep < head + N of the next FIFO for steps that send) ->
    compute and move the data -> store the next FIFO's tail -> store the own
    FIFO's head."""
    WAIT, DO, PUB_TAIL, PUB_HEAD = range(4)

    def __init__(self, rank: int, recv_fifo: SimpleFifo, send_fifo: SimpleFifo,
                 inp: np.ndarray, out: np.ndarray, items: list[tuple[str, int, int]]):
        self.rank = rank
        self.rf, self.sf = recv_fifo, send_fifo
        self.inp, self.out = inp, out
        self.es = inp.itemsize
        self.epl = recv_fifo.S // self.es            # elements per slot
        # flatten (kind, lo, hi) items into slot-steps
        self.steps = []
        for kind, lo, hi in items:
            for o in range(lo, hi, self.epl):
                self.steps.append((kind, o, min(hi, o + self.epl)))
        self.i = 0
        self.rstep = recv_fifo.head
        self.sstep = send_fifo.tail
        self.phase = self.WAIT
        self.name = f"ring-rank{rank}"

    def done(self):
        return self.i >= len(self.steps)

    def choices(self):
        if self.done():
            return []
        kind = self.steps[self.i][0]
        if self.phase == self.WAIT:
            if kind in _HAS_RECV and not self.rf.tail > self.rstep:
                return []
            if kind in _HAS_SEND and not self.sstep < self.sf.head + self.sf.N:
                return []
        return [0]

    def fire(self, choice):
        kind, lo, hi = self.steps[self.i]
        if self.phase == self.WAIT:
            self.phase = self.DO
        elif self.phase == self.DO:
            nb = (hi - lo) * self.es
            if kind in _HAS_RECV:
                got = self.rf.drain(self.rstep, nb).view(self.inp.dtype)
            if kind == SEND:
                val = self.inp[lo:hi]
            elif kind in _REDUCES:
                val = _add(got, self.inp[lo:hi])
            else:
                val = got
            if kind in _WRITES_OUT:
                self.out[lo:hi] = val
            if kind in _HAS_SEND:
                self.sf.fill(self.sstep, np.ascontiguousarray(val).view(np.uint8))
            self.phase = self.PUB_TAIL
        elif self.phase == self.PUB_TAIL:
            if kind in _HAS_SEND:
                self.sf.tail = self.sstep + 1
                self.sstep += 1
            self.phase = self.PUB_HEAD
        else:
            if kind in _HAS_RECV:
                self.rf.head = self.rstep + 1
                self.rstep += 1
            self.i += 1
            self.phase = self.WAIT

    def state(self):
        return (self.i, self.phase, self.rstep, self.sstep)


def ring_system(inputs: list[np.ndarray], outputs: list[np.ndarray], nchannels: int,
                nslots: int, slot_bytes: int) -> System:
    """State machines for every (rank, channel) of the ring allreduce."""
    P = len(inputs)
    count = len(inputs[0])
    es = inputs[0].itemsize
    if slot_bytes % 16:
        raise ValueError("slot bytes must be a multiple of 16")
    ce = ring_chunk_elems(nslots, slot_bytes, es)
    actors, fifos = [], []
    for (clo, chi) in ring_channel_ranges(count, es, nchannels):
        rounds = ring_rounds(chi - clo, P, ce, es)
        ch_fifos = [SimpleFifo(nslots, slot_bytes) for _ in range(P)]   # fifo[r]: written by r-1
        fifos += ch_fifos
        for r in range(P):
            items = []
            for rnd in rounds:
                for kind, k in ring_schedule(r, P):
                    lo, hi = rnd[k]
                    if hi > lo:
                        items.append((kind, clo + lo, clo + hi))
            actors.append(RingAgent(r, ch_fifos[r], ch_fifos[(r + 1) % P], inputs[r], outputs[r], items))
    return System(actors, fifos, outputs)
