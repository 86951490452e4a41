"""Work partition rules of the FIFO data plane (CPU oracle; test infrastructure).

The transport pages fix the FIFO geometry (NCCL_STEPS slots of
stepSize = buffSize / NCCL_STEPS bytes, "NCCL transport setup", p2pRecvConnect,
stepSize assignment; "RDMA and GPUDirect" §7.2, 4 MB channel buffer) and the
ring neighbour rule ("NCCL transport setup", 具体说明: with 8 ranks, rank 0
receives from 7 and sends to 1).  They do not say how a user buffer is cut
into channels or ring chunks; the readings used here are:

* channel c of C gets bytes [c*q, min(n, (c+1)*q)) with
  q = round_up(ceil(n / C), 16): 16-byte aligned, the last ones may be short
  or empty;
* a channel range is moved in slot-steps of S bytes; step i covers
  [i*S, min(len, (i+1)*S));
* ring allreduce: element ranges per channel use the same rule with
  16 / esize element alignment; each channel range is walked in rounds of
  P chunks; a full chunk is (N // 2) slots (half the FIFO, so that one
  chunk's slots never fill the successor's FIFO); the last round shrinks its
  chunk to round_up(ceil(m / P), 16 / esize) elements for the m elements left.
"""
from __future__ import annotations


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def round_up(a: int, b: int) -> int:
    return ceil_div(a, b) * b


def channel_byte_ranges(nbytes: int, nchannels: int) -> list[tuple[int, int]]:
    """[lo, hi) byte range of every channel (possibly empty)."""
    if nchannels < 1:
        raise ValueError("nchannels must be >= 1")
    q = round_up(ceil_div(nbytes, nchannels), 16) if nbytes else 0
    out = []
    for c in range(nchannels):
        lo = min(nbytes, c * q)
        hi = min(nbytes, (c + 1) * q)
        out.append((lo, hi))
    return out


def slot_steps(length: int, slot_bytes: int) -> list[tuple[int, int]]:
    """(offset, size) of each slot-step of a channel range of `length` units."""
    return [(o, min(slot_bytes, length - o)) for o in range(0, length, slot_bytes)]


def ring_prev(rank: int, nranks: int) -> int:
    return (rank - 1) % nranks


def ring_next(rank: int, nranks: int) -> int:
    return (rank + 1) % nranks


def ring_channel_ranges(count: int, esize: int, nchannels: int) -> list[tuple[int, int]]:
    """Element ranges per channel for the ring (16-byte aligned boundaries)."""
    align = 16 // esize
    q = round_up(ceil_div(count, nchannels), align) if count else 0
    return [(min(count, c * q), min(count, (c + 1) * q)) for c in range(nchannels)]


def ring_chunk_elems(nslots: int, slot_bytes: int, esize: int) -> int:
    """Elements in a full ring chunk: half the FIFO's slots."""
    if nslots < 2:
        raise ValueError("the ring needs at least 2 slots per FIFO")
    return (nslots // 2) * slot_bytes // esize


def ring_rounds(length: int, nranks: int, chunk_elems: int, esize: int) -> list[list[tuple[int, int]]]:
    """Rounds of a channel range of `length` elements: each a list of nranks
    chunk ranges [lo, hi) relative to the channel start."""
    align = 16 // esize
    rounds = []
    off = 0
    while off < length:
        m = min(length - off, nranks * chunk_elems)
        cs = min(chunk_elems, round_up(ceil_div(m, nranks), align))
        chunks = []
        for k in range(nranks):
            lo = off + min(m, k * cs)
            hi = off + min(m, (k + 1) * cs)
            chunks.append((lo, hi))
        rounds.append(chunks)
        off += m
    return rounds


# Ring step kinds, in the order one rank runs them within a round.
SEND, RECV_REDUCE_SEND, RECV_REDUCE_COPY_SEND, RECV_COPY_SEND, RECV = (
    "send", "recvReduceSend", "recvReduceCopySend", "recvCopySend", "recv")


def ring_schedule(rank: int, nranks: int) -> list[tuple[str, int]]:
    """(step kind, chunk index) for one round at `rank`.

    Reduce-scatter: rank r first sends chunk r-1, then for j = 2..P-1 receives
    chunk r-j, adds its own copy and forwards it, and at j = P finishes chunk r
    (recvReduceCopySend).  Allgather: for j = 2..P-1 it receives the finished
    chunk r+1-j, keeps and forwards it; finally it receives chunk r+1.
    """
    P = nranks
    sched = [(SEND, (rank - 1) % P)]
    for j in range(2, P):
        sched.append((RECV_REDUCE_SEND, (rank - j) % P))
    sched.append((RECV_REDUCE_COPY_SEND, rank % P))
    for j in range(2, P):
        sched.append((RECV_COPY_SEND, (rank + 1 - j) % P))
    sched.append((RECV, (rank + 1) % P))
    return sched
