"""Whole transfers through the oracle's FIFO state machines (test infrastructure).

Each function splits the buffer into channels by `partition.channel_byte_ranges`,
builds one sender and one receiver per non-empty channel, runs them under a
seeded random interleaving (`fifo.run`) and returns the destination with the
FIFO objects, which can be passed back in to continue their step counters in
a following transfer (the counters are monotonic across operations).
"""
from __future__ import annotations

import numpy as np

from .fifo import (CEFifo, CEProxy, CEReceiver, CESender, LL128Fifo, LL128Receiver, LL128Sender, LLFifo,
                   LLReceiver, LLSender, PostedChannel,
                   PostedReceiver, PostedSender, SimpleFifo, SimpleReceiver, SimpleSender, System, ZeroCopyChannel,
                   ZeroCopyReceiver, ZeroCopySender, run)
from .partition import channel_byte_ranges
from .ring import ring_system


def simple_transfer(src: np.ndarray, nchannels: int, nslots: int, slot_bytes: int, seed: int = 0,
                    fifos: list[SimpleFifo] | None = None):
    """SIMPLE copy of the byte buffer `src`; returns (dst, fifos, events)."""
    src = np.ascontiguousarray(src).view(np.uint8).reshape(-1)
    dst = np.zeros_like(src)
    if fifos is None:
        fifos = [SimpleFifo(nslots, slot_bytes) for _ in range(nchannels)]
    actors = []
    for f, (lo, hi) in zip(fifos, channel_byte_ranges(len(src), nchannels)):
        if hi > lo:
            actors += [SimpleSender(f, src, lo, hi), SimpleReceiver(f, dst, lo, hi)]
    ev = run(System(actors, fifos, [dst]), seed=seed)
    return dst, fifos, ev


def ll_transfer(words: np.ndarray, nchannels: int, nslots: int, slot_bytes: int, seed: int = 0,
                fifos: list[LLFifo] | None = None, window: int = 2):
    """LL copy of the uint32 buffer `words` (even count); returns (out, fifos, events)."""
    words = np.ascontiguousarray(words, dtype=np.uint32).reshape(-1)
    if len(words) % 2:
        raise ValueError("LL moves whole 8-byte lines")
    out = np.zeros_like(words)
    if fifos is None:
        fifos = [LLFifo(nslots, slot_bytes) for _ in range(nchannels)]
    actors = []
    for f, (lo, hi) in zip(fifos, channel_byte_ranges(4 * len(words), nchannels)):
        if hi > lo:
            actors += [LLSender(f, words, lo // 4, hi // 4, window=window), LLReceiver(f, out, lo // 4, hi // 4)]
    ev = run(System(actors, fifos, [out]), seed=seed)
    return out, fifos, ev


def ll128_transfer(src: np.ndarray, nchannels: int, nslots: int, slot_bytes: int, seed: int = 0,
                   fifos: list[LL128Fifo] | None = None, batch: int = 2, window: int = 2, piece_words: int = 1):
    """LL128 copy of a buffer of whole 8-byte words; returns (out, fifos, events)."""
    raw = np.ascontiguousarray(src).view(np.uint8).reshape(-1)
    if len(raw) % 8:
        raise ValueError("LL128 moves whole 8-byte words")
    words = raw.view(np.uint64)
    out = np.zeros_like(words)
    if fifos is None:
        fifos = [LL128Fifo(nslots, slot_bytes) for _ in range(nchannels)]
    actors = []
    for f, (lo, hi) in zip(fifos, channel_byte_ranges(len(raw), nchannels)):
        if hi > lo:
            actors += [LL128Sender(f, words, lo // 8, hi // 8, batch=batch, window=window, piece_words=piece_words),
                       LL128Receiver(f, out, lo // 8, hi // 8)]
    ev = run(System(actors, fifos, [out]), seed=seed)
    return out, fifos, ev


def zero_copy_transfer(src: np.ndarray, nchannels: int, nslots: int, slot_bytes: int, seed: int = 0,
                       chans: list[ZeroCopyChannel] | None = None):
    """Zero-copy transfer of the byte buffer `src`; returns (dst, channels, events)."""
    src = np.ascontiguousarray(src).view(np.uint8).reshape(-1)
    dst = np.zeros_like(src)
    if chans is None:
        chans = [ZeroCopyChannel(nslots, slot_bytes) for _ in range(nchannels)]
    actors = []
    for c, (lo, hi) in zip(chans, channel_byte_ranges(len(src), nchannels)):
        if hi > lo:
            actors += [ZeroCopySender(c, src, lo, hi), ZeroCopyReceiver(c, dst, lo, hi)]
    ev = run(System(actors, chans, [dst]), seed=seed)
    return dst, chans, ev


def posted_transfer(src: np.ndarray, nchannels: int, nslots: int, slot_bytes: int, seed: int = 0,
                    chans: list[PostedChannel] | None = None, direct: bool = False):
    """Receiver-driven credit transfer of the byte buffer `src` (copy mode
    through staging slots, or direct into dst); returns (dst, channels, events)."""
    src = np.ascontiguousarray(src).view(np.uint8).reshape(-1)
    dst = np.zeros_like(src)
    if chans is None:
        chans = [PostedChannel(nslots, slot_bytes) for _ in range(nchannels)]
    actors = []
    for c, (lo, hi) in zip(chans, channel_byte_ranges(len(src), nchannels)):
        if hi > lo:
            actors += [PostedSender(c, src, lo, hi), PostedReceiver(c, dst, lo, hi, direct=direct)]
    ev = run(System(actors, chans, [dst]), seed=seed)
    return dst, chans, ev


def ce_transfer(src: np.ndarray, nchannels: int, nslots: int, slot_bytes: int, hops: int = 1, seed: int = 0,
                fifos: list[CEFifo] | None = None):
    """Proxy-mode transfer of the byte buffer `src` through `hops` host-driven
    copies per slot-step; returns (dst, fifos, events)."""
    src = np.ascontiguousarray(src).view(np.uint8).reshape(-1)
    dst = np.zeros_like(src)
    if fifos is None:
        fifos = [CEFifo(nslots, slot_bytes, hops) for _ in range(nchannels)]
    actors = []
    for f, (lo, hi) in zip(fifos, channel_byte_ranges(len(src), nchannels)):
        if hi > lo:
            n = -(-(hi - lo) // f.S)
            actors += [CESender(f, src, lo, hi)] + [CEProxy(f, h, n) for h in range(f.H)] + [CEReceiver(f, dst, lo, hi)]
    ev = run(System(actors, fifos, [dst]), seed=seed)
    return dst, fifos, ev


def ring_allreduce(inputs: list[np.ndarray], nchannels: int, nslots: int, slot_bytes: int, seed: int = 0):
    """Ring allreduce through per-rank FIFOs; returns (outputs, events)."""
    outs = [np.zeros_like(x) for x in inputs]
    sysm = ring_system(inputs, outs, nchannels, nslots, slot_bytes)
    ev = run(sysm, seed=seed)
    return outs, ev
