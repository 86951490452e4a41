"""FIFO protocol state machines (CPU oracle; test infrastructure only).

Each endpoint is an explicit state machine over shared FIFO state.  A seeded
scheduler (`run`) fires one enabled event at a time; `explore` walks every
reachable state of a tiny system.  After every event the FIFO invariants are
checked, so a schedule that breaks the protocol raises `ProtocolViolation`
at the event that broke it.

Protocol sources (page title, section):
* copy mode: "NCCL transport data transfer (二)", p2pTransport / copy mode —
  the sender writes a slot, updates tail; the receiver sees tail, copies the
  slot to the user buffer, updates head.  "NCCL transport setup",
  整体图解 (producer/consumer model) says the same.
* zero copy: same page, zero copy — the receiver puts its buffer address in
  ptrExchange, the sender reads it, writes the data there, updates tail; the
  receiver sees tail and updates head.
* shm normal mode (host-placed FIFO): same page, shmTransport / 正常方式 —
  identical steps with the buffers and tail in host memory.
* LL: "RDMA and GPUDirect" §4.1 — the data carries the flag and the receiver
  polls memory.  Line = 16 bytes {data0, flag0, data1, flag1}.
* LL128: same section (the flag sits in the last bytes of what was written)
  and §8 (GPUDirect flush: a visible flag does not by itself mean the data
  written before it is visible).  Line = 128 bytes, 15 uint64 payload words
  and a uint64 flag in the last 8 bytes.
* initial counters: "NCCL transport setup", netTransport (head starts at 0
  outside shared-buffer mode) and the per-slot size word initialised to -1.

Readings where the pages are silent:
* credit: the sender may fill step s only while s < head + N;
* LL flag of every line of slot-step s is (s + 1) mod 2**32, so that zeroed
  memory never matches; LL still uses head for slot reuse and has no tail;
* each 8-byte half {data, flag} of an LL line becomes visible on its own
  (a 16-byte line may be seen torn), in any order within a small window;
* LL128 flag of every line of slot-step s is s + 1 as a full uint64; the
  sender makes a batch of lines' payload visible before it writes their
  flags, and the receiver reads a line's payload only after its flag; each
  8-byte word becomes visible on its own, in any order;
* zero copy: the receiver posts its address only into an empty ptrExchange;
  the sender writes chunks of at most S bytes, one tail per chunk, under the
  same credit rule; the receiver returns head per chunk; the sender empties
  ptrExchange once head reaches the last chunk.

Our design beyond the pages (modelled so that its credit rule is checked):
* LL128 lanes: a channel's lines are cut into G sender stripes and GR
  receiver stripes of ceil(L / G) and ceil(L / GR) lines; each receiver
  lane returns credit through a head of its own, and a sender lane fills
  its lines of step s only once every receiver lane whose stripe meets its
  own has head > s - N.
"""
from __future__ import annotations

import copy
from dataclasses import dataclass

import numpy as np

from .partition import ceil_div


class ProtocolViolation(AssertionError):
    """A schedule broke a FIFO invariant."""


class Deadlock(AssertionError):
    """No endpoint can move but some have not finished."""


# --------------------------------------------------------------------------
# SIMPLE
# --------------------------------------------------------------------------

class SimpleFifo:
    """Shared state of one SIMPLE channel: N slots of S bytes, head, tail."""

    def __init__(self, nslots: int, slot_bytes: int, step0: int = 0):
        if nslots < 1 or slot_bytes < 1:
            raise ValueError("need nslots >= 1 and slot_bytes >= 1")
        self.N = nslots
        self.S = slot_bytes
        self.slots = np.zeros((nslots, slot_bytes), np.uint8)
        self.size = [-1] * nslots          # per-slot size word
        self.head = step0                  # consumer cursor (credit)
        self.tail = step0                  # producer cursor
        # bookkeeping used only by the checks:
        self.owner = [None] * nslots       # step whose bytes the slot holds
        self.consumed = [True] * nslots
        self.max_occupancy = 0

    def check(self):
        occ = self.tail - self.head
        if occ < 0:
            raise ProtocolViolation(f"head {self.head} passed tail {self.tail}")
        if occ > self.N:
            raise ProtocolViolation(f"tail {self.tail} exceeds head {self.head} + N {self.N}")
        self.max_occupancy = max(self.max_occupancy, occ)

    def state(self):
        return (self.head, self.tail, self.slots.tobytes(), tuple(self.size),
                tuple(self.owner), tuple(self.consumed))

    # slot access with ownership checks
    def fill(self, step: int, data: np.ndarray):
        k = step % self.N
        if not self.consumed[k]:
            raise ProtocolViolation(f"step {step} overwrites slot {k} holding unconsumed step {self.owner[k]}")
        self.slots[k, :len(data)] = data
        self.size[k] = len(data)
        self.owner[k] = step
        self.consumed[k] = False

    def drain(self, step: int, nbytes: int) -> np.ndarray:
        k = step % self.N
        if self.owner[k] != step or self.consumed[k]:
            raise ProtocolViolation(f"step {step} reads slot {k} holding step {self.owner[k]} "
                                    f"(consumed={self.consumed[k]})")
        if self.size[k] != nbytes:
            raise ProtocolViolation(f"slot {k} size word {self.size[k]} != {nbytes}")
        self.consumed[k] = True
        return self.slots[k, :nbytes].copy()


class Actor:
    name = "actor"

    def done(self) -> bool:
        raise NotImplementedError

    def choices(self) -> list:
        raise NotImplementedError

    def fire(self, choice):
        raise NotImplementedError

    def state(self):
        raise NotImplementedError


class SimpleSender(Actor):
    """Copy src[lo:hi] into the FIFO one slot-step at a time.

    Events per step: wait credit (step < head + N) -> fill slot -> store tail.
    `fault` plants a mistake for the checker tests: "skip_credit",
    "tail_before_fill", "skip_tail" (last step's tail never stored).
    """
    WAIT, FILL, PUB, DONE = range(4)

    def __init__(self, fifo: SimpleFifo, src: np.ndarray, lo: int, hi: int, fault: str | None = None):
        self.f, self.src, self.lo, self.hi = fifo, src, lo, hi
        self.base = fifo.tail
        self.nsteps = ceil_div(hi - lo, fifo.S)
        self.step = self.base
        self.phase = self.WAIT if self.nsteps else self.DONE
        self.fault = fault
        self.name = f"simple-send[{lo}:{hi}]"
        if fault == "tail_before_fill":
            self.order = (self.WAIT, self.PUB, self.FILL)
        else:
            self.order = (self.WAIT, self.FILL, self.PUB)

    def _piece(self):
        off = self.lo + (self.step - self.base) * self.f.S
        return self.src[off:min(self.hi, off + self.f.S)]

    def done(self):
        return self.phase == self.DONE

    def choices(self):
        if self.phase == self.DONE:
            return []
        if self.phase == self.WAIT:
            ok = self.fault == "skip_credit" or self.step < self.f.head + self.f.N
            return [0] if ok else []
        if self.phase == self.PUB and self.fault == "skip_tail" and self.step == self.base + self.nsteps - 1:
            return []
        return [0]

    def _advance(self):
        i = self.order.index(self.phase)
        if i + 1 < len(self.order):
            self.phase = self.order[i + 1]
        else:
            self.step += 1
            self.phase = self.WAIT if self.step < self.base + self.nsteps else self.DONE

    def fire(self, choice):
        if self.phase == self.FILL:
            self.f.fill(self.step, self._piece())
        elif self.phase == self.PUB:
            self.f.tail = self.step + 1
        self._advance()

    def state(self):
        return (self.step, self.phase)


class SimpleReceiver(Actor):
    """Copy the FIFO's slot-steps into dst[lo:hi].

    Events per step: wait tail > step -> copy slot out -> store head.
    `fault`: "head_before_copy", "skip_tail_wait".
    """
    WAIT, COPY, PUB, DONE = range(4)

    def __init__(self, fifo: SimpleFifo, dst: np.ndarray, lo: int, hi: int, fault: str | None = None):
        self.f, self.dst, self.lo, self.hi = fifo, dst, lo, hi
        self.base = fifo.head
        self.nsteps = ceil_div(hi - lo, fifo.S)
        self.step = self.base
        self.phase = self.WAIT if self.nsteps else self.DONE
        self.fault = fault
        self.name = f"simple-recv[{lo}:{hi}]"
        if fault == "head_before_copy":
            self.order = (self.WAIT, self.PUB, self.COPY)
        else:
            self.order = (self.WAIT, self.COPY, self.PUB)

    def done(self):
        return self.phase == self.DONE

    def choices(self):
        if self.phase == self.DONE:
            return []
        if self.phase == self.WAIT:
            ok = self.fault == "skip_tail_wait" or self.f.tail > self.step
            return [0] if ok else []
        return [0]

    def _advance(self):
        i = self.order.index(self.phase)
        if i + 1 < len(self.order):
            self.phase = self.order[i + 1]
        else:
            self.step += 1
            self.phase = self.WAIT if self.step < self.base + self.nsteps else self.DONE

    def fire(self, choice):
        if self.phase == self.COPY:
            off = self.lo + (self.step - self.base) * self.f.S
            n = min(self.hi, off + self.f.S) - off
            self.dst[off:off + n] = self.f.drain(self.step, n)
        elif self.phase == self.PUB:
            self.f.head = self.step + 1
        self._advance()

    def state(self):
        return (self.step, self.phase)


# --------------------------------------------------------------------------
# LL
# --------------------------------------------------------------------------

LL_LINE_BYTES = 16      # {data0, flag0, data1, flag1}, uint32 each
LL_LINE_PAYLOAD = 8     # two uint32 data words per line


def ll_flag(step: int) -> int:
    return (step + 1) & 0xFFFFFFFF


class LLFifo:
    """Shared state of one LL channel: N slots of S bytes of 16-byte lines."""

    def __init__(self, nslots: int, slot_bytes: int, step0: int = 0):
        if nslots < 1 or slot_bytes < LL_LINE_BYTES or slot_bytes % LL_LINE_BYTES:
            raise ValueError("LL slots hold whole 16-byte lines")
        self.N = nslots
        self.S = slot_bytes
        self.L = slot_bytes // LL_LINE_BYTES
        self.lines = np.zeros((nslots, self.L, 4), np.uint32)      # visible memory
        self.half_owner = np.full((nslots, self.L, 2), -1, np.int64)  # bookkeeping
        self.head = step0
        self.started = step0          # steps the sender has been granted (bookkeeping)
        self.max_occupancy = 0

    def check(self):
        occ = self.started - self.head
        if occ < 0 or occ > self.N:
            raise ProtocolViolation(f"LL sender started {self.started} steps, head {self.head}, N {self.N}")
        self.max_occupancy = max(self.max_occupancy, occ)

    def state(self):
        return (self.head, self.started, self.lines.tobytes(), self.half_owner.tobytes())


@dataclass
class _Half:
    slot: int
    line: int
    half: int
    data: int
    flag: int
    step: int


class LLSender(Actor):
    """Send words[lo:hi] (uint32, even count) as LL lines.

    Events: wait credit for a new slot-step; issue the next line (its two
    8-byte halves enter a pending pool of at most `window` lines); make any
    pending half visible.  `fault`: "skip_credit".
    """

    def __init__(self, fifo: LLFifo, words: np.ndarray, lo: int, hi: int, window: int = 2,
                 fault: str | None = None):
        if (hi - lo) % 2:
            raise ValueError("LL moves whole 8-byte lines")
        self.f, self.words, self.lo, self.hi = fifo, words, lo, hi
        self.nlines = (hi - lo) // 2
        self.base = fifo.started
        self.nsteps = ceil_div(self.nlines, fifo.L)
        self.step = self.base          # next step to start
        self.line = 0                  # next line within the current step
        self.granted = False
        self.pending: list[_Half] = []
        self.window = window
        self.fault = fault
        self.name = f"ll-send[{lo}:{hi}]"

    def _lines_in(self, step):
        rel = step - self.base
        return min(self.f.L, self.nlines - rel * self.f.L)

    def done(self):
        return self.step >= self.base + self.nsteps and not self.pending

    def choices(self):
        opts = [("vis", i) for i in range(len(self.pending))]
        if self.step < self.base + self.nsteps:
            if not self.granted:
                if self.fault == "skip_credit" or self.step < self.f.head + self.f.N:
                    opts.append(("grant",))
            elif len(self.pending) < 2 * self.window:
                opts.append(("issue",))
        return opts

    def fire(self, choice):
        if choice[0] == "grant":
            self.granted = True
            self.f.started = self.step + 1
        elif choice[0] == "issue":
            rel = self.step - self.base
            g = rel * self.f.L + self.line            # global line index
            d0 = int(self.words[self.lo + 2 * g])
            d1 = int(self.words[self.lo + 2 * g + 1])
            k = self.step % self.f.N
            fl = ll_flag(self.step)
            self.pending.append(_Half(k, self.line, 0, d0, fl, self.step))
            self.pending.append(_Half(k, self.line, 1, d1, fl, self.step))
            self.line += 1
            if self.line == self._lines_in(self.step):
                self.step += 1
                self.line = 0
                self.granted = False
        else:
            h = self.pending.pop(choice[1])
            if h.step >= self.f.head + self.f.N:
                raise ProtocolViolation(f"LL step {h.step} overwrites slot {h.slot} before head {self.f.head}")
            self.f.lines[h.slot, h.line, 2 * h.half] = h.data
            self.f.lines[h.slot, h.line, 2 * h.half + 1] = h.flag
            self.f.half_owner[h.slot, h.line, h.half] = h.step

    def state(self):
        return (self.step, self.line, self.granted,
                tuple((h.slot, h.line, h.half, h.data, h.flag, h.step) for h in self.pending))


class LLReceiver(Actor):
    """Receive LL lines into out[lo:hi]; head = step + 1 after a slot's last line.

    A line is accepted only when both flags equal the step's flag.
    `fault`: "one_flag" (accept on flag1 alone), "head_early" (return credit
    before reading the slot's last line).
    """

    def __init__(self, fifo: LLFifo, out: np.ndarray, lo: int, hi: int, fault: str | None = None):
        self.f, self.out, self.lo, self.hi = fifo, out, lo, hi
        self.nlines = (hi - lo) // 2
        self.base = fifo.head
        self.nsteps = ceil_div(self.nlines, fifo.L)
        self.step = self.base
        self.line = 0
        self.pub = False               # all lines of `step` read, head not yet stored
        self.early = False             # planted fault: head already stored for `step`
        self.fault = fault
        self.name = f"ll-recv[{lo}:{hi}]"

    def _lines_in(self, step):
        rel = step - self.base
        return min(self.f.L, self.nlines - rel * self.f.L)

    def done(self):
        return self.step >= self.base + self.nsteps

    def choices(self):
        if self.done():
            return []
        if self.pub:
            return [("head",)]
        if (self.fault == "head_early" and not self.early
                and self.line == self._lines_in(self.step) - 1):
            return [("head",)]
        k = self.step % self.f.N
        ln = self.f.lines[k, self.line]
        fl = ll_flag(self.step)
        if self.fault == "one_flag":
            ok = int(ln[3]) == fl
        else:
            ok = int(ln[1]) == fl and int(ln[3]) == fl
        return [("read",)] if ok else []

    def _next_step(self):
        self.step += 1
        self.line = 0
        self.pub = False
        self.early = False

    def fire(self, choice):
        if choice[0] == "head":
            self.f.head = self.step + 1
            if self.pub:
                self._next_step()
            else:
                self.early = True
            return
        k = self.step % self.f.N
        own = self.f.half_owner[k, self.line]
        if own[0] != self.step or own[1] != self.step:
            raise ProtocolViolation(f"LL line {self.line} of step {self.step} accepted with halves "
                                    f"from steps {own[0]}, {own[1]}")
        g = (self.step - self.base) * self.f.L + self.line
        ln = self.f.lines[k, self.line]
        self.out[self.lo + 2 * g] = ln[0]
        self.out[self.lo + 2 * g + 1] = ln[2]
        self.line += 1
        if self.line == self._lines_in(self.step):
            if self.early:
                self._next_step()
            else:
                self.pub = True

    def state(self):
        return (self.step, self.line, self.pub, self.early)


# --------------------------------------------------------------------------
# LL128 ("RDMA and GPUDirect" §4: the data carries the flag in the buffer's
# last bytes; §8, GPUDirect flush: seeing the flag does not by itself mean
# the data before it has landed)
# --------------------------------------------------------------------------

LL128_LINE_BYTES = 128   # 16 uint64 words
LL128_LINE_WORDS = 16
LL128_DATA_WORDS = 15    # words 0..14 carry payload, word 15 is the flag


def ll128_flag(step: int) -> int:
    """Flag word of every line of slot-step `step`: step + 1 as a full
    uint64 (zeroed memory never matches; no wrap within 2**64 steps)."""
    return (step + 1) & 0xFFFFFFFFFFFFFFFF


class LL128Fifo:
    """Shared state of one LL128 channel: N slots of S bytes of 128-byte lines."""

    def __init__(self, nslots: int, slot_bytes: int, step0: int = 0):
        if nslots < 1 or slot_bytes < LL128_LINE_BYTES or slot_bytes % LL128_LINE_BYTES:
            raise ValueError("LL128 slots hold whole 128-byte lines")
        self.N = nslots
        self.S = slot_bytes
        self.L = slot_bytes // LL128_LINE_BYTES
        self.lines = np.zeros((nslots, self.L, LL128_LINE_WORDS), np.uint64)   # visible memory
        self.owner = np.full((nslots, self.L, LL128_LINE_WORDS), -1, np.int64)  # step that wrote each word
        self.head = step0
        self.started = step0
        self.max_occupancy = 0

    def check(self):
        occ = self.started - self.head
        if occ < 0 or occ > self.N:
            raise ProtocolViolation(f"LL128 sender started {self.started} steps, head {self.head}, N {self.N}")
        self.max_occupancy = max(self.max_occupancy, occ)

    def state(self):
        return (self.head, self.started, self.lines.tobytes(), self.owner.tobytes())


@dataclass
class _Piece:
    slot: int
    line: int
    w0: int            # first word of the line this piece writes
    values: tuple      # uint64 words
    step: int


def _ll128_lines(nwords: int, L: int, rel: int) -> int:
    """Lines of relative slot-step `rel` for a channel of `nwords` payload words."""
    left = nwords - rel * L * LL128_DATA_WORDS
    return min(L, ceil_div(left, LL128_DATA_WORDS))


class LL128Sender(Actor):
    """Send words[lo:hi] (uint64) as LL128 lines.

    Slot-step s carries payload words [s*L*15, (s+1)*L*15) of the channel;
    line i of a step the next 15 of them, words past the end written as 0.
    The sender writes the lines of a step in batches of at most `batch`
    lines: every payload word enters a pending pool and becomes visible on
    its own (8 bytes: the unit a store is atomic in; `piece_words` > 1
    coarsens it to keep exhaustive searches small); only when every payload
    word of the batch is visible (the fence) do the batch's flags enter the
    pool.  `window` bounds the pending payload lines.
    `fault`: "skip_credit" (no head check), "flag_with_data" (a line's flag
    enters the pool together with its payload: no fence).
    """

    def __init__(self, fifo: LL128Fifo, words: np.ndarray, lo: int, hi: int, batch: int = 2, window: int = 2,
                 piece_words: int = 1, fault: str | None = None):
        self.f, self.words, self.lo, self.hi = fifo, words, lo, hi
        self.nwords = hi - lo
        self.base = fifo.started
        self.nsteps = ceil_div(self.nwords, fifo.L * LL128_DATA_WORDS)
        self.step = self.base
        self.line = 0
        self.granted = False
        self.batch = batch
        self.window = window
        self.pw = piece_words
        self.in_batch: list[tuple[int, int, int]] = []   # (slot, line, step) written, flag not yet issued
        self.pending: list[_Piece] = []
        self.fault = fault
        self.name = f"ll128-send[{lo}:{hi}]"

    def _lines_in(self, step):
        return _ll128_lines(self.nwords, self.f.L, step - self.base)

    def done(self):
        return self.step >= self.base + self.nsteps and not self.pending and not self.in_batch

    def _data_pending(self):
        return sum(1 for p in self.pending if p.w0 < LL128_DATA_WORDS)

    def choices(self):
        opts = [("vis", i) for i in range(len(self.pending))]
        if self.in_batch and self._data_pending() == 0:
            opts.append(("fence",))
        if (self.step < self.base + self.nsteps and len(self.in_batch) < self.batch
                and all(st == self.step for (_, _, st) in self.in_batch)):
            if not self.granted:
                if self.fault == "skip_credit" or self.step < self.f.head + self.f.N:
                    opts.append(("grant",))
            elif self._data_pending() < self.window * ceil_div(LL128_DATA_WORDS, self.pw):
                opts.append(("issue",))
        return opts

    def fire(self, choice):
        if choice[0] == "grant":
            self.granted = True
            self.f.started = self.step + 1
        elif choice[0] == "issue":
            rel = self.step - self.base
            g0 = (rel * self.f.L + self.line) * LL128_DATA_WORDS     # first payload word of the line
            vals = [int(self.words[self.lo + g0 + j]) if g0 + j < self.nwords else 0
                    for j in range(LL128_DATA_WORDS)]
            k = self.step % self.f.N
            for w0 in range(0, LL128_DATA_WORDS, self.pw):
                self.pending.append(_Piece(k, self.line, w0, tuple(vals[w0:w0 + self.pw]), self.step))
            if self.fault == "flag_with_data":
                self.pending.append(_Piece(k, self.line, LL128_DATA_WORDS, (ll128_flag(self.step),), self.step))
            else:
                self.in_batch.append((k, self.line, self.step))
            self.line += 1
            if self.line == self._lines_in(self.step):
                self.step += 1
                self.line = 0
                self.granted = False
        elif choice[0] == "fence":
            for (k, ln, st) in self.in_batch:
                self.pending.append(_Piece(k, ln, LL128_DATA_WORDS, (ll128_flag(st),), st))
            self.in_batch = []
        else:
            p = self.pending.pop(choice[1])
            if p.step >= self.f.head + self.f.N:
                raise ProtocolViolation(f"LL128 step {p.step} overwrites slot {p.slot} before head {self.f.head}")
            n = len(p.values)
            self.f.lines[p.slot, p.line, p.w0:p.w0 + n] = np.array(p.values, np.uint64)
            self.f.owner[p.slot, p.line, p.w0:p.w0 + n] = p.step

    def state(self):
        return (self.step, self.line, self.granted, tuple(self.in_batch),
                tuple((p.slot, p.line, p.w0, p.values, p.step) for p in self.pending))


class LL128Receiver(Actor):
    """Receive LL128 lines into out[lo:hi] (uint64); head = step + 1 after a
    slot's last line.

    A line is read only once its flag word equals the step's flag, and the
    read comes after the flag (the receiver's fence): every payload word it
    takes must then have been written in this step.  `fault`:
    "data_before_flag" (the payload words are loaded first and kept if the
    flag then matches: no fence between), "head_early" (return credit before
    reading the slot's last line).
    """

    def __init__(self, fifo: LL128Fifo, out: np.ndarray, lo: int, hi: int, fault: str | None = None):
        self.f, self.out, self.lo, self.hi = fifo, out, lo, hi
        self.nwords = hi - lo
        self.base = fifo.head
        self.nsteps = ceil_div(self.nwords, fifo.L * LL128_DATA_WORDS)
        self.step = self.base
        self.line = 0
        self.pub = False
        self.early = False
        self.snap = None               # planted fault: payload loaded before the flag
        self.fault = fault
        self.name = f"ll128-recv[{lo}:{hi}]"

    def _lines_in(self, step):
        return _ll128_lines(self.nwords, self.f.L, step - self.base)

    def done(self):
        return self.step >= self.base + self.nsteps

    def choices(self):
        if self.done():
            return []
        if self.pub:
            return [("head",)]
        if (self.fault == "head_early" and not self.early
                and self.line == self._lines_in(self.step) - 1):
            return [("head",)]
        if self.fault == "data_before_flag" and self.snap is None:
            return [("load",)]
        k = self.step % self.f.N
        ok = int(self.f.lines[k, self.line, LL128_DATA_WORDS]) == ll128_flag(self.step)
        if self.fault == "data_before_flag":
            return [("read",)] if ok else [("drop",)]
        return [("read",)] if ok else []

    def _next_step(self):
        self.step += 1
        self.line = 0
        self.pub = False
        self.early = False

    def fire(self, choice):
        k = self.step % self.f.N
        if choice[0] == "head":
            self.f.head = self.step + 1
            if self.pub:
                self._next_step()
            else:
                self.early = True
            return
        if choice[0] == "load":
            self.snap = (self.f.lines[k, self.line, :LL128_DATA_WORDS].copy(),
                         self.f.owner[k, self.line, :LL128_DATA_WORDS].copy())
            return
        if choice[0] == "drop":
            self.snap = None
            return
        if self.snap is not None:
            vals, own = self.snap
            self.snap = None
        else:
            vals = self.f.lines[k, self.line, :LL128_DATA_WORDS]
            own = self.f.owner[k, self.line, :LL128_DATA_WORDS]
        g0 = ((self.step - self.base) * self.f.L + self.line) * LL128_DATA_WORDS
        n = min(LL128_DATA_WORDS, self.nwords - g0)
        stale = [int(o) for o in own if o != self.step]
        if stale:
            raise ProtocolViolation(f"LL128 line {self.line} of step {self.step} read with words from steps {stale}")
        self.out[self.lo + g0:self.lo + g0 + n] = vals[:n]
        self.line += 1
        if self.line == self._lines_in(self.step):
            if self.early:
                self._next_step()
            else:
                self.pub = True

    def state(self):
        snap = None if self.snap is None else (self.snap[0].tobytes(), self.snap[1].tobytes())
        return (self.step, self.line, self.pub, self.early, snap)


class LL128LaneFifo(LL128Fifo):
    """An LL128 channel whose receiver side is cut into `rlanes` lanes (our
    design; the pages have one receiver per channel): receiver lane r owns
    lines [r*LgR, (r+1)*LgR) of every slot, LgR = ceil(L / rlanes), and keeps
    a head of its own."""

    def __init__(self, nslots: int, slot_bytes: int, rlanes: int, step0: int = 0):
        super().__init__(nslots, slot_bytes, step0)
        self.GR = rlanes
        self.LgR = ceil_div(self.L, rlanes)
        self.heads = [step0] * rlanes

    def rlane(self, line: int) -> int:
        return line // self.LgR

    def check(self):
        pass   # the per-line overwrite check in the senders is the invariant

    def state(self):
        return (tuple(self.heads), self.lines.tobytes(), self.owner.tobytes())


class LL128LaneSender(Actor):
    """Sender lane g of `lanes`: writes lines [g*LgS, (g+1)*LgS) of every
    slot-step of words[lo:hi], LgS = ceil(L / lanes), as LL128Sender writes
    whole steps (payload words visible one piece at a time, the batch's flags
    only after all its payload).  It fills its lines of step s only once every
    receiver lane whose lines meet its own has head > s - N; a payload piece
    that becomes visible while the receiver lane owning its line has not
    returned that credit is a protocol violation.  `fault`: "one_lane_credit"
    (wait only for the first receiver lane its lines meet)."""

    def __init__(self, fifo: LL128LaneFifo, words: np.ndarray, lo: int, hi: int, lanes: int, lane: int,
                 batch: int = 1, piece_words: int = LL128_DATA_WORDS, fault: str | None = None):
        self.f, self.words, self.lo, self.hi = fifo, words, lo, hi
        self.nwords = hi - lo
        self.base = fifo.heads[0]
        self.nsteps = ceil_div(self.nwords, fifo.L * LL128_DATA_WORDS)
        lg = ceil_div(fifo.L, lanes)
        self.l0 = min(lane * lg, fifo.L)
        self.l1 = min(self.l0 + lg, fifo.L)
        self.rlanes = sorted({fifo.rlane(i) for i in range(self.l0, self.l1)})
        if fault == "one_lane_credit":
            self.rlanes = self.rlanes[:1]
        self.step = self.base
        self.line = self.l0
        self.granted = False
        self.batch, self.pw = batch, piece_words
        self.in_batch: list[tuple[int, int, int]] = []
        self.pending: list[_Piece] = []
        self.name = f"ll128-send-lane{lane}[{lo}:{hi}]"
        self._skip_empty()

    def _end(self, step):
        return min(self.l1, _ll128_lines(self.nwords, self.f.L, step - self.base))

    def _skip_empty(self):
        while self.step < self.base + self.nsteps and self.l0 >= self._end(self.step) and not self.in_batch:
            self.step += 1

    def done(self):
        return self.step >= self.base + self.nsteps and not self.pending and not self.in_batch

    def choices(self):
        opts = [("vis", i) for i in range(len(self.pending))]
        if self.in_batch and not any(p.w0 < LL128_DATA_WORDS for p in self.pending):
            opts.append(("fence",))
        if (self.step < self.base + self.nsteps and len(self.in_batch) < self.batch
                and all(st == self.step for (_, _, st) in self.in_batch)):
            if not self.granted:
                if all(self.step < self.f.heads[r] + self.f.N for r in self.rlanes):
                    opts.append(("grant",))
            else:
                opts.append(("issue",))
        return opts

    def fire(self, choice):
        if choice[0] == "grant":
            self.granted = True
        elif choice[0] == "issue":
            rel = self.step - self.base
            g0 = (rel * self.f.L + self.line) * LL128_DATA_WORDS
            vals = [int(self.words[self.lo + g0 + j]) if g0 + j < self.nwords else 0
                    for j in range(LL128_DATA_WORDS)]
            k = self.step % self.f.N
            for w0 in range(0, LL128_DATA_WORDS, self.pw):
                self.pending.append(_Piece(k, self.line, w0, tuple(vals[w0:w0 + self.pw]), self.step))
            self.in_batch.append((k, self.line, self.step))
            self.line += 1
            if self.line == self._end(self.step):
                self.step += 1
                self.line = self.l0
                self.granted = False
                self._skip_empty()
        elif choice[0] == "fence":
            for (k, ln, st) in self.in_batch:
                self.pending.append(_Piece(k, ln, LL128_DATA_WORDS, (ll128_flag(st),), st))
            self.in_batch = []
            self._skip_empty()
        else:
            p = self.pending.pop(choice[1])
            r = self.f.rlane(p.line)
            if p.step >= self.f.heads[r] + self.f.N:
                raise ProtocolViolation(f"LL128 step {p.step} overwrites line {p.line} of slot {p.slot} "
                                        f"before receiver lane {r} returned it (head {self.f.heads[r]})")
            n = len(p.values)
            self.f.lines[p.slot, p.line, p.w0:p.w0 + n] = np.array(p.values, np.uint64)
            self.f.owner[p.slot, p.line, p.w0:p.w0 + n] = p.step

    def state(self):
        return (self.step, self.line, self.granted, tuple(self.in_batch),
                tuple((p.slot, p.line, p.w0, p.values, p.step) for p in self.pending))


class LL128LaneReceiver(Actor):
    """Receiver lane r: reads its lines of every slot-step, each only once
    its flag is the step's (and then only words written in that step), and
    publishes its head = step + 1 after its last line of the step (at once
    for a step with none of its lines)."""

    def __init__(self, fifo: LL128LaneFifo, out: np.ndarray, lo: int, hi: int, lane: int):
        self.f, self.out, self.lo, self.hi, self.r = fifo, out, lo, hi, lane
        self.nwords = hi - lo
        self.base = fifo.heads[lane]
        self.nsteps = ceil_div(self.nwords, fifo.L * LL128_DATA_WORDS)
        self.l0 = min(lane * fifo.LgR, fifo.L)
        self.l1 = min(self.l0 + fifo.LgR, fifo.L)
        self.step = self.base
        self.line = self.l0
        self.name = f"ll128-recv-lane{lane}[{lo}:{hi}]"

    def _end(self, step):
        return min(self.l1, _ll128_lines(self.nwords, self.f.L, step - self.base))

    def done(self):
        return self.step >= self.base + self.nsteps

    def choices(self):
        if self.done():
            return []
        if self.line >= self._end(self.step):
            return [("head",)]
        k = self.step % self.f.N
        return [("read",)] if int(self.f.lines[k, self.line, LL128_DATA_WORDS]) == ll128_flag(self.step) else []

    def fire(self, choice):
        if choice[0] == "head":
            self.f.heads[self.r] = self.step + 1
            self.step += 1
            self.line = self.l0
            return
        k = self.step % self.f.N
        own = self.f.owner[k, self.line, :LL128_DATA_WORDS]
        stale = [int(o) for o in own if o != self.step]
        if stale:
            raise ProtocolViolation(f"LL128 line {self.line} of step {self.step} read with words from steps {stale}")
        g0 = ((self.step - self.base) * self.f.L + self.line) * LL128_DATA_WORDS
        n = min(LL128_DATA_WORDS, self.nwords - g0)
        self.out[self.lo + g0:self.lo + g0 + n] = self.f.lines[k, self.line, :n]
        self.line += 1

    def state(self):
        return (self.step, self.line)


# --------------------------------------------------------------------------
# Zero copy
# --------------------------------------------------------------------------

@dataclass
class DstHandle:
    """What the receiver publishes through ptrExchange: its buffer and offset."""
    buf: np.ndarray
    offset: int
    reads: int = 0


class ZeroCopyChannel:
    """head, tail and the ptrExchange word of one channel; the staging slots
    exist (poisoned) but zero copy must never touch them."""

    def __init__(self, nslots: int, slot_bytes: int, step0: int = 0, poison: int = 0xA5):
        self.N = nslots
        self.S = slot_bytes
        self.head = step0
        self.tail = step0
        self.ptr_exchange: DstHandle | None = None
        self.slots = np.full((nslots, slot_bytes), poison, np.uint8)
        self.max_occupancy = 0

    def check(self):
        occ = self.tail - self.head
        if occ < 0 or occ > self.N:
            raise ProtocolViolation(f"zero-copy tail {self.tail} head {self.head} N {self.N}")
        self.max_occupancy = max(self.max_occupancy, occ)

    def state(self):
        h = self.ptr_exchange
        return (self.head, self.tail, None if h is None else (h.offset, h.reads))


class ZeroCopyReceiver(Actor):
    """wait ptrExchange empty -> publish {dst, lo} -> per chunk: wait tail, store head."""
    WAIT_EMPTY, POST, WAIT, PUB, DONE = range(5)

    def __init__(self, ch: ZeroCopyChannel, dst: np.ndarray, lo: int, hi: int):
        self.c, self.dst, self.lo, self.hi = ch, dst, lo, hi
        self.base = ch.head
        self.nchunks = ceil_div(hi - lo, ch.S)
        self.j = 0
        self.phase = self.WAIT_EMPTY if self.nchunks else self.DONE
        self.name = f"zc-recv[{lo}:{hi}]"

    def done(self):
        return self.phase == self.DONE

    def choices(self):
        if self.phase == self.DONE:
            return []
        if self.phase == self.WAIT_EMPTY:
            return [0] if self.c.ptr_exchange is None else []
        if self.phase == self.WAIT:
            return [0] if self.c.tail > self.base + self.j else []
        return [0]

    def fire(self, choice):
        if self.phase == self.WAIT_EMPTY:
            self.phase = self.POST
        elif self.phase == self.POST:
            self.c.ptr_exchange = DstHandle(self.dst, self.lo)
            self.phase = self.WAIT
        elif self.phase == self.WAIT:
            self.phase = self.PUB
        elif self.phase == self.PUB:
            self.c.head = self.base + self.j + 1
            self.j += 1
            self.phase = self.WAIT if self.j < self.nchunks else self.DONE

    def state(self):
        return (self.j, self.phase)


class ZeroCopySender(Actor):
    """wait ptrExchange -> per chunk: wait credit, write src chunk into the
    published buffer, store tail -> wait final head -> empty ptrExchange.
    `fault`: "no_clear" (leave ptrExchange set)."""
    WAIT_PTR, WAIT, COPY, PUB, WAIT_FINAL, CLEAR, DONE = range(7)

    def __init__(self, ch: ZeroCopyChannel, src: np.ndarray, lo: int, hi: int, fault: str | None = None):
        self.c, self.src, self.lo, self.hi = ch, src, lo, hi
        self.base = ch.tail
        self.nchunks = ceil_div(hi - lo, ch.S)
        self.j = 0
        self.h: DstHandle | None = None
        self.phase = self.WAIT_PTR if self.nchunks else self.DONE
        self.fault = fault
        self.name = f"zc-send[{lo}:{hi}]"

    def done(self):
        return self.phase == self.DONE

    def choices(self):
        if self.phase == self.DONE:
            return []
        if self.phase == self.WAIT_PTR:
            return [0] if self.c.ptr_exchange is not None else []
        if self.phase == self.WAIT:
            return [0] if self.base + self.j < self.c.head + self.c.N else []
        if self.phase == self.WAIT_FINAL:
            return [0] if self.c.head == self.base + self.nchunks else []
        return [0]

    def fire(self, choice):
        if self.phase == self.WAIT_PTR:
            self.h = self.c.ptr_exchange
            self.h.reads += 1
            if self.h.reads != 1:
                raise ProtocolViolation("ptrExchange value consumed twice")
            self.phase = self.WAIT
        elif self.phase == self.WAIT:
            self.phase = self.COPY
        elif self.phase == self.COPY:
            off = self.j * self.c.S
            n = min(self.hi - self.lo - off, self.c.S)
            self.h.buf[self.h.offset + off:self.h.offset + off + n] = self.src[self.lo + off:self.lo + off + n]
            self.phase = self.PUB
        elif self.phase == self.PUB:
            self.c.tail = self.base + self.j + 1
            self.j += 1
            self.phase = self.WAIT if self.j < self.nchunks else self.WAIT_FINAL
        elif self.phase == self.WAIT_FINAL:
            self.phase = self.CLEAR
        elif self.phase == self.CLEAR:
            if self.fault != "no_clear":
                self.c.ptr_exchange = None
            self.phase = self.DONE

    def state(self):
        return (self.j, self.phase)


# --------------------------------------------------------------------------
# Receiver-driven credit FIFO ("RDMA and GPUDirect" §4.3, the sender FIFO;
# "NCCL transport data transfer (二)", netTransport copy and zero-copy modes)
# --------------------------------------------------------------------------

@dataclass
class Post:
    """One receiver post: chunk `idx - base - 1` may be written to
    buf[offset : offset + size]."""
    buf: np.ndarray
    offset: int
    size: int
    idx: int
    taken: bool = False


class PostedChannel:
    """The sender-side FIFO of N posts, the receiver-side completion queue and
    the receiver's N staging slots of S bytes.

    The receiver owns credit: it never has more than N posts outstanding
    (posted but not completed).  A post for chunk j of an operation carries
    idx = base + j + 1 (the pages' first index is 1 after a head of 0), so a
    FIFO entry left from an older post never matches.  `base` counts every
    chunk of earlier operations on the channel."""

    def __init__(self, nslots: int, slot_bytes: int, step0: int = 0):
        self.N = nslots
        self.S = slot_bytes
        self.slots = np.zeros(nslots * slot_bytes, np.uint8)
        self.posts: list[Post | None] = [None] * nslots
        self.cq: list[tuple[int, int] | None] = [None] * nslots   # (idx, size)
        self.posted = step0          # posts written (absolute chunk count)
        self.completed = step0       # chunks whose completion the receiver has consumed
        self.max_outstanding = 0

    def check(self):
        out = self.posted - self.completed
        if out < 0 or out > self.N:
            raise ProtocolViolation(f"{out} posts outstanding with N {self.N}")
        self.max_outstanding = max(self.max_outstanding, out)

    def state(self):
        return (self.posted, self.completed,
                tuple(None if q is None else (q.offset, q.size, q.idx, q.taken) for q in self.posts),
                tuple(self.cq), self.slots.tobytes())


class PostedReceiver(Actor):
    """Posts chunk j's landing place while fewer than N posts are outstanding,
    consumes completions in order and checks the size each one reports.

    direct=False (copy mode): the post names staging slot (base + j) mod N of
    S bytes; after the completion the receiver copies the slot to dst and only
    then counts the chunk consumed, which frees the slot for a new post.
    direct=True (zero copy): the post names dst itself, exactly the chunk's
    size.
    `fault`: "overpost" (ignores the N limit), "early_free" (copy mode: counts
    the chunk consumed before copying the slot out)."""

    def __init__(self, ch: PostedChannel, dst: np.ndarray, lo: int, hi: int, direct: bool = False,
                 fault: str | None = None):
        self.c, self.dst, self.lo, self.hi, self.direct = ch, dst, lo, hi, direct
        self.base = ch.completed
        self.nchunks = ceil_div(hi - lo, ch.S)
        self.next_post = 0
        self.next_done = 0
        self.landed = False          # copy mode: completion of next_done seen, slot not yet copied
        self.fault = fault
        self.name = f"posted-recv[{lo}:{hi}]"

    def _size(self, j):
        return min(self.c.S, self.hi - self.lo - j * self.c.S)

    def choices(self):
        if self.done():
            return []
        opts = []
        limit = self.next_done + (self.nchunks if self.fault == "overpost" else self.c.N)
        if self.next_post < self.nchunks and self.next_post < limit:
            opts.append(("post",))
        if self.landed:
            opts.append(("copy",))
        else:
            q = self.c.cq[(self.base + self.next_done) % self.c.N]
            if q is not None and q[0] == self.base + self.next_done + 1:
                opts.append(("complete",))
        return opts

    def fire(self, choice):
        N, S = self.c.N, self.c.S
        if choice[0] == "post":
            j = self.next_post
            k = (self.base + j) % N
            old = self.c.posts[k]
            if old is not None and not old.taken:
                raise ProtocolViolation(f"post {j} overwrites untaken post idx {old.idx}")
            if self.direct:
                self.c.posts[k] = Post(self.dst, self.lo + j * S, self._size(j), self.base + j + 1)
            else:
                self.c.posts[k] = Post(self.c.slots, k * S, S, self.base + j + 1)
            self.next_post += 1
            self.c.posted = self.base + self.next_post
        elif choice[0] == "complete":
            j = self.next_done
            idx, size = self.c.cq[(self.base + j) % N]
            if size != self._size(j):
                raise ProtocolViolation(f"completion of chunk {j} reports {size} bytes, expected {self._size(j)}")
            if self.direct:
                self._consumed()
            else:
                self.landed = True
                if self.fault == "early_free":
                    self.next_done += 1
                    self.c.completed = self.base + self.next_done
        else:
            j = self.next_done - (1 if self.fault == "early_free" else 0)
            k = (self.base + j) % N
            n = self._size(j)
            self.dst[self.lo + j * S:self.lo + j * S + n] = self.c.slots[k * S:k * S + n]
            self.landed = False
            if self.fault != "early_free":
                self._consumed()

    def _consumed(self):
        self.next_done += 1
        self.c.completed = self.base + self.next_done

    def done(self):
        return self.next_done >= self.nchunks and not self.landed

    def state(self):
        return (self.next_post, self.next_done, self.landed)


class PostedSender(Actor):
    """For chunk j: wait for the post whose idx is base + j + 1, check that the
    chunk fits its size, write the chunk at its address, then write the
    completion {idx, size} (the pages' write-with-immediate, whose immediate
    is the size).
    `fault`: "ignore_idx" (takes whatever post is in the FIFO entry)."""
    WAIT, COPY, COMPLETE, DONE = range(4)

    def __init__(self, ch: PostedChannel, src: np.ndarray, lo: int, hi: int, fault: str | None = None):
        self.c, self.src, self.lo, self.hi = ch, src, lo, hi
        self.base = ch.completed
        self.nchunks = ceil_div(hi - lo, ch.S)
        self.j = 0
        self.post: Post | None = None
        self.phase = self.WAIT if self.nchunks else self.DONE
        self.fault = fault
        self.name = f"posted-send[{lo}:{hi}]"

    def done(self):
        return self.phase == self.DONE

    def choices(self):
        if self.phase == self.DONE:
            return []
        if self.phase == self.WAIT:
            q = self.c.posts[(self.base + self.j) % self.c.N]
            ok = q is not None and (self.fault == "ignore_idx" or q.idx == self.base + self.j + 1)
            return [0] if ok else []
        return [0]

    def fire(self, choice):
        if self.phase == self.WAIT:
            q = self.c.posts[(self.base + self.j) % self.c.N]
            if q.taken:
                raise ProtocolViolation(f"post idx {q.idx} consumed twice")
            if q.idx != self.base + self.j + 1:
                raise ProtocolViolation(f"chunk {self.j} took post idx {q.idx}")
            q.taken = True
            self.post = q
            self.phase = self.COPY
        elif self.phase == self.COPY:
            off = self.lo + self.j * self.c.S
            n = min(self.c.S, self.hi - off)
            if n > self.post.size:
                raise ProtocolViolation(f"chunk of {n} bytes into a post of {self.post.size}")
            self.post.buf[self.post.offset:self.post.offset + n] = self.src[off:off + n]
            self.phase = self.COMPLETE
        else:
            n = min(self.c.S, self.hi - self.lo - self.j * self.c.S)
            self.c.cq[(self.base + self.j) % self.c.N] = (self.base + self.j + 1, n)
            self.j += 1
            self.phase = self.WAIT if self.j < self.nchunks else self.DONE

    def state(self):
        return (self.j, self.phase)


# --------------------------------------------------------------------------
# Copy-engine (proxy) mode ("NCCL transport data transfer (二)", p2pTransport
# cudaMemcopy mode (CE mode) and shmTransport useMemcpy mode)
# --------------------------------------------------------------------------

class CopyRing:
    """N slots of S bytes with the ownership checks of SimpleFifo: a slot is
    written only after its previous step was read out, and read only while it
    holds the step asked for."""

    def __init__(self, nslots: int, slot_bytes: int):
        self.N, self.S = nslots, slot_bytes
        self.slots = np.zeros((nslots, slot_bytes), np.uint8)
        self.owner = [None] * nslots
        self.consumed = [True] * nslots

    def put(self, step: int, data: np.ndarray, what: str):
        k = step % self.N
        if not self.consumed[k]:
            raise ProtocolViolation(f"{what}: step {step} overwrites slot {k} holding unread step {self.owner[k]}")
        self.slots[k, :len(data)] = data
        self.owner[k] = step
        self.consumed[k] = False

    def take(self, step: int, nbytes: int, what: str) -> np.ndarray:
        k = step % self.N
        if self.owner[k] != step or self.consumed[k]:
            raise ProtocolViolation(f"{what}: step {step} reads slot {k} holding step {self.owner[k]} "
                                    f"(read={self.consumed[k]})")
        self.consumed[k] = True
        return self.slots[k, :nbytes].copy()

    def state(self):
        return (self.slots.tobytes(), tuple(self.owner), tuple(self.consumed))


class CEFifo:
    """One channel of the proxy mode: the sender kernel fills ring 0 (its own
    send buffer) and publishes tails[0]; proxy hop h copies each step from
    ring h to ring h + 1 (one cudaMemcpy per step) and publishes tails[h + 1]
    once the copy has completed; the receiver kernel drains the last ring and
    returns head, the one credit counter of the chain.  hops = 1 is the p2p
    CE mode (send buffer -> receive buffer); hops = 2 is the shm useMemcpy
    mode (send buffer -> host shared buffer -> receive buffer).  The sender
    writes each step's size word before tails[0]; the hops copy that many
    bytes and the receiver checks it."""

    def __init__(self, nslots: int, slot_bytes: int, hops: int = 1, step0: int = 0):
        if nslots < 1 or slot_bytes < 1 or hops < 1:
            raise ValueError("need nslots, slot_bytes, hops >= 1")
        self.N, self.S, self.H = nslots, slot_bytes, hops
        self.rings = [CopyRing(nslots, slot_bytes) for _ in range(hops + 1)]
        self.tails = [step0] * (hops + 1)
        self.head = step0
        self.size = [-1] * nslots
        self.max_occupancy = 0

    def check(self):
        chain = self.tails + [self.head]
        for a, b in zip(chain, chain[1:]):
            if b > a:
                raise ProtocolViolation(f"counter chain out of order: {chain}")
        occ = self.tails[0] - self.head
        if occ > self.N:
            raise ProtocolViolation(f"tail {self.tails[0]} exceeds head {self.head} + N {self.N}")
        self.max_occupancy = max(self.max_occupancy, occ)

    def state(self):
        return (tuple(self.tails), self.head, tuple(self.size), tuple(r.state() for r in self.rings))


class _Stepper(Actor):
    """Walks steps base .. base + nsteps - 1 through a fixed order of phases."""
    DONE = -1

    def _start(self, base, nsteps, order):
        self.base, self.nsteps, self.order = base, nsteps, order
        self.step = base
        self.phase = order[0] if nsteps else self.DONE

    def done(self):
        return self.phase == self.DONE

    def _advance(self):
        i = self.order.index(self.phase)
        if i + 1 < len(self.order):
            self.phase = self.order[i + 1]
        else:
            self.step += 1
            self.phase = self.order[0] if self.step < self.base + self.nsteps else self.DONE

    def state(self):
        return (self.step, self.phase)


class CESender(_Stepper):
    """Per step: wait credit (step < head + N), fill send-ring slot and size
    word, publish tails[0].  `fault`: "skip_credit"."""
    WAIT, FILL, PUB = range(3)

    def __init__(self, fifo: CEFifo, src: np.ndarray, lo: int, hi: int, fault: str | None = None):
        self.f, self.src, self.lo, self.hi, self.fault = fifo, src, lo, hi, fault
        self._start(fifo.tails[0], ceil_div(hi - lo, fifo.S), (self.WAIT, self.FILL, self.PUB))
        self.name = f"ce-send[{lo}:{hi}]"

    def choices(self):
        if self.phase == self.DONE:
            return []
        if self.phase == self.WAIT:
            return [0] if self.fault == "skip_credit" or self.step < self.f.head + self.f.N else []
        return [0]

    def fire(self, choice):
        if self.phase == self.FILL:
            off = self.lo + (self.step - self.base) * self.f.S
            piece = self.src[off:min(self.hi, off + self.f.S)]
            self.f.rings[0].put(self.step, piece, "sender")
            self.f.size[self.step % self.f.N] = len(piece)
        elif self.phase == self.PUB:
            self.f.tails[0] = self.step + 1
        self._advance()


class CEProxy(_Stepper):
    """Hop h of the host proxy.  Per step: wait tails[h] > step, copy the
    step's size-word bytes from ring h to ring h + 1, and publish
    tails[h + 1] = step + 1 once that copy is complete.
    `fault`: "tail_before_copy" (publishes before the copy lands)."""
    WAIT, COPY, PUB = range(3)

    def __init__(self, fifo: CEFifo, hop: int, nsteps: int, fault: str | None = None):
        self.f, self.h, self.fault = fifo, hop, fault
        order = (self.WAIT, self.PUB, self.COPY) if fault == "tail_before_copy" else (self.WAIT, self.COPY, self.PUB)
        self._start(fifo.tails[hop + 1], nsteps, order)
        self.name = f"ce-proxy[{hop}]"

    def choices(self):
        if self.phase == self.DONE:
            return []
        if self.phase == self.WAIT:
            return [0] if self.f.tails[self.h] > self.step else []
        return [0]

    def fire(self, choice):
        if self.phase == self.COPY:
            n = self.f.size[self.step % self.f.N]
            if not 1 <= n <= self.f.S:
                raise ProtocolViolation(f"proxy hop {self.h}: size word {n} of step {self.step}")
            data = self.f.rings[self.h].take(self.step, n, f"proxy hop {self.h}")
            self.f.rings[self.h + 1].put(self.step, data, f"proxy hop {self.h}")
        elif self.phase == self.PUB:
            self.f.tails[self.h + 1] = self.step + 1
        self._advance()


class CEReceiver(_Stepper):
    """Per step: wait tails[H] > step, check the size word, copy the receive
    ring's slot to dst, publish head.  `fault`: "head_before_copy"."""
    WAIT, COPY, PUB = range(3)

    def __init__(self, fifo: CEFifo, dst: np.ndarray, lo: int, hi: int, fault: str | None = None):
        self.f, self.dst, self.lo, self.hi, self.fault = fifo, dst, lo, hi, fault
        order = (self.WAIT, self.PUB, self.COPY) if fault == "head_before_copy" else (self.WAIT, self.COPY, self.PUB)
        self._start(fifo.head, ceil_div(hi - lo, fifo.S), order)
        self.name = f"ce-recv[{lo}:{hi}]"

    def choices(self):
        if self.phase == self.DONE:
            return []
        if self.phase == self.WAIT:
            return [0] if self.f.tails[-1] > self.step else []
        return [0]

    def fire(self, choice):
        if self.phase == self.COPY:
            off = self.lo + (self.step - self.base) * self.f.S
            n = min(self.hi, off + self.f.S) - off
            if self.f.size[self.step % self.f.N] != n:
                raise ProtocolViolation(f"size word {self.f.size[self.step % self.f.N]} != {n}")
            self.dst[off:off + n] = self.f.rings[-1].take(self.step, n, "receiver")
        elif self.phase == self.PUB:
            self.f.head = self.step + 1
        self._advance()


# --------------------------------------------------------------------------
# Schedulers
# --------------------------------------------------------------------------

class System:
    """Endpoints plus the shared objects whose invariants are checked."""

    def __init__(self, actors: list[Actor], shared: list, buffers: list[np.ndarray] = ()):
        self.actors = list(actors)
        self.shared = list(shared)
        self.buffers = list(buffers)

    def options(self):
        return [(i, c) for i, a in enumerate(self.actors) for c in a.choices()]

    def all_done(self):
        return all(a.done() for a in self.actors)

    def check(self):
        for s in self.shared:
            s.check()

    def key(self):
        return (tuple(a.state() for a in self.actors), tuple(s.state() for s in self.shared),
                tuple(b.tobytes() for b in self.buffers))


def run(system: System, seed: int = 0, max_events: int | None = None) -> int:
    """Fire random enabled events (numpy default_rng(seed)) until every
    endpoint is done.  Returns the number of events fired."""
    rng = np.random.default_rng(seed)
    n = 0
    while True:
        opts = system.options()
        if not opts:
            if system.all_done():
                return n
            raise Deadlock("stuck: " + ", ".join(a.name for a in system.actors if not a.done()))
        i, c = opts[int(rng.integers(len(opts)))]
        system.actors[i].fire(c)
        system.check()
        n += 1
        if max_events is not None and n >= max_events:
            raise Deadlock(f"no completion within {max_events} events")


def explore(make_system, final_check, limit: int = 2_000_000) -> int:
    """Visit every state reachable by any interleaving of the endpoints'
    events (depth first, states deduplicated).  Checks the invariants in
    every state and `final_check(system)` in every terminal state; returns
    the number of distinct states."""
    start = make_system()
    start.check()
    stack = [start]
    seen = set()
    while stack:
        s = stack.pop()
        k = s.key()
        if k in seen:
            continue
        seen.add(k)
        if len(seen) > limit:
            raise RuntimeError("state space larger than limit")
        opts = s.options()
        if not opts:
            if not s.all_done():
                raise Deadlock("stuck state reached")
            final_check(s)
            continue
        for (i, c) in opts:
            t = copy.deepcopy(s)
            t.actors[i].fire(c)
            t.check()
            stack.append(t)
    return len(seen)
