"""CPU oracle for the FIFO data plane — TEST INFRASTRUCTURE ONLY.

A plain, slow, single-threaded simulation of the collective transport's
device-side producer/consumer protocol (SIMPLE slots with head/tail, LL and
LL128 lines with inline flags, zero copy through ptrExchange, the host-placed
FIFO, and the virtual ring allreduce), written from the pages' descriptions.  It shares no
code with the CUDA path and never imports it.

Only `tests/`, `__graft_entry__.smoke()` and `bench.py`'s CPU-baseline /
reference leg may import or run anything in this package.  The library itself
never routes through it: there is no CPU fallback.

Entry points:
* `simple_transfer`, `ll_transfer`, `ll128_transfer`, `zero_copy_transfer`,
  `posted_transfer`, `ce_transfer`:
  move a buffer through C channels under a seeded random interleaving and
  return the result;
* `ring_allreduce`: the ring as state machines; `ring_order_sum`: the plain
  definition of its result;
* `fifo.explore`: every interleaving of a tiny system.

Pins (tests/test_oracle_*.py): byte identity of every copy path, exhaustive
interleavings for N in {1, 2} with up to 4 slot-steps, planted protocol
mistakes that the checks must catch, the ring result against exact rational
arithmetic rounded to fp32, against int64 sums for int32, against the
fp64 sum within the standard error bound, and the pages' printed sizes and
ring-neighbour example (tests/golden/).
"""
from .fifo import (CEFifo, CEProxy, CEReceiver, CESender, Deadlock, LL128Fifo, LL128LaneFifo, LL128LaneReceiver,
                   LL128LaneSender, LL128Receiver, LL128Sender, LLFifo, LLReceiver, LLSender, PostedChannel, PostedReceiver, PostedSender,
                   ProtocolViolation, SimpleFifo, SimpleReceiver, SimpleSender, System, ZeroCopyChannel,
                   ZeroCopyReceiver, ZeroCopySender, explore, ll128_flag, ll_flag, run)
from .partition import (channel_byte_ranges, ring_channel_ranges, ring_chunk_elems, ring_next,
                        ring_prev, ring_rounds, ring_schedule, slot_steps)
from .ring import ring_order_sum, ring_system
from .transfer import (ce_transfer, ll128_transfer, ll_transfer, posted_transfer, ring_allreduce, simple_transfer,
                       zero_copy_transfer)

__all__ = [
    "Deadlock", "ProtocolViolation", "SimpleFifo", "SimpleSender", "SimpleReceiver", "LLFifo",
    "LLSender", "LLReceiver", "ZeroCopyChannel", "ZeroCopySender", "ZeroCopyReceiver", "System",
    "run", "explore", "ll_flag", "channel_byte_ranges", "slot_steps", "ring_prev", "ring_next",
    "ring_channel_ranges", "ring_chunk_elems", "ring_rounds", "ring_schedule", "ring_order_sum",
    "ring_system", "simple_transfer", "ll_transfer", "zero_copy_transfer", "ring_allreduce",
    "PostedChannel", "PostedSender", "PostedReceiver", "posted_transfer",
    "CEFifo", "CESender", "CEProxy", "CEReceiver", "ce_transfer",
    "LL128Fifo", "LL128Sender", "LL128Receiver", "ll128_flag", "ll128_transfer",
    "LL128LaneFifo", "LL128LaneSender", "LL128LaneReceiver",
]
