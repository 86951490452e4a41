// Definitions shared by the host library and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include "xp.h"

namespace xp {

constexpr int kMaxSlots = 64;
constexpr int kMaxChannels = 64;
constexpr int kMaxRanks = 16;
constexpr int kMaxCluster = 16;
constexpr int kMaxLanes = 32;     // CTAs per side of a channel (bulk-copy channel kernel)

// Per-channel control block: every word the two sides write sits on its own
// 128-byte line, so the producer's tail stores and the consumer's head stores
// never share a line (and neither shares one with the size words).
constexpr int kCtlBytes = 1024;
constexpr int kTailOff = 0;     // producer cursor (lives with the receiver)
constexpr int kHeadOff = 128;   // consumer cursor / credit (lives with the sender)
constexpr int kPtrxOff = 256;   // ptrExchange: receiver's destination for zero copy
constexpr int kBaseOff = 384;   // first step of the next operation (device-side epoch)
constexpr int kSizeOff = 512;   // int64 size word per slot, -1 = never written

// Per-channel block of the receiver-driven credit FIFO (posted transfers):
// kMaxSlots post entries of 64 bytes {addr, size, idx, pad}, written by the
// receiver and read by the sender; kMaxSlots completion entries of 16 bytes
// {size, idx}, written by the sender; and the step base of the next posted
// operation on its own line.
constexpr int kPostCtlBytes = 8192;
constexpr int kPostOff = 0;
constexpr int kComplOff = 64 * kMaxSlots;
constexpr int kPostBaseOff = kComplOff + 16 * kMaxSlots;

// Per-channel block of the proxy (copy-engine) mode, in mapped host memory:
// tail[h] for h = 0 .. 2 on their own lines (tail[0] written by the sender
// kernel, tail[h + 1] by the host pump once hop h's copy of a step has
// completed), head (written by the receiver kernel), the step base of the
// next proxy operation, and the sender's int64 size word per slot.
constexpr int kCeCtlBytes = 2048;
constexpr int kCeMaxHops = 2;
constexpr int kCeTailOff = 0;          // tail[h] at kCeTailOff + 128 h
constexpr int kCeHeadOff = 384;
constexpr int kCeBaseOff = 512;
constexpr int kCeSizeOff = 640;        // kMaxSlots int64 size words

// Per-channel arrival counters of the bulk-copy channel kernel's lanes: one
// uint64 per slot for the sender side, then one per slot for the receiver
// side; zero between operations.
constexpr int kArrBytes = 16 * kMaxSlots;

constexpr int kCopyWarps = 16;                  // data-moving warps per CTA
constexpr int kP2pThreads = 32 * (kCopyWarps + 1);   // + 1 publisher warp
constexpr int kRingThreads = 32 * (kCopyWarps + 2);  // + tail and head publishers
constexpr int kLLThreads = 32 * (kCopyWarps + 1);

// Device-side status of an object's operations (device memory).  Nothing
// clears it between operations (a memset would be one more GPU operation per
// call): every launch carries an operation id (the object's count of
// launches) and the words an operation writes are tagged with it.  A failure
// claims `claim` = (id << 32) | code unless this operation already holds it,
// then fills channel, where, observed and expected, and sets `sticky` and
// `abort`; while `sticky` is set (until a reset zeroes the block) every
// operation is refused and claims ABORTED.  The host reports `claim` and the
// occupancy word only when their id matches `last_op`, which the first CTA
// of every operation writes as it starts.
struct DevStatus {
  unsigned long long claim;       // (op << 32) | code of the operation's first failure
  int channel;
  int where;
  unsigned long long observed;
  unsigned long long expected;
  unsigned long long occupancy;   // (op << 32) | largest tail - head a sender published in operation op
  unsigned long long last_op;     // id of the last operation that started
  int abort;                      // set by the first failing wait: the others stop early
  int pad0;
  unsigned long long elapsed;     // ping-pong: round-trip total, ns
  int sticky;                     // +64
  int pad2[15];
};
static_assert(sizeof(DevStatus) == 128, "status block layout");

// Per-channel record of the last operation (device memory, one per channel),
// written by the channel kernel: slot-steps moved, device time (globaltimer)
// when the sender side started and when the receiver side published its last
// step, and how many times each side's watcher polled its remote counter.
struct ChanStats {
  unsigned long long steps;
  unsigned long long t_start;
  unsigned long long t_end;
  unsigned long long send_polls;
  unsigned long long recv_polls;
  unsigned long long pad[3];
};
static_assert(sizeof(ChanStats) == 64, "stats record layout");

struct P2pParams {
  char* ctl;                      // nchannels control blocks
  unsigned long long* arr;        // nchannels arrival blocks (bulk-copy channel kernel)
  ChanStats* stats;               // nchannels records, or nullptr
  char* pctl;                     // nchannels posted-FIFO blocks (posted transfers)
  char* ce;                       // nchannels proxy-mode blocks (mapped host memory)
  char* send_ring;                // proxy mode: the sender's own slots, same geometry as `slots`
  char* recv_ring;                // proxy mode: the slots the receiver drains
  int hops;                       // proxy mode: host-driven copies per slot-step (1 or 2)
  int discard;                    // receivers drop read slot lines from L2 (bulk-copy kernel)
  char* slots;                    // channel c's slot k at slots + c*ch_stride + k*slot_bytes
  unsigned long long ch_stride;
  const char* src;
  char* dst;
  unsigned long long nbytes;
  int nchannels;
  int nslots;
  int lanes;                      // sender CTAs per channel
  int rlanes;                     // receiver CTAs per channel (SIMPLE, HBM FIFO)
  int csize;                      // cluster size
  unsigned int slot_bytes;
  DevStatus* status;
  const volatile int* abort_word; // mapped host memory
  unsigned long long timeout_ns;
  unsigned long long op;          // operation id (DevStatus)
};

struct PingParams {
  char* ctl_ab;
  char* slots_ab;
  char* ctl_ba;
  char* slots_ba;
  int nslots_ab;
  int nslots_ba;
  unsigned int slot_bytes_ab;
  unsigned int slot_bytes_ba;
  int iters;
  unsigned long long* elapsed;    // device word
  DevStatus* status;
  const volatile int* abort_word;
  unsigned long long timeout_ns;
  unsigned long long op;
};

// Ring FIFOs keep kRingMaxLanes control blocks each: lane g of FIFO f (the
// bulk-copy ring's independent lanes) uses block f * kRingMaxLanes + g.
constexpr int kRingMaxLanes = 8;

struct RingParams {
  char* ctl;                      // FIFO (c, r) lane g control block at ctl + ((c*nranks + r)*kRingMaxLanes + g)*kCtlBytes
  char* slots;                    // its slots at slots + (c*nranks + r)*fifo_stride
  unsigned long long fifo_stride;
  const char* send[kMaxRanks];
  char* recv[kMaxRanks];
  unsigned long long count;
  int nranks;
  int nchannels;
  int nslots;
  int lanes;
  int c_first;                    // bulk-copy ring: first channel of this launch (a launch may run a group of channels)
  int dtype;                      // XP_F32 or XP_I32
  unsigned int slot_bytes;
  DevStatus* status;
  const volatile int* abort_word;
  unsigned long long timeout_ns;
  unsigned long long op;
};

}  // namespace xp
