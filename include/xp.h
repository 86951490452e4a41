/*
 * xp.h — C ABI of a single-GPU collective-transport data plane for GB300.
 *
 * A sender copies a user buffer, in slot-sized steps, into a bounded
 * circular FIFO and publishes a tail counter; a receiver waits on tail,
 * copies (or reduces) each slot into its destination and returns credit
 * through a head counter.  Every endpoint is a group of CTAs on one GPU.
 *
 * Sources (page title, section):
 *   [setup]    "NCCL transport setup" (gitcode.csdn.net): p2pRecvConnect wires
 *              tail (receiver memory), head (sender memory), ptrExchange and
 *              stepSize = buffSize / NCCL_STEPS; 具体说明 gives the ring
 *              neighbours; shmTransport places buffers and tail in host memory
 *              that the GPU reads directly; the receiver allocates the data
 *              buffers and tail, the sender only head.
 *   [transfer] "NCCL transport data transfer (二)" (cnnetsun.cn): p2pTransport
 *              zero copy through ptrExchange, copy mode (slot, tail, head),
 *              shmTransport normal mode.
 *   [rdma]     "RDMA and GPUDirect" (arganzheng.life) §4.1: the LL protocols
 *              put the flag in the data and the receiver polls memory; §7.2:
 *              4 MB channel buffers allocated once at connection time.
 *   [neuron]   "Intra-Node Transport (P2P)" (gh.evko.io) §4: POST/POLL on
 *              head/tail is device-only, the host does nothing.
 *
 * Conventions for every call:
 *   - Pointers named src/dst/send_bufs/recv_bufs are device pointers (or
 *     device-accessible mapped host pointers) owned by the caller; they must
 *     be 16-byte aligned and must stay valid until the operation completes
 *     on its stream.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream); every
 *     data-moving call is asynchronous on it and launches exactly one kernel
 *     and nothing else (xp_send_recv_staged: one per chunk, plus its copies;
 *     xp_send_recv_noalloc: one memset of its static FIFO's counters first;
 *     xp_ll_pingpong is synchronous).  The status block is not cleared
 *     between operations: each launch carries an operation id and the
 *     status words a kernel writes are tagged with it.
 *   - Operations on one FIFO (or one ring) must be ordered: issue them on one
 *     stream, or synchronise between them.  Step counters live on the device
 *     and carry over from one operation to the next, so captured CUDA graphs
 *     may be replayed.  A call made while its stream is being captured
 *     records no completion event: synchronise the stream a graph replays on
 *     before xp_fifo_status / xp_ring_status, and make the first call on a
 *     FIFO or ring outside any capture (it sets kernel attributes and
 *     queries occupancy).
 *   - Argument errors return immediately (no launch).  A CUDA error from a
 *     launch returns XP_ERR_CUDA (message in xp_last_error()).  Errors found
 *     on the device (a wait that timed out, a size word or occupancy out of
 *     bounds, an abort request) are reported by xp_fifo_status /
 *     xp_ring_status; after one, the object refuses further work (its next
 *     operations report XP_ERR_ABORTED) until xp_fifo_reset / xp_ring_reset.
 *   - No call allocates memory except *_create and xp_fifo_enable_ce; no call
 *     spins on the host except the *_status calls with sync != 0 and
 *     *_destroy (the proxy mode's own host thread aside).
 */
#ifndef XP_H
#define XP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Result codes, modelled on ncclResult_t ([setup]: ncclSuccess,
 * ncclInvalidArgument, ncclInternalError). */
typedef enum {
  XP_OK = 0,
  XP_ERR_INVALID = 1,   /* bad argument; nothing was launched            */
  XP_ERR_CUDA = 2,      /* a CUDA call failed; see xp_last_error()       */
  XP_ERR_TIMEOUT = 3,   /* a device wait exceeded the spin timeout       */
  XP_ERR_BOUNDS = 4,    /* a size word or tail-head distance was wrong   */
  XP_ERR_ABORTED = 5,   /* stopped by xp_abort() or an earlier error     */
  XP_ERR_INTERNAL = 6
} xp_status;

/* Protocols ([transfer] copy mode = SIMPLE; [rdma] §4.1 flag-in-data = LL
 * with 16-byte lines, LL128 with 128-byte lines). */
typedef enum { XP_PROTO_SIMPLE = 0, XP_PROTO_LL = 1, XP_PROTO_LL128 = 2 } xp_proto;

/* Where the FIFO (slots and counters) lives: device HBM, or pinned host
 * memory mapped into the device address space ([setup] shmTransport). */
typedef enum { XP_PLACE_DEVICE = 0, XP_PLACE_HOST_MAPPED = 1 } xp_placement;

/* Element types of the ring allreduce (add: IEEE fp32 round-to-nearest-even
 * without FMA or flush-to-zero; int32 wraps modulo 2^32). */
typedef enum { XP_U8 = 0, XP_U32 = 1, XP_I32 = 2, XP_F32 = 3, XP_BF16 = 4 } xp_dtype;

/* Which device wait reported an error (xp_report.where). */
typedef enum {
  XP_WAIT_NONE = 0, XP_WAIT_HEAD = 1, XP_WAIT_TAIL = 2, XP_WAIT_PTR_EXCHANGE = 3,
  XP_WAIT_LL_FLAG = 4, XP_WAIT_SLOT_BARRIER = 5, XP_WAIT_SIZE_WORD = 6, XP_WAIT_OCCUPANCY = 7,
  XP_WAIT_STICKY = 8, XP_WAIT_POST = 9, XP_WAIT_COMPLETION = 10
} xp_wait_site;

typedef struct xp_fifo xp_fifo;   /* opaque, owned by the library */
typedef struct xp_ring xp_ring;   /* opaque, owned by the library */
typedef struct CUstream_st* xp_stream_t;   /* same type as cudaStream_t */

/* Device-side outcome of the last operation on a FIFO or ring. */
typedef struct {
  int32_t code;            /* xp_status                                   */
  int32_t channel;         /* first channel (ring: rank*nchannels+channel) that failed, or -1 */
  int32_t where;           /* xp_wait_site                                */
  int32_t reserved;
  uint64_t observed;       /* counter value seen when the wait gave up    */
  uint64_t expected;       /* value it waited for                         */
  uint32_t max_occupancy;  /* largest tail - head a sender published      */
  uint32_t reserved2;
} xp_report;

/* Layout of one channel of a FIFO, for tests and tools (xp_fifo_describe).
 * ctl points at the channel's control block: uint64 tail at +0, uint64 head
 * at +128, uint64 ptrExchange at +256, uint64 step base at +384 and int64
 * size words (one per slot, -1 = never written) at +512; slots points at
 * slot 0, slot k at slots + k * slot_stride.  LL slots hold 16-byte lines
 * {data0, flag0, data1, flag1} (uint32 each); LL128 slots hold 128-byte
 * lines of 15 uint64 payload words and a uint64 flag (the last 8 bytes).  posted points at the
 * channel's receiver-driven credit FIFO (xp_send_recv_posted): 64 post
 * entries of 64 bytes {uint64 addr, uint64 size, uint64 idx, pad} at +0, 64
 * completion entries of 16 bytes {uint64 size, uint64 idx} at +4096 and the
 * uint64 step base of the next posted operation at +5120.  After
 * xp_fifo_enable_ce, ce points at the channel's proxy-mode block (mapped host
 * memory, device view) and send_ring / recv_ring at the channel's slot 0 of
 * the send ring and of the ring the receiver drains (NULL before). */
typedef struct {
  void* ctl;
  void* slots;
  size_t slot_stride;
  int nslots;
  int proto;
  int placement;
  int lanes;          /* sender CTAs per channel   */
  int recv_lanes;     /* receiver CTAs per channel */
  void* posted;
  void* ce;
  void* send_ring;
  void* recv_ring;
  int discard;        /* 1: the next operation's receivers drop the slot lines they read (xp_fifo_set_discard) */
} xp_channel_desc;

/* Create a FIFO of `nchannels` independent channels, each with `nslots`
 * slots of `slot_bytes` bytes ([setup] p2pRecvConnect: N steps of
 * buffSize / N bytes; [rdma] §7.2: allocated once, reused by every
 * transfer).  Counters start at 0 and size words at -1.
 *   1 <= nchannels <= 64, 1 <= nslots <= 64, slot_bytes a non-zero multiple
 *   of 16 (LL128: of 128-byte lines), nchannels * nslots * slot_bytes <= 2^40.
 * The library owns the memory (cudaMalloc, or cudaHostAlloc(Mapped|Portable)
 * for XP_PLACE_HOST_MAPPED) and frees it in xp_fifo_destroy.  The FIFO is
 * bound to the device current at creation.  Errors: XP_ERR_INVALID (bad
 * argument, *out untouched), XP_ERR_CUDA (allocation failed). */
xp_status xp_fifo_create(int nchannels, int nslots, size_t slot_bytes, xp_proto proto,
                         xp_placement place, xp_fifo** out);

/* Synchronise the device, then free the FIFO.  NULL is a no-op. */
xp_status xp_fifo_destroy(xp_fifo* f);

/* CTAs per channel side: each channel's sender and receiver are each spread
 * over CTAs ("lanes") that share the channel's one tail and one head (default
 * 1: one sender CTA and one receiver CTA per channel).  Sets the sender side
 * to `lanes` (1 <= lanes <= 32) and the receiver side to lanes if lanes <= 8,
 * else to max(1, 16 - lanes); zero copy and direct posted transfers always use
 * one receiver CTA.  HBM FIFOs: the lanes of a side meet on per-slot arrival
 * counters in device memory, and an operation runs as one cooperative grid
 * when nchannels x (sender + receiver CTAs) are resident on the GPU at once,
 * else as one thread-block cluster per channel, which needs sender + receiver
 * CTAs <= 16; an operation that fits neither way is refused (XP_ERR_INVALID).
 * Host-placed FIFOs always use clusters.  LL128 FIFOs: 1 <= lanes <= 8
 * sender and as many receiver CTAs per channel (xp_fifo_set_recv_lanes may
 * then change the receiver side), sender lane g moving the fixed stripe of
 * ceil(L / lanes) of each slot's L lines and receiver lane r that of
 * ceil(L / rlanes) lines with a head of its own; a sender lane refills its
 * stripe of a slot once every receiver lane whose stripe meets it has
 * returned the credit.  The channel's CTAs run as one cooperative grid when
 * nchannels x (lanes + rlanes) are resident at once, else as one cluster
 * per channel (lanes + rlanes <= 16).  At the end of an operation every
 * lane's head equals the channel's step base, so the counts may change from
 * one operation to the next.  LL FIFOs: refused.  Takes effect at the next
 * operation. */
xp_status xp_fifo_set_lanes(xp_fifo* f, int lanes);

/* Receiver CTAs per channel of xp_send_recv, independently of the sender's
 * (SIMPLE: 1 <= rlanes <= 32; LL128: 1 <= rlanes <= 8; the launch rules of
 * xp_fifo_set_lanes apply): the slot-step is published whole (SIMPLE) or
 * line by line (LL128), so the receiver may cut it into a different number
 * of stripes (also for copy-mode posted and proxy transfers).  Zero copy and
 * direct posted transfers always use one receiver CTA.  LL FIFOs: refused.
 * Takes effect at the next operation (xp_fifo_set_lanes resets it). */
xp_status xp_fifo_set_recv_lanes(xp_fifo* f, int rlanes);

/* Whether receivers that read FIFO slots in HBM drop each 128-byte line of
 * their stripe from L2 (discard.global.L2) once they have read it — the data
 * is dead, and this saves writing it back to DRAM when L2 would evict it
 * before the slot is refilled — (on > 0), leave it (on == 0), or choose by
 * the FIFO's size (on < 0, the default): drop when nchannels * nslots *
 * slot_bytes >= XP_DISCARD_AUTO_BYTES, whose lines compete for L2 with the
 * user buffers streaming through; a smaller FIFO's lines are rewritten
 * before eviction, and the drops would only delay its credit.  With drops on,
 * the slots' bytes after a transfer are undefined; with them off they hold
 * the last slot-steps that passed through, as in the pages' protocol.
 * Applies to xp_send_recv, copy-mode xp_send_recv_posted and xp_send_recv_ce
 * on HBM FIFOs; takes effect at the next operation; xp_fifo_describe reports
 * the choice. */
#define XP_DISCARD_AUTO_BYTES ((size_t)48 << 20)
xp_status xp_fifo_set_discard(xp_fifo* f, int on);

/* Channel layout (pointers stay valid until destroy). */
xp_status xp_fifo_describe(const xp_fifo* f, int channel, xp_channel_desc* out);

/* Copy `bytes` bytes from src to dst through the FIFO ([transfer] copy mode;
 * [neuron] §4 POST/POLL).  The buffer is cut into channels of
 * round_up(ceil(bytes / nchannels), 16) bytes (the last ones shorter or
 * empty); each channel moves its range in slot-steps of slot_bytes:
 * sender: wait step < head + nslots, copy into slot step % nslots, write the
 * slot's size word, publish tail = step + 1 (release); receiver: wait
 * tail > step (acquire), check the size word, copy out, publish head =
 * step + 1.  XP_PROTO_SIMPLE: any byte count; XP_PROTO_LL: bytes a multiple
 * of 8, sent as 16-byte lines {d0, flag, d1, flag} with flag = step + 1 and
 * no tail ([rdma] §4.1).  XP_PROTO_LL128: bytes a multiple of 8; slot-step
 * s carries 15 * slot_bytes / 128 payload words, line i of it the next 15
 * (zeros past the end) and the uint64 flag s + 1 in its last 8 bytes; the
 * sender makes a batch of lines' payload visible (fence) before it writes
 * their flags and the receiver reads a line only after its flag (fence); no
 * tail.  src and dst must not overlap.  bytes == 0 is a no-op returning
 * XP_OK. */
xp_status xp_send_recv(xp_fifo* f, const void* src, void* dst, size_t bytes, xp_stream_t stream);

/* Zero-copy transfer ([transfer] zero copy, address known only at run time):
 * per channel the receiver publishes dst + channel offset into the
 * channel's ptrExchange word once it is empty; the sender reads it and
 * writes src straight into dst in chunks of at most slot_bytes, publishing
 * tail per chunk (credit as in xp_send_recv); the receiver returns head per
 * chunk; the sender empties ptrExchange after the last head.  The FIFO's
 * slots are not touched.  SIMPLE FIFOs only; any byte count. */
xp_status xp_send_recv_zero_copy(xp_fifo* f, const void* src, void* dst, size_t bytes,
                                 xp_stream_t stream);

/* Transfer with receiver-driven credit ([rdma] §4.3: the receiver tells the
 * sender where to write through a FIFO of {addr, size, idx} entries;
 * [transfer] netTransport copy and zero-copy modes).  Per channel (split as
 * in xp_send_recv) the receiver keeps up to nslots posts outstanding: post j
 * of an operation carries idx = base + j + 1, where base counts the channel's
 * chunks of all earlier posted operations, and names where chunk j (at most
 * slot_bytes bytes) may land.  The sender waits for the post whose idx is
 * base + j + 1 in FIFO entry (base + j) % nslots, checks that the chunk fits
 * its size and that its address is 16-byte aligned (else XP_ERR_BOUNDS,
 * where = XP_WAIT_POST), writes the chunk there and then the completion
 * {size, idx} into completion entry (base + j) % nslots; the receiver takes
 * the completions in order, checks each size (else XP_ERR_BOUNDS, where =
 * XP_WAIT_COMPLETION) and posts chunk j + nslots once chunk j is consumed.
 *   direct == 0 (copy mode): posts name the FIFO's staging slots, whole; the
 *     receiver copies each landed slot to dst, then re-posts it.  Uses the
 *     FIFO's lanes and receiver lanes.
 *   direct != 0: posts name dst itself, exactly the chunk; the slots are not
 *     touched.  One receiver CTA per channel.
 * Head, tail, size words and ptrExchange are not used, so posted and other
 * operations may alternate on one FIFO.  SIMPLE FIFOs in device memory only
 * (XP_ERR_INVALID otherwise); any byte count; src and dst must not overlap. */
xp_status xp_send_recv_posted(xp_fifo* f, const void* src, void* dst, size_t bytes, int direct,
                              xp_stream_t stream);

/* Set up the proxy (copy-engine) mode on a SIMPLE FIFO ([transfer]
 * p2pTransport cudaMemcopy mode and shmTransport useMemcpy mode): allocates
 * the sender's own send ring in device memory (same geometry as the FIFO's
 * slots), for a host-placed FIFO also a receive ring in device memory, and
 * per channel a 2 KiB block in mapped host memory (uint64 tail[h] at +128 h
 * for h = 0..2, uint64 head at +384, uint64 step base at +512, int64 size
 * words at +640), and starts a host thread (the pump) that serves every
 * later xp_send_recv_ce on this FIFO until xp_fifo_destroy.  Device FIFO:
 * one hop per slot-step, send ring -> the FIFO's slots.  Host-placed FIFO:
 * two hops, send ring -> the FIFO's slots in host memory -> receive ring.
 * Calling it again is a no-op.  Errors: XP_ERR_INVALID (not SIMPLE),
 * XP_ERR_CUDA (allocation or thread setup failed). */
xp_status xp_fifo_enable_ce(xp_fifo* f);

/* Transfer through the proxy mode (after xp_fifo_enable_ce).  Channels and
 * slot-steps as in xp_send_recv.  The sender CTAs fill send-ring slot
 * step % nslots, write its size word and publish tail[0] = step + 1 at
 * system scope, under the credit step < head + nslots; for each hop h the
 * pump copies the step's size-word bytes from ring h to ring h + 1 with
 * cudaMemcpyAsync on its own stream and publishes tail[h + 1] = step + 1 once
 * that copy has completed; the receiver CTAs wait for the last tail, check
 * the size word, copy the slot out to dst and publish head.  A size word
 * outside [1, slot_bytes] stops the pump (the transfer then times out and
 * xp_fifo_status leaves the pump's message in xp_last_error()).  The pump
 * keeps serving while the FIFO exists, so captured graphs replay.  Proxy
 * operations keep their own counters; other operations may alternate with
 * them on the FIFO.  The transfer's kernel waits for the pump's copies, so
 * while it is in flight the process should not queue copies that wait for
 * it (for example a cudaMemcpy on the stream it runs on, or on the legacy
 * default stream when it runs there): such a copy can share a copy queue
 * with the pump's and hold them up until the transfer stops at its spin
 * timeout.  This library's own set-up calls never do (they use streams of
 * their own), so objects may be created, reset or destroyed meanwhile. */
xp_status xp_send_recv_ce(xp_fifo* f, const void* src, void* dst, size_t bytes, xp_stream_t stream);

/* xp_send_recv from host memory to host memory, staged through device
 * buffers the caller owns.  The pages have no counterpart: it is the
 * end-to-end form of a transfer, for callers whose data lives on the host.
 * host_src / host_dst should be pinned (cudaHostAlloc or registered), else the
 * copies are not asynchronous; dev_src / dev_dst are device buffers of `bytes`
 * bytes, 16-byte aligned, not overlapping.  The buffer is cut into chunks of
 * chunk_bytes (0 = 64 MiB; a multiple of 16); chunk i is copied host ->
 * device on a stream of the FIFO's own, moved by one xp_send_recv on
 * `stream`, and copied device -> host on a second stream of the FIFO's own,
 * so the two copy directions and the transfers of neighbouring chunks
 * overlap.  Everything starts after the work already on `stream`, and
 * `stream` waits for the last copy out: the call is asynchronous on `stream`
 * like the others.  Errors as xp_send_recv; a device error in one chunk makes
 * the later chunks refuse (xp_fifo_status then reports XP_ERR_ABORTED). */
xp_status xp_send_recv_staged(xp_fifo* f, const void* host_src, void* host_dst, void* dev_src, void* dev_dst,
                              size_t bytes, size_t chunk_bytes, xp_stream_t stream);

/* Outcome of the FIFO's last operation.  sync != 0 first waits for the
 * FIFO's last stream; sync == 0 reads whatever the device has written so far
 * (XP_OK if the operation is still running without error).  `report` may be
 * NULL.  Returns the device code (XP_OK, XP_ERR_TIMEOUT, ...). */
xp_status xp_fifo_status(xp_fifo* f, int sync, xp_report* report);

/* Per-channel record of the FIFO's last operation (after it completes):
 * slot-steps moved, the device clock (globaltimer, ns) when the channel's
 * sender side started and when its receiver side published its last step,
 * and how often each side's watcher thread polled its remote counter (0 for
 * sides and kernels without one).  Waits for the FIFO's last operation. */
typedef struct {
  uint64_t steps;
  uint64_t t_start_ns;
  uint64_t t_end_ns;
  uint64_t send_polls;
  uint64_t recv_polls;
} xp_channel_stats;
xp_status xp_fifo_stats(xp_fifo* f, int channel, xp_channel_stats* out);

/* Zero the FIFO's counters, size words, ptrExchange and error state
 * (synchronous); needed after a device error. */
xp_status xp_fifo_reset(xp_fifo* f);

/* LL ping-pong for one-way latency: `iters` round trips of one 8-byte line,
 * A -> B through `ab` and B -> A through `ba` (two LL FIFOs, channel 0 of
 * each), between two CTAs of one cluster; the device clock (globaltimer)
 * brackets the loop.  Writes the round-trip total in ns to *elapsed_ns
 * (synchronous; 1 <= iters <= 1e7). */
xp_status xp_ll_pingpong(xp_fifo* ab, xp_fifo* ba, int iters, uint64_t* elapsed_ns,
                         xp_stream_t stream);

/* Create the FIFOs of a virtual ring of `nranks` ranks in this GPU's memory
 * ([setup] 具体说明: rank r receives from r-1 and sends to r+1): for each
 * rank and channel one SIMPLE FIFO of nslots x slot_bytes owned by the
 * receiving rank.  2 <= nranks <= 16 (the ranks of a channel share one
 * cluster), 1 <= nchannels <= 64, 2 <= nslots <= 64, slot_bytes a non-zero
 * multiple of 16. */
xp_status xp_ring_create(int nranks, int nchannels, int nslots, size_t slot_bytes, xp_placement place,
                         xp_ring** out);
xp_status xp_ring_destroy(xp_ring* r);

/* CTAs per rank per channel (0 <= lanes <= 8; default 0).  0 = chosen at
 * each operation: an HBM ring runs its channels in groups, one launch per
 * group, so that the FIFO data a launch keeps live (nranks * nslots/2 *
 * slot_bytes per channel) stays within 32 MiB of L2, and gives each group the
 * largest lane count (at most 8) whose whole grid of group * lanes * nranks
 * CTAs is resident on the GPU at once, at least 1 (8 ranks x 8 channels of
 * 8 x 512 KiB: 4 launches of 2 channels at 8 lanes); a host-placed ring
 * takes 1 lane.  Explicit lanes run every channel in one launch.  HBM rings: lane g
 * moves the g-th 16-byte aligned stripe of every slot-step of every FIFO,
 * with a control block of its own per FIFO (the lanes of a channel are
 * independent rings over disjoint stripes; the result does not depend on
 * the lane count).  The ranks of a lane's ring must run at once: a grid
 * that is resident as a whole is launched cooperatively, a larger one as one
 * cluster of nranks CTAs per channel and lane.
 * Host-placed rings: the lanes of a rank share its counters, one cluster of
 * nranks * lanes CTAs per channel, so nranks * lanes <= 16. */
xp_status xp_ring_set_lanes(xp_ring* r, int lanes);

/* Allreduce (sum) of `count` elements of type dt (XP_F32 or XP_I32) over the
 * ring's ranks: send_bufs[r] / recv_bufs[r] are rank r's input and output
 * (host arrays of nranks device pointers; in place allowed).  Elements are
 * cut into channels (16-byte aligned, as xp_send_recv); each channel range is
 * walked in rounds of nranks chunks of (nslots / 2) * slot_bytes bytes (the
 * last round shrinks them).  Per round rank r runs send(chunk r-1),
 * recvReduceSend(chunk r-j) for j = 2..P-1, recvReduceCopySend(chunk r),
 * recvCopySend(chunk r+1-j) for j = 2..P-1 and recv(chunk r+1), each moved in
 * slot-steps through its FIFOs, so element i of chunk k ends as
 * ((x[k+1] + x[k+2]) + ...) + x[k] on every rank. */
xp_status xp_ring_allreduce_virtual(xp_ring* r, const void* const* send_bufs, void* const* recv_bufs,
                                    size_t count, xp_dtype dt, xp_stream_t stream);

xp_status xp_ring_status(xp_ring* r, int sync, xp_report* report);
xp_status xp_ring_reset(xp_ring* r);

/* SIMPLE transfer that allocates nothing.  The pages have no counterpart:
 * it exists for callers that must not allocate device memory while they run,
 * e.g. code inside a memory-pool or allocator hook (cudaMalloc there could
 * re-enter the allocator) or under a hard device-memory budget.  The caller
 * passes src and dst as for xp_send_recv; the FIFO (control blocks, slots,
 * status) lives in one static device array of this library, 8 MiB of slots
 * plus 32.25 KiB, that every GPU which loads the library keeps reserved until
 * the process exits.  Limits: 1 <= nchannels <= 16, 1 <= nslots <= 64,
 * slot_bytes a non-zero multiple of 16, and nchannels x
 * round_up(nslots x slot_bytes, 4096) <= 8 MiB; larger FIFOs are refused with
 * XP_ERR_INVALID and a message in xp_last_error().  One sender CTA and one
 * receiver CTA per channel; the default 2 s spin timeout; the host abort
 * word is not polled.  Each call clears the array's counters and status,
 * launches one kernel on `stream` and, if dev_status (a device pointer) is
 * not NULL, copies the device-side xp_status of the transfer there
 * asynchronously.  All calls share the one array: calls whose transfers
 * overlap in time on the GPU (other streams, other host threads) race and
 * corrupt each other.  Every call looks up the array's device address
 * (cudaGetSymbolAddress, with the caller's device current); the first call
 * on a device also sets a kernel attribute, so make it before any stream
 * capture.  Nothing here calls cudaMalloc, cudaFree or an allocating
 * library routine. */
xp_status xp_send_recv_noalloc(const void* src, void* dst, size_t bytes, int nchannels, int nslots,
                               size_t slot_bytes, int32_t* dev_status, xp_stream_t stream);

/* Spin timeout of every device wait in later launches, in ns (default 2e9,
 * or XP_SPIN_TIMEOUT_NS from the environment when the library loads;
 * 1e3 <= ns <= 6e10). */
xp_status xp_set_spin_timeout_ns(uint64_t ns);

/* Set (value != 0) or clear the process-wide abort word, which lives in
 * mapped host memory and is polled by every device wait: running and later
 * operations stop with XP_ERR_ABORTED while it is set. */
xp_status xp_abort(int value);

const char* xp_status_string(xp_status s);
/* Message of the last error on the calling thread ("" if none). */
const char* xp_last_error(void);
int xp_version(void);

#ifdef __cplusplus
}
#endif
#endif /* XP_H */
