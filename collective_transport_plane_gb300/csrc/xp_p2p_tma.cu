// Channel kernel for FIFOs in HBM, data moved with bulk (TMA) copies through
// shared memory: SIMPLE, zero copy, receiver-driven credit (copy and direct
// modes) and the proxy (copy-engine) mode, one template instance each.
//
// Per channel, CTAs [0, G) send and [G, G + GR) receive (zero copy and direct
// posts: CTA G receives), consecutive in the grid.  The lanes of a side share
// the channel's counters through per-slot arrival counters in global memory,
// so no thread-block cluster is needed: the host launches the grid
// cooperatively when all of it is resident at once (sender and receiver CTAs
// that wait on each other must run together), else as one cluster per
// channel.  Each CTA moves one contiguous stripe of every slot-step
// ("lane") through a ring of kTmaStages shared-memory stages:
//   sender    - one mover thread issues bulk loads from src up to kLookSend
//               entries ahead (they need nothing) and bulk stores into the
//               slot (they need credit);
//   receiver  - a loader thread waits for tail and bulk-loads the slot into
//               free stages, a storer thread bulk-stores each stage into dst
//               and frees it, so neither stream waits for the other's
//               memory latency;
//   watcher   - polls the one remote counter the CTA waits on (sender: head,
//               or the posts; receiver: tail, or the completions) and
//               mirrors it into shared memory, so no copying thread stalls on
//               a global-memory round trip;
//   prefetcher - sender side: asks L2 to fetch src a bulk entry or two
//               beyond the mover's loads (cp.async.bulk.prefetch);
//   discarder - receiver side: drops the slot lines its stripe has read
//               from L2;
//   publisher - in the side's leader CTA only: waits until all lanes have
//               signalled a slot-step on its arrival counter and publishes the one
//               channel-wide counter (tail = step + 1 on the sender side,
//               head = step + 1 on the receiver side; posted modes: the
//               completion, or the next post).  A side of one lane has
//               nothing to aggregate: its publisher takes the signals from
//               shared memory, a global-memory round trip shorter.
// A sender stripe is signalled once its bulk stores have completed.  The mover
// checks that only after the first store of the next step is in flight, so the
// store pipeline never drains at a step boundary, and before it blocks on
// credit it reports whatever is pending (a FIFO of one slot would otherwise
// wait on itself).  It reports through shared memory to a signaler thread,
// which does the release add on the arrival counter: a release waits for the
// issuing thread's in-flight memory traffic, and the mover always has some.
// A receiver stripe is signalled as soon as its bulk loads from the slot have
// landed in shared memory.  Slot traffic keeps L2's normal priority and
// user-buffer traffic is marked evict_first, so the FIFO stays L2-resident
// while src and dst stream through.
#include <cuda_runtime.h>

#include "xp_device.cuh"

namespace xp {

// Three stages of 32 KiB: 96 KiB of shared memory, so two CTAs fit on an SM
// (the 16-channel workload runs 288 CTAs on 152 SMs).  Each bulk copy costs
// the single issuing thread a fixed overhead (the mbarrier wait, the issue,
// the group bookkeeping), so fewer, larger entries move more per thread:
// measured on the 1 GiB workload, 16 KiB x 6 stages -> 32 KiB x 3 stages took
// one CTA pair per channel from 527 to 681 GB/s, 10 + 8 lanes from 2285 to
// 2347 GB/s and zero copy at 8 lanes from 2878 to 2984 GB/s.
constexpr int kTmaStages = 3;
constexpr uint32_t kTmaChunk = 32768;
// Loads issued ahead of the next store; the other stages hold stores that
// are still reading shared memory.
constexpr int kLookSend = 2;
constexpr int kLookZeroCopy = 2;
constexpr int kRecvStoresInFlight = 1;   // receiver: dst stores still reading their stage
// The sender's fifth warp (idle otherwise; the receiver's discards) keeps
// this many bulk entries of src beyond the mover's loads on their way into
// L2 with cp.async.bulk.prefetch (no shared memory, no completion), so more
// of the source is in flight than three stages hold.  The slot-filling
// modes take one entry (two cost 3% there: the prefetched lines crowd the
// L2-resident FIFO); zero copy and direct posts, which keep nothing in L2,
// take two.
constexpr int kPrefetchSlots = 1;
constexpr int kPrefetchToUser = 2;
// Receivers that read FIFO slots invalidate in L2, with discard.global.L2,
// the 128-byte lines of their stripe that they have read, before returning
// credit: the slot's dirty bytes are dead once read, and without this they are
// written back to DRAM whenever L2 evicts them before the slot is refilled.
// A fifth warp does it, so the copy pipeline never waits for it.  The
// operation's `discard` flag turns it off (the slots then keep the last bytes
// that passed through them).
constexpr bool kDiscard = true;
constexpr int kTmaThreads = kDiscard ? 160 : 128;
constexpr int kTmaSmem = kTmaStages * (int)kTmaChunk;
// The mover reports a step's stores complete once this many stores of the
// next step are in flight (1: the pipeline keeps one store going across the
// step boundary; 2 and 4 measured within 1%, slightly slower).
constexpr int kDefer = 1;
static_assert(kLookSend < kTmaStages && kLookZeroCopy < kTmaStages && kRecvStoresInFlight < kTmaStages,
              "a stage must be free for each look-ahead load");

// The stripe of one slot-step a lane moves: [b0, b0 + fb) in bulk entries of
// at most kTmaChunk bytes (at least one entry, possibly empty), then `rag`
// (< 16) bytes moved by the thread itself.
struct Stripe {
  u64 b0, fb, rag, nent;
};

__device__ __forceinline__ Stripe stripe_of(u64 sz, u64 lanes, u64 lane) {
  u64 b0, b1;
  piece(sz, lanes, lane, &b0, &b1);
  Stripe s;
  s.b0 = b0;
  const u64 n = b1 - b0;
  s.fb = n & ~15ull;
  s.rag = n - s.fb;
  s.nent = s.fb ? (s.fb + kTmaChunk - 1) / kTmaChunk : 1;
  return s;
}

__device__ __forceinline__ uint32_t entry_bytes(const Stripe& s, u64 e) {
  const u64 eo = e * kTmaChunk;
  if (eo >= s.fb) return 0;
  const u64 n = s.fb - eo;
  return (uint32_t)(n < kTmaChunk ? n : kTmaChunk);
}

__device__ __forceinline__ void copy_bytes(const char* src, char* dst, u64 n) {
  for (u64 i = 0; i < n; ++i) dst[i] = __ldcg(src + i);
}

// Entry numbering of one lane over all slot-steps of an operation: every
// step but the last has the stripe of a full slot, the last its own.
struct Entries {
  Stripe full, last;
  u64 nsteps, per_full, total;
  __device__ __forceinline__ void init(u64 len, u64 S, u64 G, u64 lane) {
    nsteps = (len + S - 1) / S;
    const u64 last_sz = len - (nsteps - 1) * S;
    full = stripe_of(nsteps > 1 ? S : last_sz, G, lane);
    last = stripe_of(last_sz, G, lane);
    per_full = nsteps > 1 ? full.nent : 0;
    total = per_full * (nsteps - 1) + last.nent;
  }
  // step and entry-within-step of global entry j
  __device__ __forceinline__ void locate(u64 j, u64* s, u64* e) const {
    const u64 nf = per_full * (nsteps - 1);
    if (j < nf) {
      *s = j / per_full;
      *e = j - *s * per_full;
    } else {
      *s = nsteps - 1;
      *e = j - nf;
    }
  }
  __device__ __forceinline__ const Stripe& stripe(u64 s) const { return s + 1 == nsteps ? last : full; }
};

// Modes of the kernel.  The posted modes replace head/tail by the
// receiver-driven credit FIFO ("RDMA and GPUDirect" §4.3; "NCCL transport data
// transfer (二)", netTransport): the receiver writes post entries {addr, size,
// idx} into the channel's post FIFO, the sender writes each chunk at the
// address of the post whose idx is step + 1 and answers with a completion
// {size, idx}.  Copy mode posts the receiver's staging slots (the receiver
// then copies them out, as in SIMPLE); direct mode posts dst itself.
//
// Proxy mode ("NCCL transport data transfer (二)", p2pTransport CE mode and
// shmTransport useMemcpy mode): the sender fills its own send ring and
// publishes tail[0]; a host thread copies each slot-step with the copy engines
// through `hops` rings and publishes tail[hops]; the receiver drains the last
// ring.  Counters, size words and the step base then live in mapped host
// memory and are accessed at .sys scope.
enum : int { kModeSimple = 0, kModeZeroCopy = 1, kModePostedCopy = 2, kModePostedDirect = 3, kModeProxy = 4 };

// control-word access at the scope the mode needs
template <bool kSys>
__device__ __forceinline__ u64 ctl_acquire(const u64* p) { return kSys ? ld_acquire_sys(p) : ld_acquire(p); }
template <bool kSys>
__device__ __forceinline__ u64 ctl_relaxed(const u64* p) { return kSys ? ld_relaxed_sys(p) : ld_relaxed(p); }
template <bool kSys>
__device__ __forceinline__ void ctl_release(u64* p, u64 v) {
  if (kSys) st_release_sys(p, v); else st_release(p, v);
}
template <bool kSys>
__device__ __forceinline__ void ctl_store(u64* p, u64 v) {
  if (kSys) st_relaxed_sys(p, v); else st_relaxed(p, v);
}

template <int kMode>
__global__ void __launch_bounds__(kTmaThreads, 1) p2p_tma_kernel(const P2pParams p) {
  constexpr bool kZeroCopy = kMode == kModeZeroCopy;
  constexpr bool kPosted = kMode == kModePostedCopy || kMode == kModePostedDirect;
  constexpr bool kDirect = kMode == kModePostedDirect;
  constexpr bool kToUser = kZeroCopy || kDirect;   // the sender writes dst itself
  constexpr bool kProxy = kMode == kModeProxy;
  extern __shared__ __align__(128) char stage_mem[];
  __shared__ __align__(8) u64 full[kTmaStages];
  __shared__ __align__(8) u64 empty[kTmaStages];   // receiver: stage free again
  __shared__ u64 s_base;
  __shared__ u64 s_mirror;   // latest head / post (sender) or tail / completion (receiver) seen by the watcher
  __shared__ u64 s_done;     // sender: steps [0, s_done) have their bulk stores complete
  __shared__ u64 s_read;     // receiver: steps [0, s_read) have their slot stripe in shared memory
  __shared__ u64 s_freed;    // receiver of one lane: steps [0, s_freed) may be refilled
  __shared__ u64 s_loaded;   // sender: bulk loads the mover has issued (~0: the mover is done)
  __shared__ u64 s_addr[kPosted ? kMaxSlots : 1];   // posted sender: address and size of each slot's post
  __shared__ u64 s_cap[kPosted ? kMaxSlots : 1];
  __shared__ int s_stop;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const unsigned crank = blockIdx.x % p.csize;   // CTA within its channel
  const int ch = blockIdx.x / p.csize;
  const int G = p.lanes;                        // sender lanes
  const int GR = kToUser ? 1 : p.rlanes;        // receiver lanes
  const bool sender = crank < (unsigned)G;
  const int lane_id = sender ? (int)crank : (int)crank - G;
  const int GS = sender ? G : GR;               // lanes of this CTA's side
  const unsigned leader = sender ? 0u : (unsigned)G;
  const bool leader_cta = crank == leader;
  const u64 N = (u64)p.nslots;
  const u64 S = p.slot_bytes;
  const u64 K = kTmaStages;

  char* ctl = p.ctl + (u64)ch * kCtlBytes;
  u64* tail = reinterpret_cast<u64*>(ctl + kTailOff);
  u64* head = reinterpret_cast<u64*>(ctl + kHeadOff);
  u64* ptrx = reinterpret_cast<u64*>(ctl + kPtrxOff);
  u64* basew = reinterpret_cast<u64*>(ctl + kBaseOff);
  long long* sizew = reinterpret_cast<long long*>(ctl + kSizeOff);
  char* slots = p.slots + (u64)ch * p.ch_stride;
  char* pctl = kPosted ? p.pctl + (u64)ch * kPostCtlBytes : nullptr;
  u64* posts = reinterpret_cast<u64*>(pctl + kPostOff);   // entry k: words 8k (addr), 8k+1 (size), 8k+2 (idx)
  u64* cq = reinterpret_cast<u64*>(pctl + kComplOff);     // entry k: words 2k (size), 2k+1 (idx)
  if (kPosted) basew = reinterpret_cast<u64*>(pctl + kPostBaseOff);
  u64* tail_pub = tail;         // the tail this kernel's sender publishes
  char* slots_send = slots;     // where the sender writes, and where the receiver reads
  char* slots_recv = slots;
  if (kProxy) {
    char* ce = p.ce + (u64)ch * kCeCtlBytes;
    tail_pub = reinterpret_cast<u64*>(ce + kCeTailOff);
    tail = reinterpret_cast<u64*>(ce + kCeTailOff + 128 * p.hops);
    head = reinterpret_cast<u64*>(ce + kCeHeadOff);
    basew = reinterpret_cast<u64*>(ce + kCeBaseOff);
    sizew = reinterpret_cast<long long*>(ce + kCeSizeOff);
    slots_send = p.send_ring + (u64)ch * p.ch_stride;
    slots_recv = p.recv_ring + (u64)ch * p.ch_stride;
  }

  u64 lo, hi;
  channel_range(p.nbytes, p.nchannels, ch, &lo, &hi);
  const u64 len = hi - lo;
  const u64 nsteps = (len + S - 1) / S;
  const WaitCtx w{p.status, p.abort_word, p.timeout_ns, ch, p.op};
  auto step_size = [&](u64 s) -> u64 { return (len - s * S) < S ? (len - s * S) : S; };

  if (threadIdx.x == 0) {
    const u64 b0 = ctl_relaxed<kProxy>(basew);   // in flight while op_begin reads the sticky word
    s_stop = op_begin(w) ? 1 : 0;
    s_base = b0;
    s_mirror = 0;
    s_done = 0;
    s_read = 0;
    s_freed = 0;
    s_loaded = 0;
    for (int k = 0; k < kTmaStages; ++k) {
      mbar_init(smem_addr(&full[k]), 1);
      mbar_init(smem_addr(&empty[k]), 1);
    }
    mbar_init_fence();
  }
  __syncthreads();
  const u64 base = s_base;
  const bool run = nsteps > 0 && s_stop == 0;
  const bool discard = kDiscard && !kToUser && p.discard != 0;
  ChanStats* cs = p.stats ? p.stats + ch : nullptr;
  if (cs && sender && leader_cta && threadIdx.x == 0) {
    const u64 t = globaltimer();
    cs->steps = run ? nsteps : 0;
    cs->t_start = t;
    cs->send_polls = 0;
    cs->recv_polls = 0;
    if (!run) cs->t_end = t;
  }
  const uint32_t sm0 = smem_addr(stage_mem);
  // Per-slot arrival counters of this side: each lane adds 1 when it is done
  // with its stripe of a slot-step, the side's publisher waits for all GS
  // lanes and takes them back off (so the counters are zero between
  // operations).
  u64* arrivals = p.arr + (u64)ch * (kArrBytes / 8) + (sender ? 0 : kMaxSlots);
  // FIFO slots: reused every N steps; normal priority (evict_last measured
  // 1.7-3.7% slower on the 16-channel workload, evict_first 11% slower)
  const u64 pol_slot = policy_evict_normal();
  // src / dst are read or written once: evict first where FIFO slots share the
  // L2 with them, normal priority where nothing else is kept (zero copy and
  // direct posts; measured 1-2% faster there, 9% slower for SIMPLE)
  const u64 pol_user = kToUser ? policy_evict_normal() : policy_evict_first();

  // receiver side of the posted modes: post chunk s (copy: staging slot
  // (base + s) % N, whole; direct: its place in dst, its exact size)
  auto post = [&](u64 s) {
    const u64 k = (base + s) % N;
    const u64 addr = kDirect ? reinterpret_cast<u64>(p.dst + lo + s * S) : reinterpret_cast<u64>(slots + k * S);
    st_relaxed(posts + 8 * k, addr);
    st_relaxed(posts + 8 * k + 1, kDirect ? step_size(s) : S);
    st_release(posts + 8 * k + 2, base + s + 1);
  };

  if (run && lane == 0) {
    if (kToUser && !sender) {
      if (warp == 1 && kZeroCopy) {
        // zero-copy receiver: post the destination, echo tail into head
        u64 v = 0, tcache = 0;
        if (wait_word(ptrx, 0, v, w, XP_WAIT_PTR_EXCHANGE)) {
          st_release(ptrx, reinterpret_cast<u64>(p.dst + lo));
          u64 j = 0;
          for (; j < nsteps; ++j) {
            if (!wait_geq(tail, base + j + 1, tcache, w, XP_WAIT_TAIL)) break;
            st_release(head, base + j + 1);
          }
          if (j == nsteps) st_relaxed(basew, base + nsteps);
          if (cs) cs->t_end = globaltimer();
        }
      } else if (warp == 1 && kDirect) {
        // direct-posted receiver: keep up to N posts of dst outstanding,
        // take the completions in order and check the size each reports
        const u64 first = nsteps < N ? nsteps : N;
        for (u64 s = 0; s < first; ++s) post(s);
        note_occupancy(p.status, p.op, (unsigned)first);
        u64 j = 0;
        for (; j < nsteps; ++j) {
          const u64 k = (base + j) % N;
          u64 c = 0;
          if (!wait_geq(cq + 2 * k + 1, base + j + 1, c, w, XP_WAIT_COMPLETION)) break;
          const u64 got = ld_relaxed(cq + 2 * k);
          if (c != base + j + 1 || got != step_size(j)) {
            report(w, XP_ERR_BOUNDS, XP_WAIT_COMPLETION, c != base + j + 1 ? c : got,
                   c != base + j + 1 ? base + j + 1 : step_size(j));
            break;
          }
          if (j + N < nsteps) post(j + N);
        }
        if (j == nsteps) st_relaxed(basew, base + nsteps);
        if (cs) cs->t_end = globaltimer();
      }
    } else if (warp == 0) {
      Entries en;
      en.init(len, S, (u64)GS, (u64)lane_id);
      const u64 total = en.total;
      u64 jl = 0;   // next entry to load
      u64 j = 0;    // next entry to store
      bool ok = true;
      if (sender) {
        // ---------------- sender mover ----------------
        constexpr int kLook = kToUser ? kLookZeroCopy : kLookSend;
        auto issue_load = [&](u64 q) {
          u64 s, e;
          en.locate(q, &s, &e);
          const Stripe& st = en.stripe(s);
          const uint32_t k = (uint32_t)(q % K);
          const uint32_t nb = entry_bytes(st, e);
          mbar_arrive_expect_tx(smem_addr(&full[k]), nb);
          if (nb)
            bulk_load(sm0 + k * kTmaChunk, p.src + lo + s * S + st.b0 + e * kTmaChunk, nb, smem_addr(&full[k]), pol_user);
        };
        volatile u64* loaded = &s_loaded;   // pacing for the prefetcher only
        for (; jl < total && jl < (u64)kLook; ++jl) issue_load(jl);
        *loaded = jl;
        char* dstp = nullptr;
        if (kZeroCopy) {
          u64 v = 0;
          ok = wait_word(ptrx, 1, v, w, XP_WAIT_PTR_EXCHANGE);
          dstp = reinterpret_cast<char*>(v);
        }
        u64 hcache = 0;
        long long pending = -1;   // step whose completion signal is deferred
        int since = 0;
        for (u64 s = 0; s < nsteps && ok; ++s) {
          const u64 step = base + s;
          // credit: head (SIMPLE, zero copy) or this step's post (posted modes)
          const u64 need = kPosted ? step + 1 : (step + 1 > N ? step + 1 - N : 0);
          if (need && hcache < need) {
            const u64 h = ld_acquire_cta_shared(&s_mirror);
            if (h >= need) {
              hcache = h;
            } else {
              if (pending >= 0) {
                bulk_wait<0>();
                fence_proxy_async_global();
                st_release_cta_shared(&s_done, (u64)pending + 1);
                pending = -1;
              }
              if (!wait_mirror(&s_mirror, need, hcache, w, kPosted ? XP_WAIT_POST : XP_WAIT_HEAD)) { ok = false; break; }
            }
          }
          fence_proxy_async_global();
          const u64 off = s * S;
          const Stripe& st = en.stripe(s);
          char* to;
          if (kPosted) {
            const u64 a = s_addr[step % N];
            if (a % 16 || step_size(s) > s_cap[step % N]) {
              report(w, XP_ERR_BOUNDS, XP_WAIT_POST, a % 16 ? a : step_size(s), a % 16 ? 16 : s_cap[step % N]);
              ok = false;
              break;
            }
            to = reinterpret_cast<char*>(a);
          } else {
            to = kZeroCopy ? dstp + off : slots_send + (step % N) * S;
          }
          for (u64 e = 0; e < st.nent; ++e, ++j) {
            const uint32_t k = (uint32_t)(j % K);
            if (!mbar_wait_cta(smem_addr(&full[k]), (uint32_t)((j / K) & 1), w)) { ok = false; break; }
            const uint32_t nb = entry_bytes(st, e);
            if (nb) bulk_store(to + st.b0 + e * kTmaChunk, sm0 + k * kTmaChunk, nb, kToUser ? pol_user : pol_slot);
            bulk_commit();
            if (jl < total) {
              // the stage of entry jl = j + kLook last held entry jl - K,
              // whose store group has K - kLook newer ones (j - K + kLook + 1
              // .. j): once at most that many are still reading shared
              // memory, it has finished
              bulk_wait_read<kTmaStages - kLook>();
              issue_load(jl++);
              *loaded = jl;
            }
            if (pending >= 0 && ++since == kDefer) {
              bulk_wait<kDefer>();
              fence_proxy_async_global();
              st_release_cta_shared(&s_done, (u64)pending + 1);
              pending = -1;
            }
          }
          if (!ok) break;
          if (st.rag) copy_bytes(p.src + lo + off + st.b0 + st.fb, to + st.b0 + st.fb, st.rag);
          if ((kMode == kModeSimple || kProxy) && lane_id == 0)
            ctl_store<kProxy>(reinterpret_cast<u64*>(sizew + step % N), step_size(s));
          if (pending >= 0) {
            bulk_wait<0>();
            fence_proxy_async_global();
            st_release_cta_shared(&s_done, (u64)pending + 1);
          }
          pending = (long long)s;
          since = 0;
        }
        *loaded = ~0ull;
        bulk_wait<0>();
        if (ok && pending >= 0) {
          fence_proxy_async_global();
          st_release_cta_shared(&s_done, (u64)pending + 1);
        }
      } else {
        // ---------------- receiver loader ----------------
        // waits for tail or the completion (mirrored), copies the step's
        // ragged bytes, and loads the stripe's entries from the slot as
        // stages become free
        u64 tcache = 0;
        for (u64 s = 0; s < nsteps && ok; ++s) {
          const u64 step = base + s;
          if (!wait_mirror(&s_mirror, step + 1, tcache, w, kPosted ? XP_WAIT_COMPLETION : XP_WAIT_TAIL)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
          const u64 off = s * S;
          const char* from = slots_recv + (step % N) * S;
          if (!kPosted && lane_id == 0) {
            const long long got = (long long)ctl_relaxed<kProxy>(reinterpret_cast<const u64*>(sizew + step % N));
            if (got != (long long)step_size(s)) report(w, XP_ERR_BOUNDS, XP_WAIT_SIZE_WORD, (u64)got, step_size(s));
          }
          const Stripe& st = en.stripe(s);
          if (st.rag) copy_bytes(from + st.b0 + st.fb, p.dst + lo + off + st.b0 + st.fb, st.rag);
          for (u64 e = 0; e < st.nent; ++e, ++jl) {
            const uint32_t k = (uint32_t)(jl % K);
            if (jl >= K && !mbar_wait_cta(smem_addr(&empty[k]), (uint32_t)(((jl / K) - 1) & 1), w)) {
              ok = false;
              break;
            }
            const uint32_t nb = entry_bytes(st, e);
            mbar_arrive_expect_tx(smem_addr(&full[k]), nb);
            if (nb) bulk_load(sm0 + k * kTmaChunk, from + st.b0 + e * kTmaChunk, nb, smem_addr(&full[k]), pol_slot);
          }
        }
      }
      // every issued load must land before the CTA may exit
      for (u64 i = (jl > K ? jl - K : 0); i < jl; ++i)
        mbar_wait_cta(smem_addr(&full[i % K]), (uint32_t)((i / K) & 1), w);
    } else if (warp == 1 && sender) {
      // ---------------- sender signaler ----------------
      // Turns each "stores of step s complete" from the mover into a release
      // add on the slot's arrival counter.  A release waits for the issuing
      // thread's own memory traffic; this thread has none in flight, the
      // mover always has.
      u64 done = 0;
      for (u64 s = 0; s < nsteps && GS > 1; ++s) {   // one lane: the publisher reads s_done itself
        if (!wait_mirror(&s_done, s + 1, done, w, XP_WAIT_SLOT_BARRIER)) break;
        red_add_release(arrivals + (base + s) % N, 1);
      }
    } else if (warp == 1 && !sender) {
      // ---------------- receiver storer ----------------
      // stores each loaded entry into dst; once the last entry of a step is
      // in shared memory the stripe of the slot has been read: signal it
      Entries en;
      en.init(len, S, (u64)GS, (u64)lane_id);
      u64 j = 0;
      bool ok = true;
      for (u64 s = 0; s < nsteps && ok; ++s) {
        const Stripe& st = en.stripe(s);
        for (u64 e = 0; e < st.nent; ++e, ++j) {
          const uint32_t k = (uint32_t)(j % K);
          if (!mbar_wait_cta(smem_addr(&full[k]), (uint32_t)((j / K) & 1), w)) { ok = false; break; }
          // The slot's bytes for this stripe are in shared memory (its ragged
          // bytes were copied before the first load of the step): the reads
          // are complete, so the signal carries no ordering.
          if (e + 1 == st.nent) {
            if (discard)
              st_release_cta_shared(&s_read, s + 1);   // the discarder returns the credit
            else if (GS > 1)
              red_add_relaxed(arrivals + (base + s) % N, 1);
            else
              st_release_cta_shared(&s_freed, s + 1);
          }
          const uint32_t nb = entry_bytes(st, e);
          if (nb) bulk_store(p.dst + lo + s * S + st.b0 + e * kTmaChunk, sm0 + k * kTmaChunk, nb, pol_user);
          bulk_commit();
          bulk_wait_read<kRecvStoresInFlight>();
          if (j >= (u64)kRecvStoresInFlight) mbar_arrive_local_relaxed(smem_addr(&empty[(j - kRecvStoresInFlight) % K]));
        }
      }
      bulk_wait<0>();
    } else if (warp == 2 && kPosted) {
      // ---------------- watcher (posted modes) ----------------
      // sender: takes the posts in order, keeps each one's address and size
      // in shared memory and mirrors the count; receiver (copy mode): takes
      // the completions in order, checks their sizes and mirrors the count
      WaitClock clk;
      u64 polls = 0;
      for (u64 m = 0; m < nsteps; ++m) {
        const u64 k = (base + m) % N;
        const u64* idx = sender ? posts + 8 * k + 2 : cq + 2 * k + 1;
        const u64 want = base + m + 1;
        u64 v;
        bool ok = true;
        while (++polls, (v = ld_acquire(idx)) < want) {
          if (!clk.tick(w, sender ? XP_WAIT_POST : XP_WAIT_COMPLETION, v, want)) { ok = false; break; }
        }
        if (!ok) break;
        if (v != want) {   // an entry from the future: the FIFO is corrupt
          report(w, XP_ERR_BOUNDS, sender ? XP_WAIT_POST : XP_WAIT_COMPLETION, v, want);
          break;
        }
        if (sender) {
          s_addr[k] = ld_relaxed(posts + 8 * k);
          s_cap[k] = ld_relaxed(posts + 8 * k + 1);
        } else {
          const u64 got = ld_relaxed(cq + 2 * k);
          if (got != step_size(m)) {
            report(w, XP_ERR_BOUNDS, XP_WAIT_COMPLETION, got, step_size(m));
            break;
          }
        }
        st_release_cta_shared(&s_mirror, want);
        clk = WaitClock();   // the timeout counts time without progress
      }
      if (cs && leader_cta) (sender ? cs->send_polls : cs->recv_polls) = polls;
    } else if (warp == 2) {
      // ---------------- watcher ----------------
      // sender: head, as far as the last step's credit needs it;
      // receiver: tail, up to the last step
      const u64* word = sender ? head : tail;
      const u64 target = sender ? (base + nsteps > N ? base + nsteps - N : 0) : base + nsteps;
      u64 seen = 0, polls = 0;
      WaitClock clk;
      while (seen < target) {
        ++polls;
        const u64 v = ctl_acquire<kProxy>(word);
        if (v > seen) {
          seen = v;
          st_release_cta_shared(&s_mirror, v);
          clk = WaitClock();   // the timeout counts time without progress
        } else if (!clk.tick(w, sender ? XP_WAIT_HEAD : XP_WAIT_TAIL, v, target)) {
          break;
        }
      }
      if (cs && leader_cta) (sender ? cs->send_polls : cs->recv_polls) = polls;
    } else if (warp == 3 && leader_cta) {
      // ---------------- publisher ----------------
      // SIMPLE / zero copy: tail (sender) or head (receiver) = step + 1;
      // posted: the completion of the step (sender) or the post N steps on
      // (receiver, copy mode)
      u64 s = 0;
      unsigned max_occ = 0;
      if (kPosted && !sender) {
        const u64 first = nsteps < N ? nsteps : N;
        for (u64 q = 0; q < first; ++q) post(q);
        max_occ = (unsigned)first;
      }
      u64 mine = 0;
      for (; s < nsteps; ++s) {
        const u64 step = base + s;
        if (GS == 1) {
          if (!wait_mirror(sender ? &s_done : &s_freed, s + 1, mine, w, XP_WAIT_SLOT_BARRIER)) break;
        } else {
          u64 c = 0;
          if (!wait_geq(arrivals + step % N, (u64)GS, c, w, XP_WAIT_SLOT_BARRIER)) break;
          red_add_relaxed(arrivals + step % N, 0ull - (u64)GS);
        }
        if (kPosted) {
          if (sender) {
            st_relaxed(cq + 2 * (step % N), step_size(s));
            st_release(cq + 2 * (step % N) + 1, step + 1);
          } else if (s + N < nsteps) {
            post(s + N);
          }
        } else if (sender) {
          ctl_release<kProxy>(tail_pub, step + 1);
          const u64 h = ctl_relaxed<kProxy>(head);
          const u64 occ = step + 1 - h;
          if (h > step + 1 || occ > N) {
            report(w, XP_ERR_BOUNDS, XP_WAIT_OCCUPANCY, occ, N);
            break;
          }
          if (occ > max_occ) max_occ = (unsigned)occ;
        } else {
          ctl_release<kProxy>(head, step + 1);
        }
      }
      if (sender != kPosted) note_occupancy(p.status, p.op, max_occ);
      if (sender) {
        if (kZeroCopy && s == nsteps) {
          u64 hc = 0;
          if (wait_geq(head, base + nsteps, hc, w, XP_WAIT_HEAD)) st_release(ptrx, 0);
        }
      } else if (s == nsteps) {
        ctl_store<kProxy>(basew, base + nsteps);
      }
      if (cs && !sender) cs->t_end = globaltimer();
    }
  }
  if (run && sender && warp == 4 && lane == 0) {
    // ---------------- prefetcher ----------------
    // walks the mover's entries kPrefetch ahead of its bulk loads and asks
    // L2 to fetch each from src; it only paces itself on the mover's count,
    // so it needs no ordering, and it stops when the mover is done, on the
    // operation's abort flag, or after timeout_ns without progress
    constexpr u64 kPrefetch = kToUser ? kPrefetchToUser : kPrefetchSlots;
    constexpr u64 kFirst = kToUser ? kLookZeroCopy : kLookSend;   // loads the mover issues up front
    Entries en;
    en.init(len, S, (u64)GS, (u64)lane_id);
    const volatile u64* loaded = &s_loaded;
    u64 t0 = globaltimer();
    unsigned it = 0;
    for (u64 q = kFirst; q < en.total;) {
      const u64 l = *loaded;
      if (l == ~0ull) break;
      if (q < l + kPrefetch) {
        u64 ps, pe;
        en.locate(q, &ps, &pe);
        const Stripe& pst = en.stripe(ps);
        const uint32_t nb = entry_bytes(pst, pe);
        if (nb) bulk_prefetch_l2(p.src + lo + ps * S + pst.b0 + pe * kTmaChunk, nb);
        ++q;
        t0 = globaltimer();
        continue;
      }
      if ((++it & 63u) == 0 && (op_aborted_device(w) || globaltimer() - t0 > w.timeout_ns)) break;
    }
  }
  if (discard && run && !sender && warp == 4) {
    // ---------------- discarder ----------------
    // once the storer has seen a step's stripe land in shared memory, drop
    // the 128-byte lines lying wholly inside the stripe from L2 (lines shared
    // with a neighbouring lane's stripe stay), then signal the slot consumed:
    // with a release, so the drops are performed before the sender may
    // refill the slot.  The operation's last step is signalled first and its
    // lines dropped after: nothing refills that slot before the kernel has
    // ended, so its credit need not wait for the drops.
    Entries en;
    en.init(len, S, (u64)GS, (u64)lane_id);
    u64 seen = 0;
    for (u64 s = 0; s < nsteps; ++s) {
      int ok = 1;
      if (lane == 0) ok = wait_mirror(&s_read, s + 1, seen, w, XP_WAIT_SLOT_BARRIER) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      const bool last = s + 1 == nsteps;
      if (last && lane == 0) {
        // the stripe's reads are complete: the signal carries no ordering
        if (GS > 1) red_add_relaxed(arrivals + (base + s) % N, 1);
        else st_release_cta_shared(&s_freed, s + 1);
      }
      const Stripe& st = en.stripe(s);
      const u64 from = reinterpret_cast<u64>(slots_recv + ((base + s) % N) * S);
      const u64 l0 = (from + st.b0 + 127) & ~127ull;
      const u64 l1 = (from + st.b0 + st.fb + st.rag) & ~127ull;
      for (u64 x = l0 + 128ull * lane; x < l1; x += 128ull * 32) discard_l2(reinterpret_cast<void*>(x));
      __syncwarp();
      if (!last && lane == 0) {
        if (GS > 1) {
          red_add_release(arrivals + (base + s) % N, 1);
        } else {
          fence_acq_rel_gpu();   // the warp's drops performed, then the publisher may return the credit
          st_release_cta_shared(&s_freed, s + 1);
        }
      }
    }
  }
  __syncwarp();
}

template __global__ void p2p_tma_kernel<kModeSimple>(const P2pParams);
template __global__ void p2p_tma_kernel<kModeZeroCopy>(const P2pParams);
template __global__ void p2p_tma_kernel<kModePostedCopy>(const P2pParams);
template __global__ void p2p_tma_kernel<kModePostedDirect>(const P2pParams);
template __global__ void p2p_tma_kernel<kModeProxy>(const P2pParams);

void* p2p_tma_kernel_ptr(int mode) {
  switch (mode) {
    case kModeZeroCopy: return reinterpret_cast<void*>(&p2p_tma_kernel<kModeZeroCopy>);
    case kModePostedCopy: return reinterpret_cast<void*>(&p2p_tma_kernel<kModePostedCopy>);
    case kModePostedDirect: return reinterpret_cast<void*>(&p2p_tma_kernel<kModePostedDirect>);
    case kModeProxy: return reinterpret_cast<void*>(&p2p_tma_kernel<kModeProxy>);
    default: return reinterpret_cast<void*>(&p2p_tma_kernel<kModeSimple>);
  }
}
int p2p_tma_threads() { return kTmaThreads; }
int p2p_tma_smem() { return kTmaSmem; }

}  // namespace xp
