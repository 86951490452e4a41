// Virtual ring allreduce for FIFOs in HBM, data moved with bulk (TMA) copies.
//
// Same schedule and FIFO protocol as the vector kernel in xp_ring.cu (ring
// neighbours from "NCCL transport setup", 具体说明; per round send(r-1),
// recvReduceSend(r-1-j), recvReduceCopySend(r), recvCopySend(r-1-j),
// recv(r+1); chunks of at most N/2 slots).  A channel may be spread over G
// lanes: lane g moves the g-th 16-byte aligned stripe of every slot-step of
// every FIFO, with a control block (tail, head, step base) of its own per
// FIFO, so the lanes of a channel never wait for one another and the element
// chunking (and with it the order of every sum) does not depend on G.  The
// ranks a lane's ring waits on must run at once: the grid is launched
// cooperatively when all of it fits on the GPU, else as one cluster of P CTAs
// per (channel, lane), co-resident by construction.  A launch may cover a
// group of channels starting at c_first (channels never wait on one
// another), so the host can run the channels in groups whose live FIFO data
// stays in L2.  Each CTA moves its
// stripe through a ring of kRStages stages of two buffers each (A: received
// slot, or own input for `send`; B: own input for the reducing steps).
// Threads:
//   loader     - waits for the predecessor's tail (mirrored), bulk-loads the
//                received slot and/or the own input into a free stage;
//   compute    - four warps: A += B for recvReduceSend / recvReduceCopySend
//                (fp32 __fadd_rn or wrapping int32), the ragged tail of the
//                buffer with plain loads and stores, and the "slot consumed"
//                signal once a received slot-step is in shared memory;
//   storer     - waits for credit (the successor's head, mirrored), bulk-stores
//                A into the successor's slot and/or the own output, frees the
//                stage; reports completed send slot-steps through shared
//                memory (after kDefer more store groups, so the store
//                pipeline never drains at a step boundary, and always before
//                it blocks: what it waits for may depend, around the ring,
//                on the step it has not reported yet);
//   signaler   - turns those reports into the release arrive on the send
//                slot's barrier (a release waits for the issuing thread's
//                in-flight traffic: the storer always has some, the signaler
//                none);
//   watcher    - mirrors the predecessor's tail and the successor's head into
//                shared memory;
//   publishers - store the successor FIFO's tail and the own FIFO's head (this
//                lane's control blocks) once the step is signalled.
#include <cuda_runtime.h>

#include "xp_device.cuh"

namespace xp {

namespace {

constexpr int kRStages = 6;
constexpr uint32_t kRChunk = 16384;          // bytes per buffer; a stage is A + B
constexpr int kRStoresInFlight = 2;          // store groups still reading their stage
constexpr int kRDefer = 4;
constexpr int kRComputeWarps = 4;
constexpr int kRThreads = 32 * 10;           // loader, 4 compute, storer, watcher, signaler, 2 publishers
constexpr int kRSmem = kRStages * 2 * (int)kRChunk;
static_assert(kRStoresInFlight < kRStages, "the loader needs a free stage");

enum RingKind { K_SEND = 0, K_RRS = 1, K_RRCS = 2, K_RCS = 3, K_RECV = 4 };

__device__ __forceinline__ bool kind_recv(int k) { return k != K_SEND; }
__device__ __forceinline__ bool kind_send(int k) { return k != K_RECV; }
__device__ __forceinline__ bool kind_reduce(int k) { return k == K_RRS || k == K_RRCS; }
__device__ __forceinline__ bool kind_out(int k) { return k == K_RRCS || k == K_RCS || k == K_RECV; }

// Step kind and chunk of schedule position `pos` (0 .. 2P-2) at rank r.
__device__ __forceinline__ void ring_op(int pos, int r, int P, int* kind, int* chunk) {
  int k;
  if (pos == 0) {
    *kind = K_SEND;
    k = r - 1;
  } else if (pos <= P - 2) {
    *kind = K_RRS;
    k = r - 1 - pos;
  } else if (pos == P - 1) {
    *kind = K_RRCS;
    k = r;
  } else if (pos <= 2 * P - 3) {
    *kind = K_RCS;
    k = r - 1 - (pos - P);
  } else {
    *kind = K_RECV;
    k = r + 1;
  }
  *chunk = ((k % P) + P) % P;
}

struct Stripe {
  u64 b0, fb, rag, nent;
};

// Lane `lane` of `lanes` owns bytes [lane W, (lane + 1) W) of every slot,
// W = round_up(ceil(S / lanes), 16), whatever the size sz of the slot-step:
// lanes publish their own counters, so a lane may refill its part of a slot
// while another lane still reads its own part of the previous step there,
// and the parts must not depend on the step size.
__device__ __forceinline__ Stripe stripe_of(u64 sz, u64 slot_bytes, u64 lanes, u64 lane) {
  const u64 W = ((slot_bytes + lanes - 1) / lanes + 15) & ~15ull;
  u64 b0 = lane * W, b1 = (lane + 1) * W;
  if (b0 > sz) b0 = sz;
  if (b1 > sz) b1 = sz;
  Stripe s;
  s.b0 = b0;
  const u64 n = b1 - b0;
  s.fb = n & ~15ull;
  s.rag = n - s.fb;
  s.nent = s.fb ? (s.fb + kRChunk - 1) / kRChunk : 1;
  return s;
}

__device__ __forceinline__ uint32_t entry_bytes(const Stripe& s, u64 e) {
  const u64 eo = e * kRChunk;
  if (eo >= s.fb) return 0;
  const u64 n = s.fb - eo;
  return (uint32_t)(n < kRChunk ? n : kRChunk);
}

// Walk of one lane over every entry of a rank's schedule on one channel.
struct RingWalk {
  u64 clen, P, ce, align, epl, es, G, lane;
  int r;
  u64 off, m, cs;       // current round
  int pos;
  int kind;
  u64 kstart, klen;     // current chunk, elements relative to the channel start
  u64 o, n;             // current slot-step within the chunk
  Stripe st;
  u64 e;                // entry within the stripe
  u64 rs, ss;           // receive / send slot-steps before the current one
  bool done;

  __device__ void round_setup() {
    m = clen - off;
    if (m > P * ce) m = P * ce;
    u64 c = (m + P - 1) / P;
    c = (c + align - 1) / align * align;
    cs = c < ce ? c : ce;
  }
  __device__ void step_setup() {
    n = (klen - o) < epl ? (klen - o) : epl;
    st = stripe_of(n * es, epl * es, G, lane);
    e = 0;
  }
  __device__ void next_chunk() {
    for (;;) {
      ++pos;
      if (pos > 2 * (int)P - 2) {
        off += m;
        if (off >= clen) {
          done = true;
          return;
        }
        round_setup();
        pos = 0;
      }
      int k;
      ring_op(pos, r, (int)P, &kind, &k);
      u64 lo = (u64)k * cs, hi = (u64)(k + 1) * cs;
      if (lo > m) lo = m;
      if (hi > m) hi = m;
      if (hi > lo) {
        kstart = off + lo;
        klen = hi - lo;
        o = 0;
        step_setup();
        return;
      }
    }
  }
  __device__ void init(u64 clen_, u64 P_, u64 ce_, u64 align_, u64 epl_, u64 es_, u64 G_, u64 lane_, int r_) {
    clen = clen_;
    P = P_;
    ce = ce_;
    align = align_;
    epl = epl_;
    es = es_;
    G = G_;
    lane = lane_;
    r = r_;
    off = 0;
    rs = ss = 0;
    done = clen == 0;
    if (!done) {
      round_setup();
      pos = -1;
      next_chunk();
    }
  }
  __device__ bool first() const { return e == 0; }
  __device__ bool last() const { return e + 1 == st.nent; }
  // advance to the next entry
  __device__ void next() {
    if (++e < st.nent) return;
    if (kind_recv(kind)) ++rs;
    if (kind_send(kind)) ++ss;
    o += epl;
    if (o < klen) {
      step_setup();
      return;
    }
    next_chunk();
  }
};

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
}
__device__ __forceinline__ int4 add4(int4 a, int4 b) {
  return make_int4((int)((unsigned)a.x + (unsigned)b.x), (int)((unsigned)a.y + (unsigned)b.y),
                   (int)((unsigned)a.z + (unsigned)b.z), (int)((unsigned)a.w + (unsigned)b.w));
}
__device__ __forceinline__ float add1(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ int add1(int a, int b) { return (int)((unsigned)a + (unsigned)b); }

// Slot-steps this rank receives and sends on one channel.
__device__ void count_steps(u64 clen, u64 P, u64 ce, u64 align, u64 epl, int r, u64* nrecv, u64* nsend) {
  u64 off = 0, nr = 0, ns = 0;
  while (off < clen) {
    u64 m = clen - off;
    if (m > P * ce) m = P * ce;
    u64 cs = (m + P - 1) / P;
    cs = (cs + align - 1) / align * align;
    if (cs > ce) cs = ce;
    for (int pos = 0; pos <= 2 * (int)P - 2; ++pos) {
      int kind, k;
      ring_op(pos, r, (int)P, &kind, &k);
      u64 lo = (u64)k * cs, hi = (u64)(k + 1) * cs;
      if (lo > m) lo = m;
      if (hi > m) hi = m;
      const u64 steps = (hi - lo + epl - 1) / epl;
      if (kind_recv(kind)) nr += steps;
      if (kind_send(kind)) ns += steps;
    }
    off += m;
  }
  *nrecv = nr;
  *nsend = ns;
}

// AND of `ok` over the compute warps (named barrier 1).
__device__ __forceinline__ int compute_vote(int ok) {
  uint32_t res;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(res)
      : "r"(ok), "n"(32 * kRComputeWarps)
      : "memory");
  return (int)res;
}

__device__ __forceinline__ void compute_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kRComputeWarps) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace

template <typename T, typename V>
__global__ void __launch_bounds__(kRThreads, 1) ring_tma_kernel(const RingParams p) {
  extern __shared__ __align__(128) char stage_mem[];
  __shared__ __align__(8) u64 bars_send[kMaxSlots];
  __shared__ __align__(8) u64 bars_recv[kMaxSlots];
  __shared__ __align__(8) u64 full[kRStages];
  __shared__ __align__(8) u64 computed[kRStages];
  __shared__ __align__(8) u64 empty[kRStages];
  __shared__ u64 s_rbase, s_sbase;
  __shared__ u64 m_tail, m_head;   // mirrored predecessor tail / successor head
  __shared__ u64 s_done;           // send slot-steps whose stores completed
  __shared__ int s_stop;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int P = p.nranks;
  const int G = p.lanes;
  // CTA (c, g, r) = block (c * G + g) * P + r: a cooperative grid, or one
  // cluster of P CTAs per (channel, lane) whose cluster rank is r
  const int c = p.c_first + (int)(blockIdx.x / P) / G;
  const int g = (int)(blockIdx.x / P) % G;
  const int r = (int)(blockIdx.x % P);
  const unsigned leader = cluster_ctarank();         // every CTA publishes its own lane's counters
  const bool leader_cta = true;
  const u64 N = (u64)p.nslots;
  const u64 S = p.slot_bytes;
  const u64 es = sizeof(T);
  const u64 align = 16 / es;
  const u64 epl = S / es;
  const u64 ce = (N / 2) * S / es;
  const u64 K = kRStages;

  const int f_recv = c * P + r;
  const int f_send = c * P + (r + 1) % P;
  char* ctl_r = p.ctl + ((u64)f_recv * kRingMaxLanes + g) * kCtlBytes;
  char* ctl_s = p.ctl + ((u64)f_send * kRingMaxLanes + g) * kCtlBytes;
  u64* tail_recv = reinterpret_cast<u64*>(ctl_r + kTailOff);
  u64* head_recv = reinterpret_cast<u64*>(ctl_r + kHeadOff);
  u64* base_recv = reinterpret_cast<u64*>(ctl_r + kBaseOff);
  u64* tail_send = reinterpret_cast<u64*>(ctl_s + kTailOff);
  u64* head_send = reinterpret_cast<u64*>(ctl_s + kHeadOff);
  u64* base_send = reinterpret_cast<u64*>(ctl_s + kBaseOff);
  const char* slots_r = p.slots + (u64)f_recv * p.fifo_stride;
  char* slots_s = p.slots + (u64)f_send * p.fifo_stride;
  const char* inp = p.send[r];
  char* outp = p.recv[r];

  u64 clo, chi;
  {
    u64 q = (p.count + p.nchannels - 1) / p.nchannels;
    q = (q + align - 1) / align * align;
    const u64 a = q * c, b = q * (c + 1);
    clo = a < p.count ? a : p.count;
    chi = b < p.count ? b : p.count;
  }
  const u64 clen = chi - clo;
  const WaitCtx w{p.status, p.abort_word, p.timeout_ns, c * P + r, p.op};

  if (threadIdx.x == 0) {
    s_rbase = ld_relaxed(base_recv);
    s_sbase = ld_relaxed(base_send);
    m_tail = 0;
    m_head = 0;
    s_done = 0;
    s_stop = op_begin(w) ? 1 : 0;
    for (int k = 0; k < kRStages; ++k) {
      mbar_init(smem_addr(&full[k]), 1);
      mbar_init(smem_addr(&computed[k]), 1);
      mbar_init(smem_addr(&empty[k]), 1);
    }
    if (leader_cta) {
      for (int k = 0; k < p.nslots; ++k) {
        mbar_init(smem_addr(&bars_send[k]), 1u);
        mbar_init(smem_addr(&bars_recv[k]), 1u);
      }
    }
    mbar_init_fence();
  }
  cluster_sync_all();
  const u64 rbase = s_rbase, sbase = s_sbase;
  const bool run = clen > 0 && s_stop == 0;
  const uint32_t sm0 = smem_addr(stage_mem);
  const uint32_t bs0 = map_to_rank(smem_addr(&bars_send[0]), leader);
  const uint32_t br0 = map_to_rank(smem_addr(&bars_recv[0]), leader);
  const u64 pol_slot = policy_evict_last();
  const u64 pol_user = policy_evict_first();

  // number of receive and send slot-steps of this rank on this channel
  u64 total_recv = 0, total_send = 0;
  if (run) count_steps(clen, (u64)P, ce, align, epl, r, &total_recv, &total_send);

  if (run) {
    if (warp == 0 && lane == 0) {
      // ---------------- loader ----------------
      RingWalk wk;
      wk.init(clen, (u64)P, ce, align, epl, es, (u64)G, (u64)g, r);
      u64 j = 0, tcache = 0;
      while (!wk.done) {
        if (wk.first() && kind_recv(wk.kind)) {
          if (!wait_mirror(&m_tail, rbase + wk.rs + 1, tcache, w, XP_WAIT_TAIL)) break;
          fence_proxy_async_global();
        }
        const uint32_t k = (uint32_t)(j % K);
        if (j >= K && !mbar_wait_cta(smem_addr(&empty[k]), (uint32_t)(((j / K) - 1) & 1), w)) break;
        const uint32_t nb = entry_bytes(wk.st, wk.e);
        const u64 boff = (clo + wk.kstart + wk.o) * es + wk.st.b0 + wk.e * kRChunk;
        const u64 soff = wk.st.b0 + wk.e * kRChunk;
        const uint32_t bufA = sm0 + k * 2 * kRChunk, bufB = bufA + kRChunk;
        const bool red = kind_reduce(wk.kind);
        mbar_arrive_expect_tx(smem_addr(&full[k]), nb * (red ? 2u : 1u));
        if (nb) {
          if (kind_recv(wk.kind))
            bulk_load(bufA, slots_r + ((rbase + wk.rs) % N) * S + soff, nb, smem_addr(&full[k]), pol_slot);
          else
            bulk_load(bufA, inp + boff, nb, smem_addr(&full[k]), pol_user);
          if (red) bulk_load(bufB, inp + boff, nb, smem_addr(&full[k]), pol_user);
        }
        ++j;
        wk.next();
      }
      // every issued load must land before the CTA may exit
      for (u64 i = (j > K ? j - K : 0); i < j; ++i)
        mbar_wait_cta(smem_addr(&full[i % K]), (uint32_t)((i / K) & 1), w);
    } else if (warp >= 1 && warp <= kRComputeWarps) {
      // ---------------- compute ----------------
      const int ct = threadIdx.x - 32;
      RingWalk wk;
      wk.init(clen, (u64)P, ce, align, epl, es, (u64)G, (u64)g, r);
      u64 j = 0, tcache = 0, hcache = 0;
      while (!wk.done) {
        const uint32_t k = (uint32_t)(j % K);
        int ok = mbar_wait_cta(smem_addr(&full[k]), (uint32_t)((j / K) & 1), w) ? 1 : 0;
        if (!compute_vote(ok)) break;
        const uint32_t nb = entry_bytes(wk.st, wk.e);
        const bool red = kind_reduce(wk.kind);
        char* bufA = stage_mem + (u64)k * 2 * kRChunk;
        if (red) {
          V* A = reinterpret_cast<V*>(bufA);
          const V* B = reinterpret_cast<const V*>(bufA + kRChunk);
          for (uint32_t i = ct; i < nb / 16; i += 32 * kRComputeWarps) A[i] = add4(A[i], B[i]);
        }
        const bool rag = wk.last() && wk.st.rag != 0;
        if (rag && ct == 0) {
          // the buffer's last < 16 bytes: plain loads and stores, after the
          // step's tail (receive) and credit (send) are visible to this thread
          ok = 1;
          if (kind_recv(wk.kind)) ok = wait_mirror(&m_tail, rbase + wk.rs + 1, tcache, w, XP_WAIT_TAIL);
          const u64 sstep = sbase + wk.ss;
          if (ok && kind_send(wk.kind) && sstep + 1 > N)
            ok = wait_mirror(&m_head, sstep + 1 - N, hcache, w, XP_WAIT_HEAD);
          if (ok) {
            const u64 roff = wk.st.b0 + wk.st.fb;
            const u64 eoff = (clo + wk.kstart + wk.o) * es + roff;
            for (u64 x = 0; x < wk.st.rag; x += es) {
              T a;
              if (kind_recv(wk.kind))
                a = __ldcg(reinterpret_cast<const T*>(slots_r + ((rbase + wk.rs) % N) * S + roff + x));
              else
                a = __ldcs(reinterpret_cast<const T*>(inp + eoff + x));
              if (red) a = add1(a, __ldcs(reinterpret_cast<const T*>(inp + eoff + x)));
              if (kind_send(wk.kind)) __stcg(reinterpret_cast<T*>(slots_s + (sstep % N) * S + roff + x), a);
              if (kind_out(wk.kind)) __stcs(reinterpret_cast<T*>(outp + eoff + x), a);
            }
          }
        }
        if (red) fence_proxy_async_shared();   // these smem writes are read by bulk stores
        compute_barrier();
        if (ct == 0) {
          // The received slot's bytes of this stripe are in shared memory (and
          // its ragged bytes were read above): the reads are complete, so the
          // signal carries no ordering.
          if (kind_recv(wk.kind) && wk.last()) mbar_arrive_cluster_relaxed(br0 + 8u * (uint32_t)((rbase + wk.rs) % N));
          mbar_arrive_local(smem_addr(&computed[k]));
        }
        ++j;
        wk.next();
      }
    } else if (warp == 5 && lane == 0) {
      // ---------------- storer ----------------
      RingWalk wk;
      wk.init(clen, (u64)P, ce, align, epl, es, (u64)G, (u64)g, r);
      u64 j = 0, hcache = 0;
      long long pending = -1;   // send slot-step whose completion report is deferred
      int since = 0;
      bool ok = true;
      while (!wk.done && ok) {
        const uint32_t k = (uint32_t)(j % K);
        if (wk.first() && kind_send(wk.kind)) {
          const u64 step = sbase + wk.ss;
          if (step + 1 > N && hcache < step + 1 - N) {
            const u64 h = ld_acquire_cta_shared(&m_head);
            if (h >= step + 1 - N) {
              hcache = h;
            } else {
              if (pending >= 0) {
                bulk_wait<0>();
                fence_proxy_async_global();
                st_release_cta_shared(&s_done, (u64)pending + 1);
                pending = -1;
              }
              if (!wait_mirror(&m_head, step + 1 - N, hcache, w, XP_WAIT_HEAD)) { ok = false; break; }
            }
          }
          fence_proxy_async_global();
        }
        {
          // The next entry may depend, around the ring, on the send step whose
          // completion is still unreported: report it before blocking.
          const uint32_t cb = smem_addr(&computed[k]);
          const uint32_t par = (uint32_t)((j / K) & 1);
          if (!mbar_try_wait_cta(cb, par)) {
            if (pending >= 0) {
              bulk_wait<0>();
              fence_proxy_async_global();
              st_release_cta_shared(&s_done, (u64)pending + 1);
              pending = -1;
            }
            if (!mbar_wait_cta(cb, par, w)) { ok = false; break; }
          }
        }
        const uint32_t nb = entry_bytes(wk.st, wk.e);
        const uint32_t bufA = sm0 + k * 2 * kRChunk;
        if (nb) {
          const u64 soff = wk.st.b0 + wk.e * kRChunk;
          if (kind_send(wk.kind)) bulk_store(slots_s + ((sbase + wk.ss) % N) * S + soff, bufA, nb, pol_slot);
          if (kind_out(wk.kind))
            bulk_store(outp + (clo + wk.kstart + wk.o) * es + wk.st.b0 + wk.e * kRChunk, bufA, nb, pol_user);
        }
        bulk_commit();
        bulk_wait_read<kRStoresInFlight>();
        if (j >= (u64)kRStoresInFlight) mbar_arrive_local_relaxed(smem_addr(&empty[(j - kRStoresInFlight) % K]));
        if (pending >= 0 && ++since == kRDefer) {
          bulk_wait<kRDefer>();
          fence_proxy_async_global();
          st_release_cta_shared(&s_done, (u64)pending + 1);
          pending = -1;
        }
        if (kind_send(wk.kind) && wk.last()) {
          if (pending >= 0) {
            bulk_wait<0>();
            fence_proxy_async_global();
            st_release_cta_shared(&s_done, (u64)pending + 1);
          }
          pending = (long long)wk.ss;
          since = 0;
        }
        ++j;
        wk.next();
      }
      bulk_wait<0>();
      if (ok && pending >= 0) {
        fence_proxy_async_global();
        st_release_cta_shared(&s_done, (u64)pending + 1);
      }
    } else if (warp == 6 && lane == 0) {
      // ---------------- watcher ----------------
      const u64 target_t = rbase + total_recv;
      const u64 target_h = (sbase + total_send > N) ? sbase + total_send - N : 0;
      u64 seen_t = 0, seen_h = 0;
      WaitClock clk;
      while (seen_t < target_t || seen_h < target_h) {
        bool prog = false;
        if (seen_t < target_t) {
          const u64 v = ld_acquire(tail_recv);
          if (v > seen_t) {
            seen_t = v;
            st_release_cta_shared(&m_tail, v);
            prog = true;
          }
        }
        if (seen_h < target_h) {
          const u64 v = ld_acquire(head_send);
          if (v > seen_h) {
            seen_h = v;
            st_release_cta_shared(&m_head, v);
            prog = true;
          }
        }
        if (prog)
          clk = WaitClock();
        else if (!clk.tick(w, seen_t < target_t ? XP_WAIT_TAIL : XP_WAIT_HEAD, seen_t, target_t))
          break;
      }
    } else if (warp == 7 && lane == 0) {
      // ---------------- signaler ----------------
      u64 done = 0;
      for (u64 s = 0; s < total_send; ++s) {
        if (!wait_mirror(&s_done, s + 1, done, w, XP_WAIT_SLOT_BARRIER)) break;
        mbar_arrive_cluster(bs0 + 8u * (uint32_t)((sbase + s) % N));
      }
    } else if (warp == 8 && lane == 0 && leader_cta) {
      // ---------------- tail publisher (successor's FIFO) ----------------
      u64 s = 0;
      unsigned max_occ = 0;
      for (; s < total_send; ++s) {
        const u64 step = sbase + s;
        if (!mbar_wait(smem_addr(&bars_send[step % N]), (uint32_t)((s / N) & 1), w, XP_WAIT_SLOT_BARRIER, step)) break;
        st_release(tail_send, step + 1);
        const u64 h = ld_relaxed(head_send);
        const u64 occ = step + 1 - h;
        if (h > step + 1 || occ > N) {
          report(w, XP_ERR_BOUNDS, XP_WAIT_OCCUPANCY, occ, N);
          break;
        }
        if (occ > max_occ) max_occ = (unsigned)occ;
      }
      note_occupancy(p.status, p.op, max_occ);
    } else if (warp == 9 && lane == 0 && leader_cta) {
      // ---------------- head publisher (own FIFO) ----------------
      u64 s = 0;
      for (; s < total_recv; ++s) {
        const u64 step = rbase + s;
        if (!mbar_wait(smem_addr(&bars_recv[step % N]), (uint32_t)((s / N) & 1), w, XP_WAIT_SLOT_BARRIER, step)) break;
        st_release(head_recv, step + 1);
      }
      if (s == total_recv) st_relaxed(base_recv, rbase + total_recv);
    }
  }
  __syncwarp();
  cluster_sync_all();
}

template __global__ void ring_tma_kernel<float, float4>(const RingParams);
template __global__ void ring_tma_kernel<int, int4>(const RingParams);

void* ring_tma_kernel_ptr(int dtype) {
  if (dtype == XP_F32) return reinterpret_cast<void*>(&ring_tma_kernel<float, float4>);
  if (dtype == XP_I32) return reinterpret_cast<void*>(&ring_tma_kernel<int, int4>);
  return nullptr;
}
int ring_tma_threads() { return kRThreads; }
int ring_tma_smem() { return kRSmem; }

}  // namespace xp
