// LL channel kernel and the LL ping-pong latency kernel.
//
// LL ("RDMA and GPUDirect" §4.1: the data carries the flag and the receiver
// polls memory): a slot holds 16-byte lines {data0, flag0, data1, flag1};
// every line of slot-step s carries flag (s + 1) mod 2^32 in both halves,
// so zeroed memory never matches.  A line is written by one 16-byte store of
// two u64 halves {data | flag << 32}; each half is single-copy atomic, so a
// reader that sees both flags has both data words, even if it saw the line
// torn on an earlier poll.  There is no tail: the receiver polls the lines.
// head still returns slot credit.  One cluster of two CTAs per channel
// (sender, receiver); the receiver's copy warps arrive on a per-slot mbarrier
// and its publisher warp stores head.
#include <cuda_runtime.h>

#include "xp_device.cuh"

namespace xp {

constexpr int kLLBatch = 4;   // lines a receiver thread polls together

__global__ void __launch_bounds__(kLLThreads, 1) ll_kernel(const P2pParams p) {
  __shared__ __align__(8) u64 bars[kMaxSlots];
  __shared__ u64 s_base;
  __shared__ int s_stop;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const unsigned crank = cluster_ctarank();
  const int ch = blockIdx.x / 2;
  const bool sender = crank == 0;
  const u64 N = (u64)p.nslots;
  const u64 L = p.slot_bytes / 16;   // lines per slot

  char* ctl = p.ctl + (u64)ch * kCtlBytes;
  u64* head = reinterpret_cast<u64*>(ctl + kHeadOff);
  u64* basew = reinterpret_cast<u64*>(ctl + kBaseOff);
  char* slots = p.slots + (u64)ch * p.ch_stride;

  u64 lo, hi;
  channel_range(p.nbytes, p.nchannels, ch, &lo, &hi);
  const u64 nlines = (hi - lo) / 8;
  const u64 nsteps = (nlines + L - 1) / L;
  const WaitCtx w{p.status, p.abort_word, p.timeout_ns, ch, p.op};

  if (threadIdx.x == 0) {
    const u64 b0 = ld_relaxed(basew);   // in flight while op_begin reads the sticky word
    s_stop = op_begin(w) ? 1 : 0;
    s_base = b0;
    if (!sender) {
      for (int k = 0; k < p.nslots; ++k) mbar_init(smem_addr(&bars[k]), kCopyWarps);
      mbar_init_fence();
    }
  }
  // The two CTAs of the cluster share no shared memory (each side's barriers
  // are its own), so a block barrier is enough here and none is needed at
  // the end; the cluster launch still schedules sender and receiver together.
  __syncthreads();
  const u64 base = s_base;
  const bool run = nsteps > 0 && s_stop == 0;
  ChanStats* cs = p.stats ? p.stats + ch : nullptr;
  if (cs && sender && threadIdx.x == 0) {
    const u64 t = globaltimer();
    cs->steps = run ? nsteps : 0;
    cs->t_start = t;
    cs->send_polls = cs->recv_polls = 0;
    if (!run) cs->t_end = t;
  }
  const u64 T = 32ull * kCopyWarps;
  const u64 tid = threadIdx.x;

  if (run && warp < kCopyWarps) {
    const uint2* src = reinterpret_cast<const uint2*>(p.src + lo);
    uint2* dst = reinterpret_cast<uint2*>(p.dst + lo);
    if (sender) {
      u64 hcache = 0;
      for (u64 s = 0; s < nsteps; ++s) {
        const u64 step = base + s;
        if (step + 1 > N && !warp_wait_geq(head, step + 1 - N, hcache, w, XP_WAIT_HEAD)) break;
        const u64 first = s * L;
        const u64 nl = (nlines - first) < L ? (nlines - first) : L;
        const u64 flag = (u64)(uint32_t)(step + 1) << 32;
        char* slot = slots + (step % N) * p.slot_bytes;
        for (u64 i = tid; i < nl; i += T) {
          const uint2 d = __ldcs(src + first + i);
          ll_store(slot + 16 * i, flag | d.x, flag | d.y);
        }
      }
    } else {
      const uint32_t bar0 = smem_addr(&bars[0]);
      int failed = 0;
      u64 hcache = 0;
      for (u64 r = 0; r < nsteps && !failed; ++r) {
        const u64 step = base + r;
        // A warp with no lines in this step would not wait for anything:
        // keep it from arriving on slot step % N before that slot's previous
        // phase (step - N) has completed, i.e. before head passed step - N.
        if (r >= N && !warp_wait_geq(head, step + 1 - N, hcache, w, XP_WAIT_HEAD)) break;
        const u64 first = r * L;
        const u64 nl = (nlines - first) < L ? (nlines - first) : L;
        const uint32_t flag = (uint32_t)(step + 1);
        const char* slot = slots + (step % N) * p.slot_bytes;
        // A thread's lines of the step are polled kLLBatch at a time, all
        // loads in flight together; only lines whose flags are not there
        // yet are loaded again.
        for (u64 i0 = tid; i0 < nl && !failed; i0 += T * kLLBatch) {
          u64 a[kLLBatch], b[kLLBatch];
          unsigned todo = 0;
#pragma unroll
          for (int q = 0; q < kLLBatch; ++q)
            if (i0 + q * T < nl) todo |= 1u << q;
          WaitClock clk;
          unsigned it = 0;
          while (todo) {
#pragma unroll
            for (int q = 0; q < kLLBatch; ++q)
              if (todo & (1u << q)) ll_load(slot + 16 * (i0 + q * T), a[q], b[q]);
            u64 seen = 0;   // the flags of a line still missing, for the report
#pragma unroll
            for (int q = 0; q < kLLBatch; ++q)
              if (todo & (1u << q)) {
                if ((uint32_t)(a[q] >> 32) == flag && (uint32_t)(b[q] >> 32) == flag) {
                  __stcs(dst + first + i0 + q * T, make_uint2((uint32_t)a[q], (uint32_t)b[q]));
                  todo &= ~(1u << q);
                } else {
                  seen = (a[q] >> 32) | ((b[q] >> 32) << 32);
                }
              }
            if (todo && (++it & 7u) == 0 && !clk.tick(w, XP_WAIT_LL_FLAG, seen, flag)) {
              failed = 1;
              break;
            }
          }
        }
        failed = __any_sync(0xffffffffu, failed);
        // The lines have been read (their values are in registers): the
        // slot may be refilled, so the signal needs no ordering, and a
        // release would wait for this warp's stores to dst.
        if (!failed && lane == 0) mbar_arrive_cluster_relaxed(bar0 + 8u * (uint32_t)(step % N));
      }
    }
  } else if (run && warp == kCopyWarps && lane == 0 && !sender) {
    u64 r = 0;
    for (; r < nsteps; ++r) {
      const u64 step = base + r;
      if (!mbar_wait(smem_addr(&bars[step % N]), (uint32_t)((r / N) & 1), w, XP_WAIT_SLOT_BARRIER, step)) break;
      st_release(head, step + 1);
    }
    if (r == nsteps) st_relaxed(basew, base + nsteps);
    if (cs) cs->t_end = globaltimer();
  }
}

// Ping-pong: CTA 0 (A) sends one line through `ab`, CTA 1 (B) answers
// through `ba`; `iters` round trips between two globaltimer reads.  Each
// side is the receiver of one FIFO and returns its head for every line.
__global__ void __launch_bounds__(32, 1) ll_pingpong_kernel(const PingParams p) {
  const unsigned crank = cluster_ctarank();
  const WaitCtx w{p.status, p.abort_word, p.timeout_ns, (int)crank, p.op};
  cluster_sync_all();
  if (threadIdx.x == 0 && !op_begin(w)) {
    const bool is_a = crank == 0;
    char* sctl = is_a ? p.ctl_ab : p.ctl_ba;
    char* rctl = is_a ? p.ctl_ba : p.ctl_ab;
    char* sslots = is_a ? p.slots_ab : p.slots_ba;
    const char* rslots = is_a ? p.slots_ba : p.slots_ab;
    const u64 Ns = (u64)(is_a ? p.nslots_ab : p.nslots_ba);
    const u64 Nr = (u64)(is_a ? p.nslots_ba : p.nslots_ab);
    const u64 Ss = is_a ? p.slot_bytes_ab : p.slot_bytes_ba;
    const u64 Sr = is_a ? p.slot_bytes_ba : p.slot_bytes_ab;
    u64* shead = reinterpret_cast<u64*>(sctl + kHeadOff);
    u64* rhead = reinterpret_cast<u64*>(rctl + kHeadOff);
    const u64 sbase = ld_relaxed(reinterpret_cast<u64*>(sctl + kBaseOff));
    const u64 rbase = ld_relaxed(reinterpret_cast<u64*>(rctl + kBaseOff));
    u64 hcache = 0;

    auto send_line = [&](u64 i) -> bool {
      const u64 s = sbase + i;
      if (s + 1 > Ns && !wait_geq(shead, s + 1 - Ns, hcache, w, XP_WAIT_HEAD)) return false;
      const u64 f = (u64)(uint32_t)(s + 1) << 32;
      ll_store(sslots + (s % Ns) * Ss, f | (uint32_t)i, f | (uint32_t)(i ^ 0x5a5a5a5au));
      return true;
    };
    auto recv_line = [&](u64 i) -> bool {
      const u64 r = rbase + i;
      const uint32_t f = (uint32_t)(r + 1);
      const char* line = rslots + (r % Nr) * Sr;
      u64 a, b;
      WaitClock clk;
      unsigned it = 0;
      for (;;) {
        ll_load(line, a, b);
        if ((uint32_t)(a >> 32) == f && (uint32_t)(b >> 32) == f) break;
        if ((++it & 7u) == 0 && !clk.tick(w, XP_WAIT_LL_FLAG, a >> 32, f)) return false;
      }
      if ((uint32_t)a != (uint32_t)i || (uint32_t)b != ((uint32_t)i ^ 0x5a5a5a5au)) {
        report(w, XP_ERR_BOUNDS, XP_WAIT_LL_FLAG, a, i);
        return false;
      }
      return true;
    };
    // Credit for line i goes back after the next line is sent: the release
    // orders this thread's memory traffic and would delay the reply if it
    // came first (measured: 1067 ns one way with it in front, 698 ns after).
    auto pub = [&](u64 i) { st_release(rhead, rbase + i + 1); };

    const u64 iters = (u64)p.iters;
    const u64 t0 = globaltimer();
    u64 i = 0;
    for (; i < iters; ++i) {
      if (is_a) {
        if (!send_line(i)) break;
        if (i > 0) pub(i - 1);
        if (!recv_line(i)) break;
        if (i + 1 == iters) pub(i);
      } else {
        if (!recv_line(i) || !send_line(i)) break;
        pub(i);
      }
    }
    const u64 t1 = globaltimer();
    if (i == iters) {
      if (is_a) *p.elapsed = t1 - t0;
      st_relaxed(reinterpret_cast<u64*>(rctl + kBaseOff), rbase + iters);
    }
  }
  __syncwarp();
  cluster_sync_all();
}

void* ll_kernel_ptr() { return reinterpret_cast<void*>(&ll_kernel); }
void* ll_pingpong_kernel_ptr() { return reinterpret_cast<void*>(&ll_pingpong_kernel); }

}  // namespace xp
