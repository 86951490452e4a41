// SIMPLE and zero-copy channel kernels.
//
// One thread-block cluster per channel.  SIMPLE: CTAs [0, G) are the sender
// lanes and [G, G + GR) the receiver lanes; zero copy: [0, G) senders and
// CTA G the receiver.  Every CTA has kCopyWarps copy warps and one publisher warp.
// Each slot-step is split into G*kCopyWarps contiguous 16-byte-vector pieces,
// one per copy warp of the side; a warp that finished its piece arrives
// (release, cluster scope) on the slot's mbarrier in the side's leader CTA
// (lane 0).  The leader's publisher thread waits for all G*kCopyWarps
// arrivals of the slot and then publishes the one channel-wide counter:
// tail = step + 1 on the sender side, head = step + 1 on the receiver side
// ("NCCL transport data transfer (二)", copy mode and zero copy).  Because
// sender and receiver of a channel are CTAs of one cluster, they are always
// co-resident: a waiting side can never starve the side it waits for.
#include <cuda_runtime.h>

#include "xp_device.cuh"

namespace xp {

__device__ __forceinline__ bool sticky_stop(const WaitCtx& w) {
  if (op_begin(w)) return true;
  return false;
}

template <bool kZeroCopy>
__global__ void __launch_bounds__(kP2pThreads, 1) p2p_kernel(const P2pParams p) {
  __shared__ __align__(8) u64 bars[kMaxSlots];
  __shared__ u64 s_base;
  __shared__ int s_stop;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const unsigned crank = cluster_ctarank();
  const int ch = blockIdx.x / p.csize;
  const int G = p.lanes;                          // sender lanes
  const bool sender = crank < (unsigned)G;
  const int lane_id = sender ? (int)crank : (int)crank - G;
  const unsigned leader = sender ? 0u : (unsigned)G;
  const int GS = (sender || kZeroCopy) ? G : p.rlanes;   // lanes of this CTA's side
  const bool leader_cta = crank == leader;
  const u64 N = (u64)p.nslots;
  const u64 S = p.slot_bytes;

  char* ctl = p.ctl + (u64)ch * kCtlBytes;
  u64* tail = reinterpret_cast<u64*>(ctl + kTailOff);
  u64* head = reinterpret_cast<u64*>(ctl + kHeadOff);
  u64* ptrx = reinterpret_cast<u64*>(ctl + kPtrxOff);
  u64* basew = reinterpret_cast<u64*>(ctl + kBaseOff);
  long long* sizew = reinterpret_cast<long long*>(ctl + kSizeOff);
  char* slots = p.slots + (u64)ch * p.ch_stride;

  u64 lo, hi;
  channel_range(p.nbytes, p.nchannels, ch, &lo, &hi);
  const u64 len = hi - lo;
  const u64 nsteps = (len + S - 1) / S;
  const WaitCtx w{p.status, p.abort_word, p.timeout_ns, ch, p.op};

  if (threadIdx.x == 0) {
    s_base = ld_relaxed(basew);
    s_stop = sticky_stop(w) ? 1 : 0;
    if (leader_cta) {
      const uint32_t count = (uint32_t)(GS * kCopyWarps);
      for (int k = 0; k < p.nslots; ++k) mbar_init(smem_addr(&bars[k]), count);
      mbar_init_fence();
    }
  }
  cluster_sync_all();   // barriers initialised before any remote arrive
  const u64 base = s_base;
  const bool run = nsteps > 0 && s_stop == 0;
  ChanStats* cs = p.stats ? p.stats + ch : nullptr;
  if (cs && sender && leader_cta && threadIdx.x == 0) {
    const u64 t = globaltimer();
    cs->steps = run ? nsteps : 0;
    cs->t_start = t;
    cs->send_polls = cs->recv_polls = 0;
    if (!run) cs->t_end = t;
  }

  if (run && warp < kCopyWarps) {
    const u64 parts = (u64)GS * kCopyWarps;
    const u64 my_piece = (u64)lane_id * kCopyWarps + warp;
    const uint32_t bar0 = map_to_rank(smem_addr(&bars[0]), leader);
    if (sender) {
      u64 hcache = 0;
      char* dstp = nullptr;
      if (kZeroCopy) {
        u64 v = 0;
        int ok = 1;
        if (lane == 0) ok = wait_word(ptrx, 1, v, w, XP_WAIT_PTR_EXCHANGE);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        v = __shfl_sync(0xffffffffu, v, 0);
        __syncwarp();
        if (!ok) goto done;
        dstp = reinterpret_cast<char*>(v);
      }
      for (u64 s = 0; s < nsteps; ++s) {
        const u64 step = base + s;
        if (step + 1 > N && !warp_wait_geq(head, step + 1 - N, hcache, w, XP_WAIT_HEAD)) break;
        const u64 off = s * S;
        const u64 sz = (len - off) < S ? (len - off) : S;
        u64 b0, b1;
        piece(sz, parts, my_piece, &b0, &b1);
        if (kZeroCopy) {
          warp_copy<LD_STREAM, ST_STREAM>(p.src + lo + off + b0, dstp + off + b0, b1 - b0);
        } else {
          warp_copy<LD_STREAM, ST_L2>(p.src + lo + off + b0, slots + (step % N) * S + b0, b1 - b0);
          if (my_piece == 0 && lane == 0) sizew[step % N] = (long long)sz;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(bar0 + 8u * (uint32_t)(step % N));
      }
    } else if (!kZeroCopy) {
      u64 tcache = 0;
      for (u64 r = 0; r < nsteps; ++r) {
        const u64 step = base + r;
        if (!warp_wait_geq(tail, step + 1, tcache, w, XP_WAIT_TAIL)) break;
        const u64 off = r * S;
        const u64 sz = (len - off) < S ? (len - off) : S;
        if (my_piece == 0 && lane == 0) {
          const long long got = (long long)ld_relaxed(reinterpret_cast<const u64*>(sizew + step % N));
          if (got != (long long)sz) report(w, XP_ERR_BOUNDS, XP_WAIT_SIZE_WORD, (u64)got, sz);
        }
        u64 b0, b1;
        piece(sz, parts, my_piece, &b0, &b1);
        warp_copy<LD_L2, ST_STREAM>(slots + (step % N) * S + b0, p.dst + lo + off + b0, b1 - b0);
        __syncwarp();
        // the piece of the slot has been read (the values went to dst): the
        // slot may be refilled, so no ordering is needed, and a release would
        // wait for this warp's stores to dst
        if (lane == 0) mbar_arrive_cluster_relaxed(bar0 + 8u * (uint32_t)(step % N));
      }
    }
  } else if (run && warp == kCopyWarps && lane == 0) {
    if (kZeroCopy && !sender) {
      // the zero-copy receiver: post the destination, echo tail into head
      u64 v = 0, tcache = 0;
      if (wait_word(ptrx, 0, v, w, XP_WAIT_PTR_EXCHANGE)) {
        st_release(ptrx, reinterpret_cast<u64>(p.dst + lo));
        u64 j = 0;
        for (; j < nsteps; ++j) {
          if (!wait_geq(tail, base + j + 1, tcache, w, XP_WAIT_TAIL)) break;
          st_release(head, base + j + 1);
        }
        if (j == nsteps) st_relaxed(basew, base + nsteps);
      }
      if (cs) cs->t_end = globaltimer();
    } else if (leader_cta) {
      u64 s = 0;
      unsigned max_occ = 0;
      for (; s < nsteps; ++s) {
        const u64 step = base + s;
        if (!mbar_wait(smem_addr(&bars[step % N]), (uint32_t)((s / N) & 1), w, XP_WAIT_SLOT_BARRIER, step))
          break;
        if (sender) {
          st_release(tail, step + 1);
          const u64 h = ld_relaxed(head);
          const u64 occ = step + 1 - h;
          if (h > step + 1 || occ > N) {
            report(w, XP_ERR_BOUNDS, XP_WAIT_OCCUPANCY, occ, N);
            break;
          }
          if (occ > max_occ) max_occ = (unsigned)occ;
        } else {
          st_release(head, step + 1);
        }
      }
      if (sender) {
        note_occupancy(p.status, p.op, max_occ);
        if (kZeroCopy && s == nsteps) {
          u64 hc = 0;
          if (wait_geq(head, base + nsteps, hc, w, XP_WAIT_HEAD)) st_release(ptrx, 0);
        }
      } else if (s == nsteps) {
        st_relaxed(basew, base + nsteps);
      }
      if (cs && !sender) cs->t_end = globaltimer();
    }
  }
done:
  __syncwarp();
  cluster_sync_all();   // no CTA leaves while others may still arrive on its barriers
}

template __global__ void p2p_kernel<false>(const P2pParams);
template __global__ void p2p_kernel<true>(const P2pParams);

void* p2p_kernel_ptr(bool zero_copy) {
  return zero_copy ? reinterpret_cast<void*>(&p2p_kernel<true>) : reinterpret_cast<void*>(&p2p_kernel<false>);
}

}  // namespace xp
