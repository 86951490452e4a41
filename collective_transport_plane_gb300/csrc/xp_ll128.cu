// LL128 channel kernel.
//
// LL128 ("RDMA and GPUDirect" §4: the data carries its flag in the last bytes
// written, and the receiver polls memory) with 128-byte lines: words 0..14
// (uint64) carry payload, word 15 is the flag, step + 1 for every line of
// slot-step `step`.  Eight threads own a line, 16 bytes each; the eighth
// holds payload word 14 and the flag.
//
// The flag is what the receiver waits for, so the payload of its line must
// be visible first.  PTX promises single-copy atomicity per element only,
// not for a 128-byte line ("RDMA and GPUDirect" §8 makes the same point for
// a NIC's writes: seeing the flag does not mean the data has landed), so
// the order is made explicit and paid for once per batch of lines instead
// of once per line:
//   sender   — store the payload of kBatch lines per thread, __syncwarp,
//              fence (release), store the batch's flags;
//   receiver — poll the batch's flags, fence (acquire), __syncwarp, load the
//              batch's payload.
// There is no tail; head returns slot credit.  One cluster of two CTAs per
// channel (sender, receiver); the receiver's copy warps arrive on a per-slot
// mbarrier and its publisher warp stores head.
#include <cuda_runtime.h>

#include "xp_device.cuh"

namespace xp {

namespace {

constexpr u64 kLineBytes = 128;
constexpr u64 kDataWords = 15;
constexpr int kBatch = 8;          // lines per thread between two fences

__device__ __forceinline__ void fence_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void st_v2(void* p, u64 a, u64 b) {
  asm volatile("st.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ void st_u64(void* p, u64 a) {
  asm volatile("st.global.u64 [%0], %1;" ::"l"(p), "l"(a) : "memory");
}
__device__ __forceinline__ void st_flag(void* p, u64 a) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(a) : "memory");
}
__device__ __forceinline__ u64 ld_flag(const void* p) {
  u64 v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ u64 ld_word(const void* p) {
  u64 v;
  asm volatile("ld.volatile.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

}  // namespace

__global__ void __launch_bounds__(kLLThreads, 1) ll128_kernel(const P2pParams p) {
  __shared__ __align__(8) u64 bars[kMaxSlots];
  __shared__ u64 s_base;
  __shared__ int s_stop;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const unsigned crank = cluster_ctarank();
  const int ch = blockIdx.x / 2;
  const bool sender = crank == 0;
  const u64 N = (u64)p.nslots;
  const u64 L = p.slot_bytes / kLineBytes;     // lines per slot
  const u64 W = L * kDataWords;                // payload words per slot-step

  char* ctl = p.ctl + (u64)ch * kCtlBytes;
  u64* head = reinterpret_cast<u64*>(ctl + kHeadOff);
  u64* basew = reinterpret_cast<u64*>(ctl + kBaseOff);
  char* slots = p.slots + (u64)ch * p.ch_stride;

  u64 lo, hi;
  channel_range(p.nbytes, p.nchannels, ch, &lo, &hi);
  const u64 nwords = (hi - lo) / 8;
  const u64 nsteps = (nwords + W - 1) / W;
  const WaitCtx w{p.status, p.abort_word, p.timeout_ns, ch};

  if (threadIdx.x == 0) {
    s_base = ld_relaxed(basew);
    s_stop = 0;
    if (*reinterpret_cast<volatile int*>(&p.status->sticky)) {
      s_stop = 1;
      if (atomicCAS(&p.status->code, 0, XP_ERR_ABORTED) == 0) p.status->where = XP_WAIT_STICKY;
    }
    if (!sender) {
      for (int k = 0; k < p.nslots; ++k) mbar_init(smem_addr(&bars[k]), kCopyWarps);
      mbar_init_fence();
    }
  }
  cluster_sync_all();
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
  // thread -> (line, 16-byte position in the line): a warp covers 4 lines
  // per pass, the copy warps G lines; loops run per warp (wline), so the
  // warp-wide barriers and votes inside them see every lane
  constexpr u64 G = 32ull * kCopyWarps / 8;
  const u64 wline = (u64)warp * 4;
  const u64 sub = (threadIdx.x >> 3) & 3;
  const u64 pos = threadIdx.x & 7;
  const bool flag_lane = pos == 7;

  if (run && warp < kCopyWarps) {
    const u64* src = reinterpret_cast<const u64*>(p.src + lo);
    u64* dst = reinterpret_cast<u64*>(p.dst + lo);
    if (sender) {
      u64 hcache = 0;
      for (u64 s = 0; s < nsteps; ++s) {
        const u64 step = base + s;
        if (step + 1 > N && !warp_wait_geq(head, step + 1 - N, hcache, w, XP_WAIT_HEAD)) break;
        const u64 left = nwords - s * W;
        const u64 nl = left >= W ? L : (left + kDataWords - 1) / kDataWords;
        const u64 flag = step + 1;
        char* slot = slots + (step % N) * p.slot_bytes;
        const u64* ssrc = src + s * W;
        for (u64 w0 = wline; w0 < nl; w0 += G * kBatch) {
          const u64 i0 = w0 + sub;
          // payload of up to kBatch lines: loads first, all in flight together
          u64 a[kBatch], b[kBatch];
#pragma unroll
          for (int q = 0; q < kBatch; ++q) {
            const u64 i = i0 + q * G;
            const u64 wd = i * kDataWords + 2 * pos;   // first payload word of this thread
            a[q] = b[q] = 0;
            if (i < nl) {
              if (wd < left) a[q] = __ldcs(reinterpret_cast<const unsigned long long*>(ssrc + wd));
              if (!flag_lane && wd + 1 < left) b[q] = __ldcs(reinterpret_cast<const unsigned long long*>(ssrc + wd + 1));
            }
          }
#pragma unroll
          for (int q = 0; q < kBatch; ++q) {
            const u64 i = i0 + q * G;
            if (i < nl) {
              char* line = slot + i * kLineBytes + 16 * pos;
              if (flag_lane) st_u64(line, a[q]);
              else st_v2(line, a[q], b[q]);
            }
          }
          // every payload store of the warp's lines before any of their flags
          __syncwarp();
          fence_gpu();
          if (flag_lane) {
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
              const u64 i = i0 + q * G;
              if (i < nl) st_flag(slot + i * kLineBytes + 8 * kDataWords, flag);
            }
          }
        }
      }
    } else {
      const uint32_t bar0 = smem_addr(&bars[0]);
      int failed = 0;
      u64 hcache = 0;
      for (u64 r = 0; r < nsteps && !failed; ++r) {
        const u64 step = base + r;
        // a warp with no lines in this step must not arrive on slot step % N
        // before that slot's previous phase has completed (head > step - N)
        if (r >= N && !warp_wait_geq(head, step + 1 - N, hcache, w, XP_WAIT_HEAD)) break;
        const u64 left = nwords - r * W;
        const u64 nl = left >= W ? L : (left + kDataWords - 1) / kDataWords;
        const u64 flag = step + 1;
        const char* slot = slots + (step % N) * p.slot_bytes;
        u64* sdst = dst + r * W;
        for (u64 w0 = wline; w0 < nl && !failed; w0 += G * kBatch) {
          const u64 i0 = w0 + sub;
          int ok = 1;
          if (flag_lane) {
            unsigned todo = 0;
#pragma unroll
            for (int q = 0; q < kBatch; ++q)
              if (i0 + q * G < nl) todo |= 1u << q;
            WaitClock clk;
            unsigned it = 0;
            while (todo) {
              u64 seen = 0;
#pragma unroll
              for (int q = 0; q < kBatch; ++q)
                if (todo & (1u << q)) {
                  const u64 f = ld_flag(slot + (i0 + q * G) * kLineBytes + 8 * kDataWords);
                  if (f == flag) todo &= ~(1u << q);
                  else seen = f;
                }
              if (todo && (++it & 7u) == 0 && !clk.tick(w, XP_WAIT_LL_FLAG, seen, flag)) {
                ok = 0;
                break;
              }
            }
          }
          // the flag loads, then the payload loads of every thread of the warp
          fence_gpu();
          __syncwarp();
          if (__any_sync(0xffffffffu, !ok)) {
            failed = 1;
            break;
          }
          u64 a[kBatch], b[kBatch];
#pragma unroll
          for (int q = 0; q < kBatch; ++q) {
            const u64 i = i0 + q * G;
            a[q] = b[q] = 0;
            if (i < nl) {
              const char* line = slot + i * kLineBytes + 16 * pos;
              if (flag_lane) a[q] = ld_word(line);
              else ll_load(line, a[q], b[q]);
            }
          }
#pragma unroll
          for (int q = 0; q < kBatch; ++q) {
            const u64 i = i0 + q * G;
            const u64 wd = i * kDataWords + 2 * pos;
            if (i < nl) {
              if (wd < left) __stcs(reinterpret_cast<unsigned long long*>(sdst + wd), a[q]);
              if (!flag_lane && wd + 1 < left) __stcs(reinterpret_cast<unsigned long long*>(sdst + wd + 1), b[q]);
            }
          }
        }
        failed = __any_sync(0xffffffffu, failed);
        // the lines are read (their values are in registers): the slot may
        // be refilled, so the signal needs no ordering
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
  __syncwarp();
  cluster_sync_all();
}

void* ll128_kernel_ptr() { return reinterpret_cast<void*>(&ll128_kernel); }

}  // namespace xp
