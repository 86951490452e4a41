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
// the order is made explicit and paid for once per chunk of lines instead
// of once per line:
//   sender   — the copy warps store a chunk's payload (kBatch lines per
//              thread) and arrive on the chunk's barrier (release); a
//              flagger warp waits for it, fences once and stores the
//              chunk's flags, so the copy warps never wait on a fence;
//   receiver — poll the batch's flags (with acquire one per sender lane the
//              batch's lines come from, the rest relaxed), __syncwarp, load
//              the batch's payload.
// There is no tail; head returns slot credit.  A channel runs on G sender
// and GR receiver CTAs ("lanes"), consecutive in the grid and resident
// together (a cooperative grid, else one cluster per channel): sender lane g
// owns the fixed stripe of ceil(L / G) lines of every slot, receiver lane r
// that of ceil(L / GR) lines, and each receiver lane keeps a head of its own;
// a sender lane refills a slot's stripe once every receiver lane whose
// stripe meets it has returned the credit.  The receiver's copy warps
// arrive on a per-slot mbarrier and its publisher warp stores the lane's
// head.  The last receiver lane of a channel to finish an operation moves
// the channel's step base on and sets every lane's head to it, so the next
// operation may cut the slots into different stripes.
#include <cuda_runtime.h>

#include "xp_device.cuh"

namespace xp {

namespace {

constexpr int kL128Warps = 16;     // copy warps per CTA (two more: producer and flagger, or publisher)
constexpr int kL128Threads = 32 * (kL128Warps + 2);
constexpr u64 kLineBytes = 128;
constexpr u64 kDataWords = 15;
constexpr int kBatch = 8;          // lines per thread per chunk
constexpr u64 kChunkLines = 32ull * kL128Warps / 8 * kBatch;   // lines the copy warps write per stage
// a stage holds a chunk's payload from the 16-byte boundary at or below its
// first byte: at most 8 bytes of lead plus 120 bytes per line
constexpr uint32_t kStageBytes = (uint32_t)((kChunkLines * 8 * kDataWords + 8 + 15) / 16 * 16);
constexpr int kStages = 3;
constexpr int kMaxLL128Lanes = 8;
constexpr u64 kRowLines = 32ull * kL128Warps / 8 * kLineBytes;   // bytes of slot between a thread's lines
constexpr uint32_t kRowPayload = (uint32_t)(32ull * kL128Warps / 8 * 8 * kDataWords);   // and of payload

constexpr u64 kDirectBytes = 8192;   // chunks of less payload are read from src directly

// End of the bulk-staged part [a0, end) of a chunk whose payload is bytes
// [b0, b1) of src: the 16-byte boundary at or above b1 if that is still
// inside the channel's range [., hi), else the one below; nothing is staged
// for a short chunk, whose copy would only add the bulk copy's latency.
__device__ __forceinline__ u64 staged_end(u64 b0, u64 b1, u64 hi) {
  const u64 a0 = b0 & ~15ull;
  if (b1 - b0 < kDirectBytes) return a0;
  const u64 up = (b1 + 15) & ~15ull;
  return up <= hi ? up : b1 & ~15ull;
}

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
__device__ __forceinline__ u64 ld_flag_acquire(const void* p) {
  u64 v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ u64 atom_add_acq_rel(u64* p, u64 v) {
  u64 old;
  asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}
__device__ __forceinline__ u64 ld_shared_u64(uint32_t saddr) {
  u64 v;
  asm volatile("ld.shared.u64 %0, [%1];" : "=l"(v) : "r"(saddr) : "memory");
  return v;
}
__device__ __forceinline__ u64 ld_word(const void* p) {
  u64 v;
  asm volatile("ld.volatile.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

}  // namespace

__global__ void __launch_bounds__(kL128Threads, 1) ll128_kernel(const P2pParams p) {
  extern __shared__ __align__(128) unsigned char stage_mem[];
  __shared__ __align__(8) u64 bars[kMaxSlots];
  __shared__ __align__(8) u64 full[kStages], empty[kStages], pdone[kStages];
  __shared__ u64 s_base;
  __shared__ int s_stop;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Channel ch runs G sender and GR receiver CTAs, consecutive in the grid
  // (a cooperative grid, or one cluster per channel).
  const unsigned G = (unsigned)p.lanes;
  const unsigned GR = (unsigned)p.rlanes;
  const int ch = (int)(blockIdx.x / (G + GR));
  const unsigned crank = blockIdx.x % (G + GR);
  const bool sender = crank < G;
  const unsigned g = sender ? crank : crank - G;   // lane within the side
  const u64 N = (u64)p.nslots;
  const u64 L = p.slot_bytes / kLineBytes;     // lines per slot
  const u64 W = L * kDataWords;                // payload words per slot-step
  const u64 LgS = (L + G - 1) / G;             // stripe of lines per sender lane
  const u64 LgR = (L + GR - 1) / GR;           // and per receiver lane
  const u64 Lg = sender ? LgS : LgR;
  const u64 l0 = g * Lg < L ? g * Lg : L;
  const u64 l1 = l0 + Lg < L ? l0 + Lg : L;

  char* ctl = p.ctl + (u64)ch * kCtlBytes;
  // receiver lane 0's head is the channel's head word; lanes 1 .. 7 keep
  // theirs on lines 1 .. 7 of the channel's block of the arrival region, whose
  // line 0 counts the receiver lanes that have finished the operation
  u64* arr = p.arr + (u64)ch * (kArrBytes / 8);
  auto head_of = [&](unsigned rl) { return rl == 0 ? reinterpret_cast<u64*>(ctl + kHeadOff) : arr + 16 * rl; };
  u64* head = head_of(g);   // the receiver's own
  // a sender lane refills a slot's lines [l0, l1) once every receiver lane
  // whose stripe meets them has returned the credit
  const unsigned rlo = sender && l1 > l0 ? (unsigned)(l0 / LgR) : 0;
  const unsigned rhi = sender && l1 > l0 ? (unsigned)((l1 - 1) / LgR) : 0;
  u64* basew = reinterpret_cast<u64*>(ctl + kBaseOff);
  char* slots = p.slots + (u64)ch * p.ch_stride;

  u64 lo, hi;
  channel_range(p.nbytes, p.nchannels, ch, &lo, &hi);
  const u64 nwords = (hi - lo) / 8;
  const u64 nsteps = (nwords + W - 1) / W;
  const WaitCtx w{p.status, p.abort_word, p.timeout_ns, ch, p.op};

  if (threadIdx.x == 0) {
    const u64 b0 = ld_relaxed(basew);   // in flight while op_begin reads the sticky word
    s_stop = op_begin(w) ? 1 : 0;
    s_base = b0;
    if (!sender) {
      for (int k = 0; k < p.nslots; ++k) mbar_init(smem_addr(&bars[k]), kL128Warps);
      mbar_init_fence();
    }
    if (sender) {
      for (int k = 0; k < kStages; ++k) {
        mbar_init(smem_addr(&full[k]), 1);
        mbar_init(smem_addr(&empty[k]), kL128Warps + 1);   // the copy warps and the flagger
        mbar_init(smem_addr(&pdone[k]), kL128Warps);       // the chunk's payload is stored
      }
      mbar_init_fence();
    }
  }
  // Each CTA's barriers are its own (no shared memory is used across CTAs),
  // so a block barrier is enough here and none is needed at the end; the
  // launch (cooperative, or a cluster per channel) keeps the channel's CTAs
  // resident together.
  __syncthreads();
  const u64 base = s_base;
  const bool run = nsteps > 0 && s_stop == 0;
  ChanStats* cs = p.stats ? p.stats + ch : nullptr;
  if (cs && sender && g == 0 && threadIdx.x == 0) {
    const u64 t = globaltimer();
    cs->steps = run ? nsteps : 0;
    cs->t_start = t;
    cs->send_polls = cs->recv_polls = 0;
    if (!run) cs->t_end = t;
  }
  // thread -> (line, 16-byte position in the line): a warp covers 4 lines
  // of the lane's stripe per pass, the copy warps P lines; loops run per
  // warp (wline), so the warp-wide barriers and votes inside them see every
  // lane
  constexpr u64 P = 32ull * kL128Warps / 8;
  const u64 wline = l0 + (u64)warp * 4;
  const u64 sub = (threadIdx.x >> 3) & 3;
  const u64 pos = threadIdx.x & 7;
  const bool flag_lane = pos == 7;

  if (run && warp < kL128Warps) {
    u64* dst = reinterpret_cast<u64*>(p.dst + lo);
    if (sender) {
      // The producer thread (below) stages each chunk of the lane's payload
      // in shared memory with a bulk copy; the copy warps turn it into lines.
      const uint32_t sm0 = smem_addr(stage_mem);
      u64 hcache[kMaxLL128Lanes] = {};
      u64 j = 0;           // chunks consumed
      int failed = 0;
      for (u64 s = 0; s < nsteps && !failed; ++s) {
        const u64 step = base + s;
        if (step + 1 > N && l1 > l0) {
          for (unsigned rl = rlo; rl <= rhi && !failed; ++rl)
            if (!warp_wait_geq(head_of(rl), step + 1 - N, hcache[rl], w, XP_WAIT_HEAD)) failed = 1;
          if (failed) break;
        }
        const u64 left = nwords - s * W;
        const u64 nla = left >= W ? L : (left + kDataWords - 1) / kDataWords;
        const u64 nl = nla < l1 ? nla : l1;         // end of this lane's lines in the step
        char* slot = slots + (step % N) * p.slot_bytes;
        const u64 sbyte = lo + 8 * s * W;           // src offset of the step's first payload word
        for (u64 c0 = l0; c0 < nl; c0 += kChunkLines, ++j) {
          const int k = (int)(j % kStages);
          if (!mbar_wait_cta(smem_addr(&full[k]), (uint32_t)((j / kStages) & 1), w)) {
            failed = 1;
            break;
          }
          const u64 c1 = c0 + kChunkLines < nl ? c0 + kChunkLines : nl;
          const u64 wend = kDataWords * c1 < left ? kDataWords * c1 : left;
          const u64 b0 = sbyte + 8 * kDataWords * c0;
          const u64 a0 = b0 & ~15ull;
          const u64 a1 = staged_end(b0, sbyte + 8 * wend, hi);   // staged: [a0, a1); a word past it is read directly
          const u64 i0 = c0 + (u64)warp * 4 + sub;
          const uint32_t stage = sm0 + k * kStageBytes;
          if (kDataWords * c1 <= left && sbyte + 8 * wend <= a1) {
            // every line of the chunk is whole payload and staged: fixed
            // strides, one check per line
            const uint32_t so = stage + (uint32_t)(b0 - a0) + (uint32_t)(8 * kDataWords * ((u64)warp * 4 + sub) + 16 * pos);
            char* line = slot + i0 * kLineBytes + 16 * pos;
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
              if (i0 + q * P < c1) {
                const u64 x = ld_shared_u64(so + q * kRowPayload);
                if (flag_lane) {
                  st_u64(line + q * kRowLines, x);
                } else {
                  st_v2(line + q * kRowLines, x, ld_shared_u64(so + q * kRowPayload + 8));
                }
              }
            }
            __syncwarp();
            if (lane == 0) {
              mbar_arrive_local_relaxed(smem_addr(&empty[k]));
              mbar_arrive_local(smem_addr(&pdone[k]));
            }
            continue;
          }
          u64 a[kBatch], b[kBatch];
#pragma unroll
          for (int q = 0; q < kBatch; ++q) {
            const u64 i = i0 + q * P;
            const u64 wd = i * kDataWords + 2 * pos;   // first payload word of this thread in the step
            a[q] = b[q] = 0;
            if (i < c1) {
              const u64 g = sbyte + 8 * wd;
              if (wd < left) a[q] = g < a1 ? ld_shared_u64(stage + (uint32_t)(g - a0))
                                           : __ldcs(reinterpret_cast<const unsigned long long*>(p.src + g));
              if (!flag_lane && wd + 1 < left)
                b[q] = g + 8 < a1 ? ld_shared_u64(stage + (uint32_t)(g + 8 - a0))
                                  : __ldcs(reinterpret_cast<const unsigned long long*>(p.src + g + 8));
            }
          }
#pragma unroll
          for (int q = 0; q < kBatch; ++q) {
            const u64 i = i0 + q * P;
            if (i < c1) {
              char* line = slot + i * kLineBytes + 16 * pos;
              if (flag_lane) st_u64(line, a[q]);
              else st_v2(line, a[q], b[q]);
            }
          }
          // the stage's values are in registers (the stores above used them)
          __syncwarp();
          if (lane == 0) {
            mbar_arrive_local_relaxed(smem_addr(&empty[k]));
            mbar_arrive_local(smem_addr(&pdone[k]));
          }
        }
      }
    } else {
      const uint32_t bar0 = map_to_rank(smem_addr(&bars[0]), cluster_ctarank());
      int failed = 0;
      u64 hcache = 0;
      for (u64 r = 0; r < nsteps && !failed; ++r) {
        const u64 step = base + r;
        // a warp with no lines in this step must not arrive on slot step % N
        // before that slot's previous phase has completed (head > step - N)
        if (r >= N && !warp_wait_geq(head, step + 1 - N, hcache, w, XP_WAIT_HEAD)) break;
        const u64 left = nwords - r * W;
        const u64 nla = left >= W ? L : (left + kDataWords - 1) / kDataWords;
        const u64 nl = nla < l1 ? nla : l1;
        const u64 flag = step + 1;
        const char* slot = slots + (step % N) * p.slot_bytes;
        u64* sdst = dst + r * W;
        // first sender-lane boundary above this thread's lines (a batch that
        // crosses one holds lines of two senders, ordered by two fences)
        u64 nb = ((u64)((uint32_t)(wline + sub) / (uint32_t)LgS) + 1) * LgS;
        for (u64 w0 = wline; w0 < nl && !failed; w0 += P * kBatch) {
          const u64 i0 = w0 + sub;
          // every line of the step up to nl carries payload in every word:
          // fixed strides, one check per line
          const bool whole = kDataWords * nl <= left;
          const char* line = slot + i0 * kLineBytes + 16 * pos;
          // Every flag of the batch is polled with relaxed loads, all in
          // flight together, except the last line's (the anchor), which is
          // loaded with acquire, and, when the batch's lines cross from one
          // sender lane's stripe into the next, also the last line before
          // the boundary.  A sender's copy warps store a chunk's payload
          // before its flagger's fence for the chunk, and the flagger stores
          // the chunk's flags after that fence; the flagger takes its chunks
          // in order, so that fence also follows the payload of the lane's
          // earlier chunks.  An acquire that sees a flag therefore makes the
          // payload of every line of the batch from that sender lane, up to
          // that line, visible to the loads below (the warp barrier passes
          // that on to the other threads).  A batch whose lines come from
          // three or more sender lanes (stripes shorter than the batch)
          // loads every flag with acquire.
          int ok = 1;
          if (flag_lane) {
            unsigned todo = 0;
#pragma unroll
            for (int q = 0; q < kBatch; ++q)
              if (i0 + q * P < nl) todo |= 1u << q;
            const unsigned anchor = todo ? 1u << (31 - __clz(todo)) : 0u;
            while (nb <= i0) nb += LgS;
            unsigned anchor2 = 0;
            bool every = false;   // three or more senders: every flag with acquire
            if (anchor) {
              const u64 itop = i0 + (31 - __clz(anchor)) * P;
              if (itop >= nb + LgS) every = true;
              else if (itop >= nb) anchor2 = 1u << (unsigned)((nb - 1 - i0) / P);
            }
            WaitClock clk;
            unsigned it = 0;
            while (todo) {
              u64 seen = 0;
              if (every) {
#pragma unroll
                for (int q = 0; q < kBatch; ++q)
                  if (todo & (1u << q)) {
                    const u64 f = ld_flag_acquire(line + 8 + q * kRowLines);
                    if (f == flag) todo &= ~(1u << q);
                    else seen = f;
                  }
              } else {
#pragma unroll
                for (int q = 0; q < kBatch; ++q)
                  if ((todo & ~(anchor | anchor2)) & (1u << q)) {
                    const u64 f = ld_flag(line + 8 + q * kRowLines);
                    if (f == flag) todo &= ~(1u << q);
                    else seen = f;
                  }
                if (todo & anchor2) {
                  const u64 f = ld_flag_acquire(line + 8 + (31 - __clz(anchor2)) * kRowLines);
                  if (f == flag) todo &= ~anchor2;
                  else seen = f;
                }
                if (todo & anchor) {
                  const u64 f = ld_flag_acquire(line + 8 + (31 - __clz(anchor)) * kRowLines);
                  if (f == flag) todo &= ~anchor;
                  else seen = f;
                }
              }
              if (todo && (++it & 7u) == 0 && !clk.tick(w, XP_WAIT_LL_FLAG, seen, flag)) {
                ok = 0;
                break;
              }
            }
          }
          __syncwarp();
          if (__any_sync(0xffffffffu, !ok)) {
            failed = 1;
            break;
          }
          u64 a[kBatch], b[kBatch];
          unsigned long long* d = reinterpret_cast<unsigned long long*>(sdst + i0 * kDataWords + 2 * pos);
          if (whole) {
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
              a[q] = b[q] = 0;
              if (i0 + q * P < nl) {
                if (flag_lane) a[q] = ld_word(line + q * kRowLines);
                else ll_load(line + q * kRowLines, a[q], b[q]);
              }
            }
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
              if (i0 + q * P < nl) {
                __stcs(d + q * P * kDataWords, a[q]);
                if (!flag_lane) __stcs(d + q * P * kDataWords + 1, b[q]);
              }
            }
            continue;
          }
#pragma unroll
          for (int q = 0; q < kBatch; ++q) {
            const u64 i = i0 + q * P;
            a[q] = b[q] = 0;
            if (i < nl) {
              if (flag_lane) a[q] = ld_word(line + q * kRowLines);
              else ll_load(line + q * kRowLines, a[q], b[q]);
            }
          }
#pragma unroll
          for (int q = 0; q < kBatch; ++q) {
            const u64 i = i0 + q * P;
            const u64 wd = i * kDataWords + 2 * pos;
            if (i < nl) {
              if (wd < left) __stcs(d + q * P * kDataWords, a[q]);
              if (!flag_lane && wd + 1 < left) __stcs(d + q * P * kDataWords + 1, b[q]);
            }
          }
        }
        failed = __any_sync(0xffffffffu, failed);
        // the lines are read (their values are in registers): the slot may
        // be refilled, so the signal needs no ordering
        if (!failed && lane == 0) mbar_arrive_cluster_relaxed(bar0 + 8u * (uint32_t)(step % N));
      }
    }
  } else if (run && warp == kL128Warps && lane == 0 && sender) {
    // producer: stage chunk j of the lane's payload in stage j % kStages once
    // the copy warps have released that stage's previous chunk.  Reading src
    // needs no slot credit, so it runs up to kStages chunks ahead.
    const uint32_t sm0 = smem_addr(stage_mem);
    const u64 pol = policy_evict_first();
    u64 j = 0;
    bool ok = true;
    for (u64 s = 0; s < nsteps && ok; ++s) {
      const u64 left = nwords - s * W;
      const u64 nla = left >= W ? L : (left + kDataWords - 1) / kDataWords;
      const u64 nl = nla < l1 ? nla : l1;
      const u64 sbyte = lo + 8 * s * W;
      for (u64 c0 = l0; c0 < nl; c0 += kChunkLines, ++j) {
        const int k = (int)(j % kStages);
        if (j >= kStages && !mbar_wait_cta(smem_addr(&empty[k]), (uint32_t)(((j / kStages) - 1) & 1), w)) {
          ok = false;
          break;
        }
        const u64 c1 = c0 + kChunkLines < nl ? c0 + kChunkLines : nl;
        const u64 wend = kDataWords * c1 < left ? kDataWords * c1 : left;
        const u64 a0 = (sbyte + 8 * kDataWords * c0) & ~15ull;
        const u64 a1 = staged_end(sbyte + 8 * kDataWords * c0, sbyte + 8 * wend, hi);
        const uint32_t nb = a1 > a0 ? (uint32_t)(a1 - a0) : 0u;
        mbar_arrive_expect_tx(smem_addr(&full[k]), nb);
        if (nb) bulk_load(sm0 + k * kStageBytes, p.src + a0, nb, smem_addr(&full[k]), pol);
      }
    }
  } else if (run && warp == kL128Warps + 1 && sender) {
    // flagger: once every copy warp has stored a chunk's payload, one fence
    // per lane orders it before the chunk's flags, which the warp stores
    u64 j = 0;
    bool ok = true;
    for (u64 s = 0; s < nsteps && ok; ++s) {
      const u64 step = base + s;
      const u64 left = nwords - s * W;
      const u64 nla = left >= W ? L : (left + kDataWords - 1) / kDataWords;
      const u64 nl = nla < l1 ? nla : l1;
      const u64 flag = step + 1;
      char* slot = slots + (step % N) * p.slot_bytes;
      for (u64 c0 = l0; c0 < nl; c0 += kChunkLines, ++j) {
        const int k = (int)(j % kStages);
        if (!mbar_wait_cta(smem_addr(&pdone[k]), (uint32_t)((j / kStages) & 1), w)) {
          ok = false;
          break;
        }
        fence_gpu();
        const u64 c1 = c0 + kChunkLines < nl ? c0 + kChunkLines : nl;
        for (u64 i = c0 + lane; i < c1; i += 32) st_flag(slot + i * kLineBytes + 8 * kDataWords, flag);
        __syncwarp();
        if (lane == 0) mbar_arrive_local_relaxed(smem_addr(&empty[k]));
      }
    }
  } else if (run && warp == kL128Warps && lane == 0 && !sender) {
    u64 r = 0;
    for (; r < nsteps; ++r) {
      const u64 step = base + r;
      if (!mbar_wait(smem_addr(&bars[step % N]), (uint32_t)((r / N) & 1), w, XP_WAIT_SLOT_BARRIER, step)) break;
      st_release(head, step + 1);
    }
    if (r == nsteps) {
      // every lane has read the step base at its start; the last one to
      // finish moves it on and leaves every lane's head there
      const u64 done = atom_add_acq_rel(arr, 1);
      if (done + 1 == GR) {
        const u64 nb = base + nsteps;
        st_relaxed(reinterpret_cast<u64*>(ctl + kHeadOff), nb);
        for (int h = 1; h < kMaxLL128Lanes; ++h) st_relaxed(arr + 16 * h, nb);
        st_relaxed(basew, nb);
        st_relaxed(arr, 0);
        if (cs) cs->t_end = globaltimer();
      }
    }
  }
}

void* ll128_kernel_ptr() { return reinterpret_cast<void*>(&ll128_kernel); }
int ll128_smem() { return kStages * (int)kStageBytes; }
int ll128_threads() { return kL128Threads; }

}  // namespace xp
