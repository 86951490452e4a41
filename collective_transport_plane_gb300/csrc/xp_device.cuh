// Device primitives of the FIFO data plane: ordered counter access, bounded
// waits, cluster mbarriers and warp-wide copies.  sm_103a only.
#pragma once

#include <cstdint>

#include "xp_internal.h"

namespace xp {

typedef unsigned long long u64;

// ---- ordered accesses on the control words (.gpu scope: every endpoint is
// ---- a thread of this GPU, also when the word lives in mapped host memory)
__device__ __forceinline__ u64 ld_acquire(const u64* p) {
  u64 v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ u64 ld_relaxed(const u64* p) {
  u64 v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(u64* p, u64 v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed(u64* p, u64 v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// Drop the 128-byte line at p (128-byte aligned) from L2 without writing it
// back; its contents become undefined.
__device__ __forceinline__ void discard_l2(void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}
__device__ __forceinline__ void red_add_release(u64* p, u64 v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void red_add_relaxed(u64* p, u64 v) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// .sys scope: words shared with a host thread (the proxy mode's pump)
__device__ __forceinline__ u64 ld_acquire_sys(const u64* p) {
  u64 v;
  asm volatile("ld.acquire.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ u64 ld_relaxed_sys(const u64* p) {
  u64 v;
  asm volatile("ld.relaxed.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_sys(u64* p, u64 v) {
  asm volatile("st.release.sys.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_sys(u64* p, u64 v) {
  asm volatile("st.relaxed.sys.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ u64 globaltimer() {
  u64 t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- LL line: two 8-byte halves {data, flag}, each a single-copy-atomic u64
__device__ __forceinline__ void ll_store(void* p, u64 a, u64 b) {
  asm volatile("st.volatile.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ void ll_load(const void* p, u64& a, u64& b) {
  asm volatile("ld.volatile.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

// ---- cluster and mbarrier helpers
__device__ __forceinline__ unsigned cluster_ctarank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_init(uint32_t saddr, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Arrive (release, cluster scope) on an mbarrier in any CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_saddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_saddr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t saddr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(saddr), "r"(parity)
      : "memory");
  return ok != 0;
}

// ---- error reporting and bounded waits
struct WaitCtx {
  DevStatus* st;
  const volatile int* abort_word;
  u64 timeout_ns;
  int channel;
  u64 op;
};

// The first failure of operation w.op claims the status block (a claim of
// an earlier operation is replaced) and records where it happened.
__device__ __forceinline__ void report(const WaitCtx& w, int code, int where, u64 observed, u64 expected) {
  const u64 mine = (w.op << 32) | (u64)(uint32_t)code;
  u64 old = *reinterpret_cast<volatile u64*>(&w.st->claim);
  for (;;) {
    if ((old >> 32) == (w.op & 0xffffffffull) && (uint32_t)old != 0) break;   // already claimed
    const u64 seen = atomicCAS(&w.st->claim, old, mine);
    if (seen == old) {
      w.st->channel = w.channel;
      w.st->where = where;
      w.st->observed = observed;
      w.st->expected = expected;
      break;
    }
    old = seen;
  }
  atomicExch(&w.st->sticky, 1);
  atomicExch(&w.st->abort, 1);
}

// At the start of an operation: the first CTA records the operation id, and
// an object with a sticky failure refuses the operation (true).  One thread
// per CTA.
__device__ __forceinline__ bool op_begin(const WaitCtx& w) {
  if (blockIdx.x == 0) *reinterpret_cast<volatile u64*>(&w.st->last_op) = w.op;
  if (*reinterpret_cast<volatile int*>(&w.st->sticky)) {
    report(w, XP_ERR_ABORTED, XP_WAIT_STICKY, 0, 0);
    return true;
  }
  return false;
}

// Largest occupancy seen in operation `op` (the tag keeps older ones out).
__device__ __forceinline__ void note_occupancy(DevStatus* st, u64 op, unsigned occ) {
  atomicMax(&st->occupancy, (op << 32) | occ);
}

__device__ __forceinline__ bool op_aborted_device(const WaitCtx& w) {
  return *reinterpret_cast<volatile int*>(&w.st->abort) != 0;
}
__device__ __forceinline__ bool op_aborted(const WaitCtx& w) {
  if (op_aborted_device(w)) return true;
  if (w.abort_word && *w.abort_word) {
    report(w, XP_ERR_ABORTED, XP_WAIT_NONE, 0, 0);
    return true;
  }
  return false;
}

// Clock of one bounded wait.  The first kQuietNs of a wait only spin; after
// that the operation's abort flag (device memory) is checked every
// kCheckNs, the host abort word (mapped host memory, a slow read) every
// kHostCheckNs, and the wait gives up after timeout_ns.
constexpr u64 kQuietNs = 20000;
constexpr u64 kCheckNs = 20000;
constexpr u64 kHostCheckNs = 200000;

struct WaitClock {
  u64 start = 0, next = 0, next_host = 0;
  // false: stop waiting (the reason is already reported)
  __device__ __forceinline__ bool tick(const WaitCtx& w, int where, u64 observed, u64 expected) {
    const u64 now = globaltimer();
    if (start == 0) {
      start = now;
      next = now + kQuietNs;
      next_host = now + kHostCheckNs;
      return true;
    }
    if (now < next) return true;
    next = now + kCheckNs;
    if (op_aborted_device(w)) return false;
    if (now >= next_host) {
      next_host = now + kHostCheckNs;
      if (w.abort_word && *w.abort_word) {
        report(w, XP_ERR_ABORTED, XP_WAIT_NONE, 0, 0);
        return false;
      }
    }
    if (now - start > w.timeout_ns) {
      report(w, XP_ERR_TIMEOUT, where, observed, expected);
      return false;
    }
    return true;
  }
};

// Poll `*p` (acquire) until it is >= target.  One thread.  Gives up on the
// operation's abort flag, the host abort word, or after timeout_ns.
static __device__ __noinline__ bool wait_geq(const u64* p, u64 target, u64& cache, const WaitCtx& w, int where) {
  if (cache >= target) return true;
  WaitClock clk;
  unsigned it = 0;
  for (;;) {
    u64 v = ld_acquire(p);
    if (v >= target) {
      cache = v;
      return true;
    }
    if ((++it & 7u) == 0 && !clk.tick(w, where, v, target)) return false;
  }
}

// Same for a word that must become zero (mode 0) or non-zero (mode 1).
static __device__ __noinline__ bool wait_word(const u64* p, int nonzero, u64& value, const WaitCtx& w, int where) {
  WaitClock clk;
  unsigned it = 0;
  for (;;) {
    u64 v = ld_acquire(p);
    if ((v != 0) == (nonzero != 0)) {
      value = v;
      return true;
    }
    if ((++it & 7u) == 0 && !clk.tick(w, where, v, nonzero ? 1 : 0)) return false;
  }
}

// Warp-wide wait: lane 0 polls with acquire, __syncwarp orders the other
// lanes' later accesses after it.
__device__ __forceinline__ bool warp_wait_geq(const u64* p, u64 target, u64& cache, const WaitCtx& w, int where) {
  if (cache >= target) return true;   // warp-uniform: every lane holds the same cache
  const int lane = threadIdx.x & 31;
  int ok = 1;
  u64 c = cache;
  if (lane == 0) ok = wait_geq(p, target, c, w, where);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  cache = __shfl_sync(0xffffffffu, c, 0);
  __syncwarp();
  return ok != 0;
}

static __device__ __noinline__ bool mbar_wait(uint32_t saddr, uint32_t parity, const WaitCtx& w, int where, u64 step) {
  WaitClock clk;
  while (!mbar_try_wait(saddr, parity)) {
    if (!clk.tick(w, where, step, step + 1)) return false;
  }
  return true;
}

// ---- copies: one warp moves [0, nbytes) with 16-byte vectors (src, dst
// ---- 16-byte aligned; a ragged tail of < 16 bytes is moved bytewise)
enum { LD_STREAM = 0, LD_L2 = 1 };
enum { ST_STREAM = 0, ST_L2 = 1 };

template <int LD>
__device__ __forceinline__ uint4 vload(const uint4* p) {
  if (LD == LD_STREAM) return __ldcs(p);
  return __ldcg(p);
}
template <int ST>
__device__ __forceinline__ void vstore(uint4* p, uint4 v) {
  if (ST == ST_STREAM)
    __stcs(p, v);
  else
    __stcg(p, v);
}

template <int LD, int ST>
__device__ __forceinline__ void warp_copy(const char* src, char* dst, u64 nbytes) {
  const int lane = threadIdx.x & 31;
  const u64 nvec = nbytes >> 4;
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
  u64 i = lane;
  for (; i + 96 < nvec; i += 128) {
    uint4 a = vload<LD>(s + i);
    uint4 b = vload<LD>(s + i + 32);
    uint4 c = vload<LD>(s + i + 64);
    uint4 e = vload<LD>(s + i + 96);
    vstore<ST>(d + i, a);
    vstore<ST>(d + i + 32, b);
    vstore<ST>(d + i + 64, c);
    vstore<ST>(d + i + 96, e);
  }
  for (; i < nvec; i += 32) vstore<ST>(d + i, vload<LD>(s + i));
  const u64 done = nvec << 4;
  if (done + lane < nbytes) dst[done + lane] = __ldcg(src + done + lane);
}

// Balanced split of `nbytes` (16-byte vectors, the last possibly short) into
// `parts` contiguous pieces; returns piece `i` as [*b0, *b1).
__device__ __forceinline__ void piece(u64 nbytes, u64 parts, u64 i, u64* b0, u64* b1) {
  const u64 nvec = (nbytes + 15) >> 4;
  const u64 v0 = (nvec * i) / parts;
  const u64 v1 = (nvec * (i + 1)) / parts;
  *b0 = v0 << 4;
  *b1 = (v1 << 4) < nbytes ? (v1 << 4) : nbytes;
  if (*b0 > *b1) *b0 = *b1;
}

// Channel c's byte range [lo, hi): q = round_up(ceil(n / C), 16).
__device__ __forceinline__ void channel_range(u64 n, int C, int c, u64* lo, u64* hi) {
  u64 q = (n + C - 1) / C;
  q = (q + 15) & ~15ull;
  u64 a = q * c, b = q * (c + 1);
  *lo = a < n ? a : n;
  *hi = b < n ? b : n;
}

}  // namespace xp

namespace xp {

// ---- bulk (TMA) copies between global and shared memory, 16-byte granular
__device__ __forceinline__ void mbar_arrive_local(uint32_t saddr) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr) : "memory");
}
// Arm a stage barrier for `bytes` of bulk-copy data.  Relaxed: the thread
// that arms it is the one that waits on it, so it orders nothing else.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t saddr, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cta.shared::cta.b64 _, [%0], %1;" ::"r"(saddr), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_local_relaxed(uint32_t saddr) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(saddr) : "memory");
}
// Relaxed arrive on an mbarrier anywhere in the cluster: for signals that
// carry no memory ordering (the reads they report have already completed).
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_saddr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_saddr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cta(uint32_t saddr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(saddr), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on a CTA-local mbarrier phase.
static __device__ __noinline__ bool mbar_wait_cta(uint32_t saddr, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait_cta(saddr, parity)) return true;
  WaitClock clk;
  while (!mbar_try_wait_cta(saddr, parity)) {
    if (!clk.tick(w, XP_WAIT_SLOT_BARRIER, parity, 0)) return false;
  }
  return true;
}
// L2 cache policies for bulk copies: FIFO slots are recycled every N steps and
// should stay in L2 (evict_last); user buffers stream through once (evict_first).
__device__ __forceinline__ u64 policy_evict_last() {
  u64 p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ u64 policy_evict_normal() {
  u64 p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ u64 policy_evict_first() {
  u64 p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void bulk_load(uint32_t sdst, const void* gsrc, uint32_t bytes, uint32_t bar, u64 policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(sdst), "l"(gsrc), "r"(bytes), "r"(bar), "l"(policy) : "memory");
}
__device__ __forceinline__ void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes, u64 policy) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(gdst),
               "r"(ssrc), "r"(bytes), "l"(policy) : "memory");
}
// Ask L2 to fetch [gsrc, gsrc + bytes) (16-byte aligned, a multiple of 16
// bytes); no completion is tracked.
__device__ __forceinline__ void bulk_prefetch_l2(const void* gsrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gsrc), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// A counter mirrored in shared memory by a watcher thread of the same CTA.
__device__ __forceinline__ u64 ld_acquire_cta_shared(const u64* p) {
  u64 v;
  asm volatile("ld.acquire.cta.shared::cta.u64 %0, [%1];" : "=l"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_cta_shared(u64* p, u64 v) {
  asm volatile("st.release.cta.shared::cta.u64 [%0], %1;" ::"r"(smem_addr(p)), "l"(v) : "memory");
}
// Wait until the mirrored counter is >= target (one thread).
static __device__ __noinline__ bool wait_mirror(const u64* m, u64 target, u64& cache, const WaitCtx& w, int where) {
  if (cache >= target) return true;
  WaitClock clk;
  for (;;) {
    const u64 v = ld_acquire_cta_shared(m);
    if (v >= target) {
      cache = v;
      return true;
    }
    if (!clk.tick(w, where, v, target)) return false;
  }
}

// Everything this thread has done or observed in memory is performed at GPU
// scope before anything it does next.
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// Order this thread's async-proxy (bulk copy) accesses of global memory with
// its generic-proxy accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

}  // namespace xp
