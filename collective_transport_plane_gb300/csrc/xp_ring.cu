// Virtual ring allreduce over P ranks that all live in this GPU's memory.
//
// Ring: rank r receives from r-1 and sends to r+1 ("NCCL transport setup",
// 具体说明).  Each rank owns, per channel, the SIMPLE FIFO its predecessor
// writes into.  One thread-block cluster per channel holds every rank's
// CTAs (P*G of them: G lanes per rank), so the whole ring of a channel is
// co-resident and a rank waiting on its neighbour can never starve it.
//
// Per round of P chunks, rank r runs send(r-1), recvReduceSend(r-1-j) for
// j = 1..P-2, recvReduceCopySend(r), recvCopySend(r-1-j) for j = 0..P-3 and
// recv(r+1), each chunk moved in slot-steps.  A fused step waits for the
// predecessor's tail (if it receives) and for credit on the successor's FIFO
// (if it sends), reads the received slot and/or its own input, adds them
// (fp32: __fadd_rn, no FMA, no flush-to-zero; int32: wrapping), and writes
// the successor's slot and/or its own output in one pass.  Copy warps arrive
// on per-slot mbarriers in the rank's leader CTA; two publisher warps there
// store the successor FIFO's tail and the own FIFO's head.
#include <cuda_runtime.h>

#include "xp_device.cuh"

namespace xp {

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

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
}
__device__ __forceinline__ int4 add4(int4 a, int4 b) {
  return make_int4((int)((unsigned)a.x + (unsigned)b.x), (int)((unsigned)a.y + (unsigned)b.y),
                   (int)((unsigned)a.z + (unsigned)b.z), (int)((unsigned)a.w + (unsigned)b.w));
}
__device__ __forceinline__ float add1(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ int add1(int a, int b) { return (int)((unsigned)a + (unsigned)b); }

template <typename V>
__device__ __forceinline__ V ldcs4(const V* p) { return __ldcs(p); }
template <typename V>
__device__ __forceinline__ V ldcg4(const V* p) { return __ldcg(p); }

// One warp: elementwise step over `nbytes` bytes (multiple of the element
// size).  rs: received slot, in: own input, ss: successor's slot, out: own output.
template <typename T, typename V, int KIND>
__device__ __forceinline__ void warp_ring_op(const char* rs, const char* in, char* ss, char* out, u64 nbytes) {
  const int lane = threadIdx.x & 31;
  const u64 nvec = nbytes >> 4;
  const V* R = reinterpret_cast<const V*>(rs);
  const V* I = reinterpret_cast<const V*>(in);
  V* Sd = reinterpret_cast<V*>(ss);
  V* O = reinterpret_cast<V*>(out);
  u64 i = lane;
  for (; i + 32 < nvec; i += 64) {
    V a0, a1;
    if (KIND == K_SEND) {
      a0 = ldcs4(I + i);
      a1 = ldcs4(I + i + 32);
    } else {
      a0 = ldcg4(R + i);
      a1 = ldcg4(R + i + 32);
      if (KIND == K_RRS || KIND == K_RRCS) {
        a0 = add4(a0, ldcs4(I + i));
        a1 = add4(a1, ldcs4(I + i + 32));
      }
    }
    if (KIND != K_RECV) {
      __stcg(Sd + i, a0);
      __stcg(Sd + i + 32, a1);
    }
    if (KIND == K_RRCS || KIND == K_RCS || KIND == K_RECV) {
      __stcs(O + i, a0);
      __stcs(O + i + 32, a1);
    }
  }
  for (; i < nvec; i += 32) {
    V a0;
    if (KIND == K_SEND) {
      a0 = ldcs4(I + i);
    } else {
      a0 = ldcg4(R + i);
      if (KIND == K_RRS || KIND == K_RRCS) a0 = add4(a0, ldcs4(I + i));
    }
    if (KIND != K_RECV) __stcg(Sd + i, a0);
    if (KIND == K_RRCS || KIND == K_RCS || KIND == K_RECV) __stcs(O + i, a0);
  }
  // ragged tail: fewer than 16 bytes, whole elements
  const u64 done = nvec << 4;
  const u64 e = done / sizeof(T) + lane;
  if (done + (u64)lane * sizeof(T) < nbytes) {
    const T* Rt = reinterpret_cast<const T*>(rs);
    const T* It = reinterpret_cast<const T*>(in);
    T* St = reinterpret_cast<T*>(ss);
    T* Ot = reinterpret_cast<T*>(out);
    T a;
    if (KIND == K_SEND) {
      a = __ldcs(It + e);
    } else {
      a = __ldcg(Rt + e);
      if (KIND == K_RRS || KIND == K_RRCS) a = add1(a, __ldcs(It + e));
    }
    if (KIND != K_RECV) __stcg(St + e, a);
    if (KIND == K_RRCS || KIND == K_RCS || KIND == K_RECV) __stcs(Ot + e, a);
  }
}

template <typename T, typename V>
__device__ __forceinline__ void ring_dispatch(int kind, const char* rs, const char* in, char* ss, char* out,
                                              u64 nbytes) {
  switch (kind) {
    case K_SEND: warp_ring_op<T, V, K_SEND>(rs, in, ss, out, nbytes); break;
    case K_RRS: warp_ring_op<T, V, K_RRS>(rs, in, ss, out, nbytes); break;
    case K_RRCS: warp_ring_op<T, V, K_RRCS>(rs, in, ss, out, nbytes); break;
    case K_RCS: warp_ring_op<T, V, K_RCS>(rs, in, ss, out, nbytes); break;
    default: warp_ring_op<T, V, K_RECV>(rs, in, ss, out, nbytes); break;
  }
}

// Element range of channel c: 16-byte aligned quota q = round_up(ceil(n / C), 16 / esize).
__device__ __forceinline__ void ring_channel(u64 count, u64 align, int C, int c, u64* lo, u64* hi) {
  u64 q = (count + C - 1) / C;
  q = (q + align - 1) / align * align;
  const u64 a = q * c, b = q * (c + 1);
  *lo = a < count ? a : count;
  *hi = b < count ? b : count;
}

// Chunk size of the round starting at `off` in a channel range of `len`
// elements: full chunks of `ce` elements, the last round shrinks them to
// round_up(ceil(m / P), align).
__device__ __forceinline__ u64 round_chunk(u64 len, u64 off, u64 P, u64 ce, u64 align, u64* m_out) {
  u64 m = len - off;
  if (m > P * ce) m = P * ce;
  u64 cs = (m + P - 1) / P;
  cs = (cs + align - 1) / align * align;
  if (cs > ce) cs = ce;
  *m_out = m;
  return cs;
}

template <typename T, typename V>
__global__ void __launch_bounds__(kRingThreads, 1) ring_kernel(const RingParams p) {
  __shared__ __align__(8) u64 bars_send[kMaxSlots];
  __shared__ __align__(8) u64 bars_recv[kMaxSlots];
  __shared__ u64 s_rbase, s_sbase;
  __shared__ int s_stop;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int P = p.nranks;
  const int G = p.lanes;
  const unsigned crank = cluster_ctarank();
  const int c = blockIdx.x / (P * G);
  const int r = (int)crank / G;
  const int g = (int)crank % G;
  const unsigned leader = (unsigned)(r * G);
  const bool leader_cta = crank == leader;
  const u64 N = (u64)p.nslots;
  const u64 S = p.slot_bytes;
  const u64 es = sizeof(T);
  const u64 align = 16 / es;
  const u64 epl = S / es;                         // elements per slot
  const u64 ce = (N / 2) * S / es;                // elements per full chunk

  const int f_recv = c * P + r;
  const int f_send = c * P + (r + 1) % P;
  char* ctl_r = p.ctl + (u64)f_recv * kRingMaxLanes * kCtlBytes;   // lane block 0: one counter set per FIFO
  char* ctl_s = p.ctl + (u64)f_send * kRingMaxLanes * kCtlBytes;
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
  ring_channel(p.count, align, p.nchannels, c, &clo, &chi);
  const u64 clen = chi - clo;
  const WaitCtx w{p.status, p.abort_word, p.timeout_ns, c * P + r, p.op};

  if (threadIdx.x == 0) {
    s_rbase = ld_relaxed(base_recv);
    s_sbase = ld_relaxed(base_send);
    s_stop = op_begin(w) ? 1 : 0;
    if (leader_cta) {
      const uint32_t count = (uint32_t)(G * kCopyWarps);
      for (int k = 0; k < p.nslots; ++k) {
        mbar_init(smem_addr(&bars_send[k]), count);
        mbar_init(smem_addr(&bars_recv[k]), count);
      }
      mbar_init_fence();
    }
  }
  cluster_sync_all();
  const u64 rbase = s_rbase, sbase = s_sbase;
  const bool run = clen > 0 && s_stop == 0;

  if (run && warp < kCopyWarps) {
    const u64 parts = (u64)G * kCopyWarps;
    const u64 my_piece = (u64)g * kCopyWarps + warp;
    const uint32_t bs0 = map_to_rank(smem_addr(&bars_send[0]), leader);
    const uint32_t br0 = map_to_rank(smem_addr(&bars_recv[0]), leader);
    u64 rstep = rbase, sstep = sbase, tcache = 0, hcache = 0;
    bool ok = true;
    for (u64 off = 0; off < clen && ok;) {
      u64 m;
      const u64 cs = round_chunk(clen, off, (u64)P, ce, align, &m);
      for (int pos = 0; pos <= 2 * P - 2 && ok; ++pos) {
        int kind, k;
        ring_op(pos, r, P, &kind, &k);
        u64 klo = (u64)k * cs, khi = (u64)(k + 1) * cs;
        if (klo > m) klo = m;
        if (khi > m) khi = m;
        const u64 base_el = clo + off + klo;     // absolute element index of the chunk
        const u64 klen = khi - klo;
        for (u64 o = 0; o < klen; o += epl) {
          const u64 n = (klen - o) < epl ? (klen - o) : epl;
          if (kind_recv(kind) && !warp_wait_geq(tail_recv, rstep + 1, tcache, w, XP_WAIT_TAIL)) { ok = false; break; }
          if (kind_send(kind) && sstep + 1 > N &&
              !warp_wait_geq(head_send, sstep + 1 - N, hcache, w, XP_WAIT_HEAD)) { ok = false; break; }
          u64 b0, b1;
          piece(n * es, parts, my_piece, &b0, &b1);
          const u64 eoff = (base_el + o) * es + b0;
          ring_dispatch<T, V>(kind, slots_r + (rstep % N) * S + b0, inp + eoff, slots_s + (sstep % N) * S + b0,
                              outp + eoff, b1 - b0);
          __syncwarp();
          if (lane == 0) {
            if (kind_send(kind)) mbar_arrive_cluster(bs0 + 8u * (uint32_t)(sstep % N));
            if (kind_recv(kind)) mbar_arrive_cluster(br0 + 8u * (uint32_t)(rstep % N));
          }
          if (kind_send(kind)) ++sstep;
          if (kind_recv(kind)) ++rstep;
        }
      }
      off += m;
    }
  } else if (run && leader_cta && warp >= kCopyWarps && lane == 0) {
    // publishers: count this rank's send (warp kCopyWarps) or receive
    // (warp kCopyWarps + 1) slot-steps by walking the same schedule
    const bool pub_tail = warp == kCopyWarps;
    u64 total = 0;
    for (u64 off = 0; off < clen;) {
      u64 m;
      const u64 cs = round_chunk(clen, off, (u64)P, ce, align, &m);
      for (int pos = 0; pos <= 2 * P - 2; ++pos) {
        int kind, k;
        ring_op(pos, r, P, &kind, &k);
        u64 klo = (u64)k * cs, khi = (u64)(k + 1) * cs;
        if (klo > m) klo = m;
        if (khi > m) khi = m;
        const bool counts = pub_tail ? kind_send(kind) : kind_recv(kind);
        if (counts) total += (khi - klo + epl - 1) / epl;
      }
      off += m;
    }
    const u64 b = pub_tail ? sbase : rbase;
    u64* word = pub_tail ? tail_send : head_recv;
    u64* bars = pub_tail ? bars_send : bars_recv;
    u64 s = 0;
    unsigned max_occ = 0;
    for (; s < total; ++s) {
      const u64 step = b + s;
      if (!mbar_wait(smem_addr(&bars[step % N]), (uint32_t)((s / N) & 1), w, XP_WAIT_SLOT_BARRIER, step)) break;
      st_release(word, step + 1);
      if (pub_tail) {
        const u64 h = ld_relaxed(head_send);
        const u64 occ = step + 1 - h;
        if (h > step + 1 || occ > N) {
          report(w, XP_ERR_BOUNDS, XP_WAIT_OCCUPANCY, occ, N);
          break;
        }
        if (occ > max_occ) max_occ = (unsigned)occ;
      }
    }
    if (pub_tail) note_occupancy(p.status, p.op, max_occ);
    if (!pub_tail && s == total) st_relaxed(base_recv, rbase + total);
  }
  __syncwarp();
  cluster_sync_all();
}

template __global__ void ring_kernel<float, float4>(const RingParams);
template __global__ void ring_kernel<int, int4>(const RingParams);

void* ring_kernel_ptr(int dtype) {
  if (dtype == XP_F32) return reinterpret_cast<void*>(&ring_kernel<float, float4>);
  if (dtype == XP_I32) return reinterpret_cast<void*>(&ring_kernel<int, int4>);
  return nullptr;
}

}  // namespace xp
