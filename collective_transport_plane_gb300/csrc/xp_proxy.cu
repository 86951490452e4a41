// Host pump of the proxy (copy-engine) mode ("NCCL transport data transfer
// (二)": p2pTransport cudaMemcopy mode, shmTransport useMemcpy mode).
//
// The sender kernel fills ring 0 (its own send ring) and publishes tail[0] in
// mapped host memory.  This thread watches every channel's tail[0], copies
// newly available slot-steps from ring h to ring h + 1 for every hop h with
// the copy engines' calls (hop h + 1's copy waits on the device for hop h's
// copy of the same steps), and publishes tail[h + 1] = step + 1 once hop h's
// copy has completed.  The receiver kernel drains the last ring.  The pump
// never decides credit: the sender only fills step s once head >= s + 1 - N,
// which already implies that every ring's slot s mod N has been read out.
//
// Host calls bound this mode, so each call moves as much as it can:
// consecutive available steps that do not wrap around the ring go in one
// copy (a run of whole slots, possibly ending with a short one, so every
// ring receives exactly the bytes of one copy per step), and runs of whole
// slots that start at the same step on consecutive channels of a group of
// kPumpGroup channels go in one 2D copy whose rows are the channels (row
// pitch = the rings' channel stride).  Each group has its own stream per
// hop, so the groups' copies run side by side and a channel's copies
// complete in order.  Measured on the 1 GiB, 16-channel workload (device
// FIFO, 4 lanes): one copy per step 122 GB/s; runs per channel, a stream per
// channel 511; 2D copies over groups of 1, 2, 4, 8, 16 channels 475, 654,
// 700-717, 449, 211 GB/s (fewer streams run fewer copies at once).
// Through a host-placed FIFO (two hops) every variant gave 100-111 GB/s.
//
// The pump runs from xp_fifo_enable_ce until the FIFO is destroyed or reset.
// It spins while steps move (and for a while after a kick), then sleeps 50 us
// between polls.  It never blocks on the device: copies are asynchronous and
// completion is polled with cudaEventQuery.  A size word outside [1, S] or a
// CUDA error stops it; the kernel then times out and the error message is
// kept for xp_fifo_status.
#include <cuda_runtime.h>

#include <atomic>
#include <chrono>
#include <cstring>
#include <deque>
#include <mutex>
#include <set>
#include <string>
#include <thread>
#include <vector>

#include "xp_proxy.h"

namespace xp {

namespace {

using Clock = std::chrono::steady_clock;

constexpr int kPumpGroup = 4;   // channels that share a stream and may share a 2D copy

uint64_t load_acquire(const char* p) {
  return __atomic_load_n(reinterpret_cast<const uint64_t*>(p), __ATOMIC_ACQUIRE);
}
void store_release(char* p, uint64_t v) { __atomic_store_n(reinterpret_cast<uint64_t*>(p), v, __ATOMIC_RELEASE); }

}  // namespace

struct Pump {
  // One copy of the same slot-steps [first, end) for the consecutive channels
  // [c0, c1) of one hop: a 2D copy whose rows are the channels (row pitch =
  // the channel stride of the rings), or a plain copy for one channel.
  struct Batch {
    cudaEvent_t ev;
    int c0, c1;
    uint64_t end;
  };

  PumpConfig cfg;
  std::thread th;
  std::atomic<bool> stop{false};
  std::atomic<int64_t> active_until{0};   // steady-clock ns: spin at least until then
  std::atomic<bool> failed{false};
  std::string error;                      // written once before `failed` is set
  int G = 1;                              // channels per group
  std::vector<cudaStream_t> streams;      // [g * hops + h]: the copies of hop h for group g, in order
  std::vector<cudaEvent_t> pool;          // free events
  std::vector<std::deque<Batch>> queue;   // [g * hops + h]: copies in flight, oldest first
  std::vector<uint64_t> issued;           // [c]: first step not yet handed to the copies
  std::vector<uint64_t> done;             // [c * hops + h]: steps hop h has completed
  std::vector<uint64_t> avail;            // [c]: tail[0] as last read

  char* ctl(int c) const { return cfg.ce_host + (size_t)c * kCeCtlBytes; }
  char* slot(int h, int c, uint64_t step) const {
    return cfg.rings[h] + (size_t)c * cfg.ch_stride + (size_t)(step % (uint64_t)cfg.nslots) * cfg.slot_bytes;
  }

  void fail(const std::string& msg) {
    if (failed.load()) return;
    error = msg;
    failed.store(true, std::memory_order_release);
  }

  // The next run of channel c: steps [first, end) that tail[0] has made
  // available, that fit in the N steps allowed in flight (from tail[0] to the
  // last hop's completion), and that do not wrap around the ring; a short
  // step ends it.  Returns false (and fails the pump) on a bad size word.
  bool run_of(int c, uint64_t* end, size_t* bytes, bool* full) {
    const uint64_t N = (uint64_t)cfg.nslots;
    const uint64_t first = issued[c];
    const uint64_t dl = done[(size_t)c * cfg.hops + cfg.hops - 1];
    uint64_t lim = avail[c] < dl + N ? avail[c] : dl + N;
    if (lim > first + (N - first % N)) lim = first + (N - first % N);
    uint64_t e = first;
    size_t b = 0;
    *full = true;
    while (e < lim) {
      const int64_t sz = (int64_t)__atomic_load_n(
          reinterpret_cast<const uint64_t*>(ctl(c) + kCeSizeOff) + e % N, __ATOMIC_RELAXED);
      if (sz < 1 || (uint64_t)sz > cfg.slot_bytes) {
        fail("proxy: channel " + std::to_string(c) + " step " + std::to_string(e) + " has size word " +
             std::to_string(sz));
        return false;
      }
      b += (size_t)sz;
      ++e;
      if ((uint64_t)sz != cfg.slot_bytes) {
        *full = false;
        break;
      }
    }
    *end = e;
    *bytes = b;
    return true;
  }

  // Copy steps [first, end) of channels [c0, c1) through every hop: hop h's
  // copy waits on the device for hop h - 1's copy of the same steps.
  bool issue(int c0, int c1, uint64_t first, uint64_t end, size_t bytes) {
    const int H = cfg.hops;
    for (int h = 0; h < H; ++h) {
      if (pool.empty()) {
        fail("proxy: no free event");
        return false;
      }
      cudaEvent_t ev = pool.back();
      cudaError_t e = cudaSuccess;
      const int q = (c0 / G) * H + h;
      if (h > 0) e = cudaStreamWaitEvent(streams[q], queue[q - 1].back().ev, 0);
      if (e == cudaSuccess) {
        if (c1 - c0 == 1)
          e = cudaMemcpyAsync(slot(h + 1, c0, first), slot(h, c0, first), bytes, cudaMemcpyDefault, streams[q]);
        else
          e = cudaMemcpy2DAsync(slot(h + 1, c0, first), cfg.ch_stride, slot(h, c0, first), cfg.ch_stride, bytes,
                                (size_t)(c1 - c0), cudaMemcpyDefault, streams[q]);
      }
      if (e == cudaSuccess) e = cudaEventRecord(ev, streams[q]);
      if (e != cudaSuccess) {
        fail(std::string("proxy: cudaMemcpyAsync: ") + cudaGetErrorString(e));
        return false;
      }
      pool.pop_back();
      queue[q].push_back(Batch{ev, c0, c1, end});
    }
    for (int c = c0; c < c1; ++c) issued[c] = end;
    return true;
  }

  // one pass over every channel; true if anything moved
  bool poll() {
    bool moved = false;
    const int C = cfg.nchannels;
    const int H = cfg.hops;
    for (int c = 0; c < C; ++c) avail[c] = load_acquire(ctl(c) + kCeTailOff);
    // Runs of whole slots that start at the same step on consecutive
    // channels go in one 2D copy per hop, up to the shortest of them; a run
    // that ends with a short step goes alone.
    for (int c = 0; c < C && !failed.load(std::memory_order_relaxed);) {
      uint64_t end;
      size_t bytes;
      bool full;
      if (!run_of(c, &end, &bytes, &full)) return moved;
      const uint64_t first = issued[c];
      if (end == first) {
        ++c;
        continue;
      }
      int c1 = c + 1;
      if (full) {
        while (c1 < C && c1 % G != 0 && issued[c1] == first) {
          uint64_t e1;
          size_t b1;
          bool f1;
          if (!run_of(c1, &e1, &b1, &f1)) return moved;
          if (!f1 || e1 == first) break;
          if (e1 < end) end = e1;
          ++c1;
        }
        bytes = (size_t)(end - first) * cfg.slot_bytes;
      }
      if (!issue(c, c1, first, end, bytes)) return moved;
      moved = true;
      c = c1;
    }
    for (int q = 0; q < (int)queue.size() && !failed.load(std::memory_order_relaxed); ++q) {
      const int h = q % H;
      while (!queue[q].empty()) {
        const Batch& b = queue[q].front();
        const cudaError_t e = cudaEventQuery(b.ev);
        if (e == cudaErrorNotReady) break;
        if (e != cudaSuccess) {
          fail(std::string("proxy: copy failed: ") + cudaGetErrorString(e));
          return moved;
        }
        for (int c = b.c0; c < b.c1; ++c) {
          done[(size_t)c * H + h] = b.end;
          store_release(ctl(c) + kCeTailOff + 128 * (h + 1), b.end);
        }
        pool.push_back(b.ev);
        queue[q].pop_front();
        moved = true;
      }
    }
    return moved;
  }

  void run() {
    cudaSetDevice(cfg.device);
    // other threads' global-mode stream captures must not forbid these calls
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaThreadExchangeStreamCaptureMode(&mode);
    auto last = Clock::now();
    while (!stop.load(std::memory_order_acquire)) {
      if (!failed.load(std::memory_order_relaxed) && poll()) {
        last = Clock::now();
        continue;
      }
      const auto now = Clock::now();
      const int64_t ns = std::chrono::duration_cast<std::chrono::nanoseconds>(now.time_since_epoch()).count();
      if (now - last < std::chrono::milliseconds(2) || ns < active_until.load(std::memory_order_relaxed))
        std::this_thread::yield();
      else
        std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
    // nothing may still read the rings once the owner frees them
    for (cudaStream_t s : streams) cudaStreamSynchronize(s);
  }
};

namespace {
// Pumps still running at unload (FIFOs never destroyed) are stopped and
// joined before the library goes away.
std::mutex g_live_mu;
std::set<Pump*> g_live;
struct Reaper {
  ~Reaper() {
    std::lock_guard<std::mutex> lk(g_live_mu);
    for (Pump* p : g_live) {
      p->stop.store(true, std::memory_order_release);
      if (p->th.joinable()) p->th.join();
    }
    g_live.clear();
  }
} g_reaper;
}  // namespace

Pump* pump_start(const PumpConfig& cfg, std::string* err) {
  Pump* p = new Pump();
  p->cfg = cfg;
  const int C = cfg.nchannels, H = cfg.hops;
  p->G = kPumpGroup;
  const int ngroups = (C + p->G - 1) / p->G;
  p->streams.assign((size_t)ngroups * H, nullptr);
  p->queue.assign((size_t)ngroups * H, std::deque<Pump::Batch>());
  p->issued.assign(C, 0);
  p->done.assign((size_t)C * H, 0);
  p->avail.assign(C, 0);
  // counters continue from what the control blocks hold (zero after create
  // or reset); every hop has completed what was issued
  for (int c = 0; c < C; ++c) {
    p->issued[c] = load_acquire(p->ctl(c) + kCeTailOff + 128 * H);
    for (int h = 0; h < H; ++h) p->done[(size_t)c * H + h] = load_acquire(p->ctl(c) + kCeTailOff + 128 * (h + 1));
  }
  cudaError_t e = cudaSuccess;
  for (size_t q = 0; q < p->streams.size() && e == cudaSuccess; ++q)
    e = cudaStreamCreateWithFlags(&p->streams[q], cudaStreamNonBlocking);
  // at most N steps of a channel are in flight, each batch holds at least one
  p->pool.assign((size_t)H * C * cfg.nslots, nullptr);
  for (size_t i = 0; i < p->pool.size() && e == cudaSuccess; ++i)
    e = cudaEventCreateWithFlags(&p->pool[i], cudaEventDisableTiming);
  if (e != cudaSuccess) {
    *err = std::string("proxy setup: ") + cudaGetErrorString(e);
    pump_stop(p);
    return nullptr;
  }
  p->th = std::thread([p] { p->run(); });
  std::lock_guard<std::mutex> lk(g_live_mu);
  g_live.insert(p);
  return p;
}

void pump_stop(Pump* p) {
  if (!p) return;
  {
    std::lock_guard<std::mutex> lk(g_live_mu);
    g_live.erase(p);
  }
  p->stop.store(true, std::memory_order_release);
  if (p->th.joinable()) p->th.join();
  for (cudaEvent_t ev : p->pool)
    if (ev) cudaEventDestroy(ev);
  for (auto& q : p->queue)
    for (auto& b : q) cudaEventDestroy(b.ev);
  for (cudaStream_t s : p->streams)
    if (s) cudaStreamDestroy(s);
  delete p;
}

void pump_kick(Pump* p) {
  if (!p) return;
  const int64_t now = std::chrono::duration_cast<std::chrono::nanoseconds>(Clock::now().time_since_epoch()).count();
  p->active_until.store(now + 20000000, std::memory_order_relaxed);   // spin for the next 20 ms
}

const char* pump_error(const Pump* p) {
  if (!p || !p->failed.load(std::memory_order_acquire)) return nullptr;
  return p->error.c_str();
}

}  // namespace xp
