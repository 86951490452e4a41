// Host pump of the proxy (copy-engine) mode ("NCCL transport data transfer
// (二)": p2pTransport cudaMemcopy mode, shmTransport useMemcpy mode).
//
// The sender kernel fills ring 0 (its own send ring) and publishes tail[0] in
// mapped host memory.  For every channel this thread watches tail[0], copies
// newly available slot-steps from ring h to ring h + 1 for every hop h with
// cudaMemcpyAsync on a stream of each hop's own (hop h + 1's copy waits on the
// device for hop h's copy of the same steps), and publishes tail[h + 1] =
// step + 1 once hop h's copy has completed.  Consecutive available steps that do not wrap around the ring
// go in one copy (a run of full slots, possibly ending with a short one), so
// every ring receives exactly the bytes of one copy per step, with far fewer
// host calls.  (Measured on the 1 GiB, 16-channel workload: one copy per
// step 122 GB/s, runs of up to N steps 511 GB/s; capping runs at N/2, N/4 or
// N/8 steps was slower, 355, 219 and 117 GB/s: host calls, not overlap,
// bound this mode.  Through a host-placed FIFO (two hops) runs of 1, 2, 4 or
// N steps all gave 92-107 GB/s.)  The receiver kernel drains the last ring.  The pump never
// decides credit: the sender only fills step s once head >= s + 1 - N, which
// already implies that every ring's slot s mod N has been read out.
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
#include <mutex>
#include <set>
#include <string>
#include <thread>
#include <vector>

#include "xp_proxy.h"

namespace xp {

namespace {

using Clock = std::chrono::steady_clock;

uint64_t load_acquire(const char* p) {
  return __atomic_load_n(reinterpret_cast<const uint64_t*>(p), __ATOMIC_ACQUIRE);
}
void store_release(char* p, uint64_t v) { __atomic_store_n(reinterpret_cast<uint64_t*>(p), v, __ATOMIC_RELEASE); }

}  // namespace

struct Pump {
  PumpConfig cfg;
  std::thread th;
  std::atomic<bool> stop{false};
  std::atomic<int64_t> active_until{0};   // steady-clock ns: spin at least until then
  std::atomic<bool> failed{false};
  std::string error;                      // written once before `failed` is set
  std::vector<cudaStream_t> streams;      // [c * hops + h]
  std::vector<cudaEvent_t> events;        // [(c * hops + h) * N + batch % N]
  std::vector<uint64_t> issued, done;     // [c * hops + h], absolute steps
  std::vector<uint64_t> nb_issued, nb_done;   // [c * hops + h], copies (batches)
  std::vector<uint64_t> batch_end;        // [(c * hops + h) * N + batch % N]: first step after the batch

  char* ctl(int c) const { return cfg.ce_host + (size_t)c * kCeCtlBytes; }
  char* slot(int h, int c, uint64_t step) const {
    return cfg.rings[h] + (size_t)c * cfg.ch_stride + (size_t)(step % (uint64_t)cfg.nslots) * cfg.slot_bytes;
  }

  void fail(const std::string& msg) {
    if (failed.load()) return;
    error = msg;
    failed.store(true, std::memory_order_release);
  }

  // one pass over every channel; true if anything moved
  bool poll() {
    bool moved = false;
    const int H = cfg.hops;
    const uint64_t N = (uint64_t)cfg.nslots;
    for (int c = 0; c < cfg.nchannels && !failed.load(std::memory_order_relaxed); ++c) {
      const int q0 = c * H;
      const uint64_t avail = load_acquire(ctl(c) + kCeTailOff);
      // a batch is issued to every hop at once; hop h waits for hop h - 1's
      // copy of the same batch on the device, so the host reacts only to
      // completions.  At most N steps are in flight from tail[0] to the last
      // hop's completion.
      while (issued[q0] < avail && issued[q0] - done[q0 + H - 1] < N) {
        const uint64_t first = issued[q0];
        uint64_t lim = avail < done[q0 + H - 1] + N ? avail : done[q0 + H - 1] + N;
        if (lim > first + (N - first % N)) lim = first + (N - first % N);   // no wrap within one copy
        uint64_t end = first;
        size_t bytes = 0;
        while (end < lim) {
          const int64_t sz = (int64_t)__atomic_load_n(
              reinterpret_cast<const uint64_t*>(ctl(c) + kCeSizeOff) + end % N, __ATOMIC_RELAXED);
          if (sz < 1 || (uint64_t)sz > cfg.slot_bytes) {
            fail("proxy: channel " + std::to_string(c) + " step " + std::to_string(end) + " has size word " +
                 std::to_string(sz));
            return moved;
          }
          bytes += (size_t)sz;
          ++end;
          if ((uint64_t)sz != cfg.slot_bytes) break;   // a short step ends the run
        }
        for (int h = 0; h < H; ++h) {
          const int q = q0 + h;
          const size_t b = (size_t)q * N + nb_issued[q] % N;
          cudaError_t e = cudaSuccess;
          if (h > 0) e = cudaStreamWaitEvent(streams[q], events[(size_t)(q - 1) * N + (nb_issued[q - 1] - 1) % N], 0);
          if (e == cudaSuccess)
            e = cudaMemcpyAsync(slot(h + 1, c, first), slot(h, c, first), bytes, cudaMemcpyDefault, streams[q]);
          if (e == cudaSuccess) e = cudaEventRecord(events[b], streams[q]);
          if (e != cudaSuccess) {
            fail(std::string("proxy: cudaMemcpyAsync: ") + cudaGetErrorString(e));
            return moved;
          }
          batch_end[b] = end;
          ++nb_issued[q];
          issued[q] = end;
        }
        moved = true;
      }
      for (int h = 0; h < H; ++h) {
        const int q = q0 + h;
        while (nb_done[q] < nb_issued[q]) {
          const size_t b = (size_t)q * N + nb_done[q] % N;
          const cudaError_t e = cudaEventQuery(events[b]);
          if (e == cudaErrorNotReady) break;
          if (e != cudaSuccess) {
            fail(std::string("proxy: copy failed: ") + cudaGetErrorString(e));
            return moved;
          }
          ++nb_done[q];
          done[q] = batch_end[b];
          store_release(ctl(c) + kCeTailOff + 128 * (h + 1), done[q]);
          moved = true;
        }
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
  const int Q = cfg.nchannels * cfg.hops;
  p->streams.assign(Q, nullptr);
  p->events.assign((size_t)Q * cfg.nslots, nullptr);
  p->issued.assign(Q, 0);
  p->done.assign(Q, 0);
  p->nb_issued.assign(Q, 0);
  p->nb_done.assign(Q, 0);
  p->batch_end.assign((size_t)Q * cfg.nslots, 0);
  // counters continue from what the control blocks hold (zero after create or reset)
  for (int c = 0; c < cfg.nchannels; ++c)
    for (int h = 0; h < cfg.hops; ++h)
      p->issued[c * cfg.hops + h] = p->done[c * cfg.hops + h] =
          load_acquire(p->ctl(c) + kCeTailOff + 128 * (h + 1));
  cudaError_t e = cudaSuccess;
  for (int q = 0; q < Q && e == cudaSuccess; ++q) e = cudaStreamCreateWithFlags(&p->streams[q], cudaStreamNonBlocking);
  for (size_t i = 0; i < p->events.size() && e == cudaSuccess; ++i)
    e = cudaEventCreateWithFlags(&p->events[i], cudaEventDisableTiming);
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
  for (cudaEvent_t ev : p->events)
    if (ev) cudaEventDestroy(ev);
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
