// Host side of the C ABI declared in include/xp.h: argument checks, FIFO
// memory (allocated once at create, as the channel buffers of "RDMA and
// GPUDirect" §7.2), and one cluster launch per operation.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "xp_internal.h"
#include "xp_proxy.h"

namespace xp {
void* p2p_kernel_ptr(bool zero_copy);
void* p2p_tma_kernel_ptr(int mode);   // 0 SIMPLE, 1 zero copy, 2 posted copy, 3 posted direct
int p2p_tma_threads();
int p2p_tma_smem();
void* ll_kernel_ptr();
void* ll128_kernel_ptr();
int ll128_smem();
int ll128_threads();
void* ll_pingpong_kernel_ptr();
void* ring_kernel_ptr(int dtype);
void* ring_tma_kernel_ptr(int dtype);
int ring_tma_threads();
int ring_tma_smem();
}  // namespace xp

using xp::DevStatus;

namespace {

thread_local std::string g_err;
// Spin timeout of device waits; XP_SPIN_TIMEOUT_NS in the environment sets the
// starting value (1e3 .. 6e10 ns), xp_set_spin_timeout_ns changes it.
unsigned long long initial_timeout_ns() {
  const char* e = getenv("XP_SPIN_TIMEOUT_NS");
  if (!e || !*e) return 2000000000ull;
  char* end = nullptr;
  const unsigned long long v = strtoull(e, &end, 10);
  if (*end || v < 1000ull || v > 60000000000ull) return 2000000000ull;
  return v;
}
std::atomic<unsigned long long> g_timeout_ns{initial_timeout_ns()};
std::mutex g_mu;
int* g_abort_host = nullptr;
int* g_abort_dev = nullptr;

xp_status fail(xp_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

#define XP_CUDA(call)                                                                     \
  do {                                                                                    \
    cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess) return fail(XP_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

size_t round_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

xp_status ensure_abort_word() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_abort_host) return XP_OK;
  int* h = nullptr;
  XP_CUDA(cudaHostAlloc(reinterpret_cast<void**>(&h), 64, cudaHostAllocMapped | cudaHostAllocPortable));
  memset(h, 0, 64);
  int* d = nullptr;
  cudaError_t e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&d), h, 0);
  if (e != cudaSuccess) {
    cudaFreeHost(h);
    return fail(XP_ERR_CUDA, "cudaHostGetDevicePointer: %s", cudaGetErrorString(e));
  }
  g_abort_host = h;
  g_abort_dev = d;
  return XP_OK;
}

// One allocation holding control blocks and slots, in HBM or mapped host memory.
struct Mem {
  char* host = nullptr;   // host view (mapped placement only)
  char* dev = nullptr;    // device view
  size_t bytes = 0;
  xp_placement place = XP_PLACE_DEVICE;
};

xp_status mem_alloc(Mem& m, size_t bytes, xp_placement place) {
  m.bytes = bytes;
  m.place = place;
  if (place == XP_PLACE_DEVICE) {
    XP_CUDA(cudaMalloc(reinterpret_cast<void**>(&m.dev), bytes));
  } else {
    XP_CUDA(cudaHostAlloc(reinterpret_cast<void**>(&m.host), bytes, cudaHostAllocMapped | cudaHostAllocPortable));
    cudaError_t e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&m.dev), m.host, 0);
    if (e != cudaSuccess) {
      cudaFreeHost(m.host);
      m.host = nullptr;
      return fail(XP_ERR_CUDA, "cudaHostGetDevicePointer: %s", cudaGetErrorString(e));
    }
  }
  return XP_OK;
}

void mem_free(Mem& m) {
  if (m.place == XP_PLACE_DEVICE) {
    if (m.dev) cudaFree(m.dev);
  } else if (m.host) {
    cudaFreeHost(m.host);
  }
  m.host = m.dev = nullptr;
}

// Zero the whole region, then set every size word of `nfifos` control
// blocks to -1.
// Set-up and reset write device memory on the object's own non-blocking
// stream (`st`) and wait for that stream only.  A copy on the legacy default
// stream would queue behind whatever runs there, such as a proxy-mode
// transfer that waits for the pump's copies, and could hold those copies up
// in a shared copy queue until the transfer times out.
xp_status mem_init(Mem& m, int nfifos, cudaStream_t st) {
  const size_t ctl_bytes = (size_t)nfifos * xp::kCtlBytes;
  std::vector<char> img(ctl_bytes, 0);
  for (int f = 0; f < nfifos; ++f) {
    long long* sz = reinterpret_cast<long long*>(img.data() + (size_t)f * xp::kCtlBytes + xp::kSizeOff);
    for (int k = 0; k < xp::kMaxSlots; ++k) sz[k] = -1;
  }
  if (m.place == XP_PLACE_DEVICE) {
    XP_CUDA(cudaMemsetAsync(m.dev, 0, m.bytes, st));
    XP_CUDA(cudaMemcpyAsync(m.dev, img.data(), ctl_bytes, cudaMemcpyHostToDevice, st));
    XP_CUDA(cudaStreamSynchronize(st));
  } else {
    memset(m.host, 0, m.bytes);
    memcpy(m.host, img.data(), ctl_bytes);
  }
  return XP_OK;
}

struct Common {
  int device = 0;
  unsigned long long ops = 0;    // operations launched: the id of the next one is ops + 1
  DevStatus* status = nullptr;   // device memory
  cudaEvent_t done = nullptr;
  cudaStream_t query = nullptr;
  bool used = false;
};

xp_status common_init(Common& c) {
  XP_CUDA(cudaGetDevice(&c.device));
  XP_CUDA(cudaMalloc(reinterpret_cast<void**>(&c.status), sizeof(DevStatus)));
  XP_CUDA(cudaEventCreateWithFlags(&c.done, cudaEventDisableTiming));
  XP_CUDA(cudaStreamCreateWithFlags(&c.query, cudaStreamNonBlocking));
  XP_CUDA(cudaMemsetAsync(c.status, 0, sizeof(DevStatus), c.query));
  XP_CUDA(cudaStreamSynchronize(c.query));
  return XP_OK;
}

void common_free(Common& c) {
  if (c.done) cudaEventSynchronize(c.done);
  if (c.status) cudaFree(c.status);
  if (c.done) cudaEventDestroy(c.done);
  if (c.query) cudaStreamDestroy(c.query);
  c = Common();
}

xp_status check_device(const Common& c) {
  int d = -1;
  XP_CUDA(cudaGetDevice(&d));
  if (d != c.device) return fail(XP_ERR_INVALID, "current device %d is not the object's device %d", d, c.device);
  return XP_OK;
}

xp_status read_status(Common& c, int sync, xp_report* rep) {
  if (sync && c.used) XP_CUDA(cudaEventSynchronize(c.done));
  DevStatus h;
  XP_CUDA(cudaMemcpyAsync(&h, c.status, sizeof h, cudaMemcpyDeviceToHost, c.query));
  XP_CUDA(cudaStreamSynchronize(c.query));
  // only the last operation's claim and occupancy count (their ids match
  // the one the operation wrote as it started)
  const unsigned long long id = h.last_op & 0xffffffffull;
  const int code = (h.claim >> 32) == id ? (int)(uint32_t)h.claim : 0;
  const uint32_t occupancy = (h.occupancy >> 32) == id ? (uint32_t)h.occupancy : 0u;
  if (rep) {
    rep->code = code;
    rep->channel = code ? h.channel : -1;
    rep->where = h.where;
    rep->reserved = 0;
    rep->observed = h.observed;
    rep->expected = h.expected;
    rep->max_occupancy = occupancy;
    rep->reserved2 = 0;
  }
  if (code < 0 || code > XP_ERR_INTERNAL) return XP_ERR_INTERNAL;
  return static_cast<xp_status>(code);
}

// Cluster co-residency: every cluster of the launch must fit on the GPU.
std::map<std::tuple<const void*, int, int>, int> g_fits;

// csize > 0: thread-block clusters of csize CTAs, each of which must fit on
// the GPU.  csize == 0: a cooperative launch without clusters, which the
// driver runs only if every CTA of the grid is resident at once.
xp_status launch(const void* kernel, int grid, int block, int csize, void* params, cudaStream_t stream,
                 int smem = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  if (csize > 0) {
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = csize;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
  } else {
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
  }
  cfg.attrs = at;
  cfg.numAttrs = 1;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_tuple(kernel, csize, block);
    auto it = g_fits.find(key);
    if (it == g_fits.end()) {
      if (csize > 8) XP_CUDA(cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
      if (smem > 48 * 1024) XP_CUDA(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
      int n = 0;
      if (csize > 0) {
        XP_CUDA(cudaOccupancyMaxActiveClusters(&n, kernel, &cfg));
      } else {
        int per_sm = 0, dev = 0, sms = 0;
        XP_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, block, (size_t)smem));
        XP_CUDA(cudaGetDevice(&dev));
        XP_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
        n = per_sm * sms;   // CTAs resident at once
      }
      it = g_fits.emplace(key, n).first;
    }
    if (csize > 0 && it->second < 1)
      return fail(XP_ERR_INVALID, "a cluster of %d CTAs x %d threads cannot be resident on this GPU", csize, block);
    if (csize == 0 && it->second < grid)
      return fail(XP_ERR_INVALID, "a cooperative grid of %d CTAs does not fit (%d resident at most)", grid, it->second);
  }
  void* args[] = {params};
  XP_CUDA(cudaLaunchKernelExC(&cfg, kernel, args));
  return XP_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// CTAs of `kernel` (block threads, smem bytes of dynamic shared memory)
// resident on this GPU at once; 0 if unknown.
std::map<const void*, int> g_resident;
int resident_ctas(const void* kernel, int block, int smem) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_resident.find(kernel);
    if (it != g_resident.end()) return it->second;
  }
  int per_sm = 0, dev = 0, sms = 0;
  if ((smem > 48 * 1024 &&
       cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, block, (size_t)smem) != cudaSuccess ||
      cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  g_resident[kernel] = per_sm * sms;
  return per_sm * sms;
}

// Live FIFO data one launch of an automatic-lane HBM ring may keep, about a
// quarter of L2.  Measured on 8 ranks x 256 MiB fp32, 8 channels of
// 8 x 512 KiB (16 MiB of live slots per channel): all 8 channels in one
// launch at 2 lanes 1.74 ms; groups of 4 channels at 4 lanes 1.67 ms; of 2 at
// 8 lanes 1.57 ms; of 1 at 16 lanes 1.93-2.01 ms (stripes too short).
constexpr size_t kRingLiveBytes = (size_t)32 << 20;

// CTAs of the bulk-copy ring kernel resident on this GPU at once
int ring_tma_resident() {
  const int a = resident_ctas(xp::ring_tma_kernel_ptr(XP_F32), xp::ring_tma_threads(), xp::ring_tma_smem());
  const int b = resident_ctas(xp::ring_tma_kernel_ptr(XP_I32), xp::ring_tma_threads(), xp::ring_tma_smem());
  return a < b ? a : b;
}

// Marks the object's last operation on `st`.  Inside a stream capture the
// operation becomes a graph node and nothing is recorded (an event recorded
// during capture cannot be waited on afterwards): the caller synchronises the
// graph's replays before reading the status.
xp_status record_done(Common& c, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
    (void)cudaGetLastError();
    cs = cudaStreamCaptureStatusNone;
  }
  if (cs != cudaStreamCaptureStatusNone) return XP_OK;
  XP_CUDA(cudaEventRecord(c.done, st));
  c.used = true;
  return XP_OK;
}

}  // namespace

namespace xp {
// Sets the message xp_last_error() returns on this thread.
void set_last_error(const char* msg) { g_err = msg; }
}  // namespace xp

struct xp_fifo {
  Common cm;
  int C = 0, N = 0;
  size_t S = 0;
  xp_proto proto = XP_PROTO_SIMPLE;
  xp_placement place = XP_PLACE_DEVICE;
  int lanes = 1;           // sender CTAs per channel
  int rlanes = 1;          // receiver CTAs per channel
  int discard = -1;        // receivers drop the slot lines they read from L2: 1, 0, or -1 (by FIFO size)
  Mem mem;
  char* ctl = nullptr;     // device view
  char* slots = nullptr;   // device view
  char* pctl = nullptr;    // device view: posted-FIFO blocks
  unsigned long long* arr = nullptr;   // device: lane arrival counters (always HBM)
  xp::ChanStats* stats = nullptr;   // device: one record per channel
  size_t ctl_region = 0;
  size_t pctl_region = 0;
  size_t ch_stride = 0;
  // proxy (copy-engine) mode, set up by xp_fifo_enable_ce
  Mem ce_mem;              // mapped host memory: per-channel proxy blocks
  Mem ring_mem;            // device: send ring (+ receive ring for 2 hops)
  char* send_ring = nullptr;
  char* recv_ring = nullptr;
  int hops = 0;
  xp::Pump* pump = nullptr;
  // staged (host -> device -> FIFO -> device -> host) transfers, made on first use
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
};

struct xp_ring {
  Common cm;
  int P = 0, C = 0, N = 0;
  size_t S = 0;
  xp_placement place = XP_PLACE_DEVICE;
  int lanes = 0;           // 0: chosen per operation (HBM rings), else CTAs per rank per channel
  Mem mem;
  char* ctl = nullptr;
  char* slots = nullptr;
  size_t ctl_region = 0;
  size_t fifo_stride = 0;
};

extern "C" {

int xp_version(void) { return 1; }

const char* xp_last_error(void) { return g_err.c_str(); }

const char* xp_status_string(xp_status s) {
  switch (s) {
    case XP_OK: return "ok";
    case XP_ERR_INVALID: return "invalid argument";
    case XP_ERR_CUDA: return "CUDA error";
    case XP_ERR_TIMEOUT: return "device wait timed out";
    case XP_ERR_BOUNDS: return "size word or occupancy out of bounds";
    case XP_ERR_ABORTED: return "aborted";
    case XP_ERR_INTERNAL: return "internal error";
  }
  return "unknown status";
}

xp_status xp_set_spin_timeout_ns(uint64_t ns) {
  if (ns < 1000ull || ns > 60000000000ull) return fail(XP_ERR_INVALID, "timeout %llu ns out of range", (unsigned long long)ns);
  g_timeout_ns = ns;
  return XP_OK;
}

xp_status xp_abort(int value) {
  xp_status s = ensure_abort_word();
  if (s != XP_OK) return s;
  *reinterpret_cast<volatile int*>(g_abort_host) = value ? 1 : 0;
  return XP_OK;
}

xp_status xp_fifo_create(int nchannels, int nslots, size_t slot_bytes, xp_proto proto, xp_placement place,
                         xp_fifo** out) {
  if (!out) return fail(XP_ERR_INVALID, "out is NULL");
  if (nchannels < 1 || nchannels > xp::kMaxChannels) return fail(XP_ERR_INVALID, "nchannels %d not in [1, 64]", nchannels);
  if (nslots < 1 || nslots > xp::kMaxSlots) return fail(XP_ERR_INVALID, "nslots %d not in [1, 64]", nslots);
  if (slot_bytes == 0 || slot_bytes % 16 || slot_bytes > (1ull << 31))
    return fail(XP_ERR_INVALID, "slot_bytes %zu must be a non-zero multiple of 16, at most 2^31", slot_bytes);
  if (proto != XP_PROTO_SIMPLE && proto != XP_PROTO_LL && proto != XP_PROTO_LL128)
    return fail(XP_ERR_INVALID, "unknown protocol %d", (int)proto);
  if (proto == XP_PROTO_LL128 && slot_bytes % 128)
    return fail(XP_ERR_INVALID, "LL128 slot_bytes %zu is not a multiple of 128-byte lines", slot_bytes);
  if (place != XP_PLACE_DEVICE && place != XP_PLACE_HOST_MAPPED) return fail(XP_ERR_INVALID, "unknown placement %d", (int)place);
  if ((unsigned long long)nchannels * nslots * slot_bytes > (1ull << 40)) return fail(XP_ERR_INVALID, "FIFO larger than 2^40 bytes");
  xp_status s = ensure_abort_word();
  if (s != XP_OK) return s;
  xp_fifo* f = new xp_fifo();
  f->C = nchannels;
  f->N = nslots;
  f->S = slot_bytes;
  f->proto = proto;
  f->place = place;
  f->ctl_region = round_up((size_t)nchannels * xp::kCtlBytes, 4096);
  f->pctl_region = (size_t)nchannels * xp::kPostCtlBytes;
  f->ch_stride = round_up((size_t)nslots * slot_bytes, 4096);
  if ((s = common_init(f->cm)) != XP_OK ||
      (s = mem_alloc(f->mem, f->ctl_region + f->pctl_region + nchannels * f->ch_stride, place)) != XP_OK ||
      (s = mem_init(f->mem, nchannels, f->cm.query)) != XP_OK) {
    common_free(f->cm);
    mem_free(f->mem);
    delete f;
    return s;
  }
  if (cudaMalloc(reinterpret_cast<void**>(&f->stats), (size_t)nchannels * sizeof(xp::ChanStats)) != cudaSuccess ||
      cudaMemsetAsync(f->stats, 0, (size_t)nchannels * sizeof(xp::ChanStats), f->cm.query) != cudaSuccess ||
      cudaMalloc(reinterpret_cast<void**>(&f->arr), (size_t)nchannels * xp::kArrBytes) != cudaSuccess ||
      cudaMemsetAsync(f->arr, 0, (size_t)nchannels * xp::kArrBytes, f->cm.query) != cudaSuccess ||
      cudaStreamSynchronize(f->cm.query) != cudaSuccess) {
    if (f->stats) cudaFree(f->stats);
    if (f->arr) cudaFree(f->arr);
    common_free(f->cm);
    mem_free(f->mem);
    delete f;
    return fail(XP_ERR_CUDA, "allocating the channel records failed");
  }
  f->ctl = f->mem.dev;
  f->pctl = f->mem.dev + f->ctl_region;
  f->slots = f->pctl + f->pctl_region;
  *out = f;
  return XP_OK;
}

xp_status xp_fifo_destroy(xp_fifo* f) {
  if (!f) return XP_OK;
  cudaDeviceSynchronize();
  xp::pump_stop(f->pump);
  for (cudaEvent_t e : f->ev)
    if (e) cudaEventDestroy(e);
  if (f->s_in) cudaStreamDestroy(f->s_in);
  if (f->s_out) cudaStreamDestroy(f->s_out);
  common_free(f->cm);
  mem_free(f->mem);
  if (f->stats) cudaFree(f->stats);
  if (f->arr) cudaFree(f->arr);
  mem_free(f->ce_mem);
  mem_free(f->ring_mem);
  delete f;
  return XP_OK;
}

static xp::PumpConfig pump_config(const xp_fifo* f) {
  xp::PumpConfig cfg;
  cfg.device = f->cm.device;
  cfg.nchannels = f->C;
  cfg.nslots = f->N;
  cfg.slot_bytes = f->S;
  cfg.ch_stride = f->ch_stride;
  cfg.hops = f->hops;
  cfg.ce_host = f->ce_mem.host;
  cfg.rings[0] = f->send_ring;
  if (f->hops == 1) {
    cfg.rings[1] = f->slots;
  } else {
    cfg.rings[1] = f->mem.host + (f->slots - f->mem.dev);   // the FIFO's own slots, host view
    cfg.rings[2] = f->recv_ring;
  }
  return cfg;
}

xp_status xp_fifo_enable_ce(xp_fifo* f) {
  if (!f) return fail(XP_ERR_INVALID, "fifo is NULL");
  if (f->proto != XP_PROTO_SIMPLE) return fail(XP_ERR_INVALID, "the proxy mode needs a SIMPLE FIFO");
  if (f->pump) return XP_OK;
  xp_status s = check_device(f->cm);
  if (s != XP_OK) return s;
  const int hops = f->place == XP_PLACE_DEVICE ? 1 : 2;
  const size_t ring = (size_t)f->C * f->ch_stride;
  if ((s = mem_alloc(f->ring_mem, hops * ring, XP_PLACE_DEVICE)) != XP_OK) return s;
  if ((s = mem_alloc(f->ce_mem, (size_t)f->C * xp::kCeCtlBytes, XP_PLACE_HOST_MAPPED)) != XP_OK) {
    mem_free(f->ring_mem);
    return s;
  }
  memset(f->ce_mem.host, 0, f->ce_mem.bytes);
  f->hops = hops;
  f->send_ring = f->ring_mem.dev;
  f->recv_ring = hops == 1 ? f->slots : f->ring_mem.dev + ring;
  std::string err;
  f->pump = xp::pump_start(pump_config(f), &err);
  if (!f->pump) {
    mem_free(f->ce_mem);
    mem_free(f->ring_mem);
    f->hops = 0;
    f->send_ring = f->recv_ring = nullptr;
    return fail(XP_ERR_CUDA, "%s", err.c_str());
  }
  return XP_OK;
}

xp_status xp_fifo_set_lanes(xp_fifo* f, int lanes) {
  if (!f) return fail(XP_ERR_INVALID, "fifo is NULL");
  if (f->proto == XP_PROTO_LL128) {
    // sender and receiver lanes (the receiver side may then be changed with
    // xp_fifo_set_recv_lanes); each receiver lane keeps a head of its own
    // (lane 0: the channel's head word, lanes 1 .. 7: lines of the channel's
    // arrival block)
    if (lanes < 1 || lanes > 8) return fail(XP_ERR_INVALID, "LL128 lanes %d not in [1, 8]", lanes);
    f->lanes = f->rlanes = lanes;
    return XP_OK;
  }
  if (f->proto != XP_PROTO_SIMPLE) return fail(XP_ERR_INVALID, "lanes apply to SIMPLE and LL128 FIFOs only");
  if (lanes < 1 || lanes > xp::kMaxLanes) return fail(XP_ERR_INVALID, "lanes %d not in [1, 32]", lanes);
  f->lanes = lanes;
  f->rlanes = lanes <= xp::kMaxCluster / 2 ? lanes : (lanes < xp::kMaxCluster ? xp::kMaxCluster - lanes : 1);
  return XP_OK;
}

xp_status xp_fifo_set_recv_lanes(xp_fifo* f, int rlanes) {
  if (!f) return fail(XP_ERR_INVALID, "fifo is NULL");
  if (f->proto == XP_PROTO_LL128) {
    if (rlanes < 1 || rlanes > 8) return fail(XP_ERR_INVALID, "LL128 receiver lanes %d not in [1, 8]", rlanes);
    f->rlanes = rlanes;
    return XP_OK;
  }
  if (f->proto != XP_PROTO_SIMPLE) return fail(XP_ERR_INVALID, "lanes apply to SIMPLE and LL128 FIFOs only");
  if (rlanes < 1 || rlanes > xp::kMaxLanes) return fail(XP_ERR_INVALID, "receiver lanes %d not in [1, 32]", rlanes);
  f->rlanes = rlanes;
  return XP_OK;
}

xp_status xp_fifo_set_discard(xp_fifo* f, int on) {
  if (!f) return fail(XP_ERR_INVALID, "fifo is NULL");
  f->discard = on > 0 ? 1 : on == 0 ? 0 : -1;
  return XP_OK;
}

// Automatic choice: a FIFO whose slots take a small part of L2 has its lines
// rewritten before L2 would evict them, so dropping them saves no DRAM
// traffic and only lengthens the credit path; a large one gains.  Measured
// with 1 GiB through 16 channels x 8 slots: 4, 8 and 16 MiB of slots move the
// same either way, 32 MiB 1.4% faster without drops, 64 MiB 16% faster with
// them; the 1 MiB loopback through 8 x 64 KiB takes 3 us less without.
static bool discard_on(const xp_fifo* f) {
  if (f->discard >= 0) return f->discard != 0;
  return (size_t)f->C * (size_t)f->N * f->S >= XP_DISCARD_AUTO_BYTES;
}

xp_status xp_fifo_describe(const xp_fifo* f, int channel, xp_channel_desc* out) {
  if (!f || !out) return fail(XP_ERR_INVALID, "NULL argument");
  if (channel < 0 || channel >= f->C) return fail(XP_ERR_INVALID, "channel %d out of range", channel);
  out->ctl = f->ctl + (size_t)channel * xp::kCtlBytes;
  out->slots = f->slots + (size_t)channel * f->ch_stride;
  out->slot_stride = f->S;
  out->nslots = f->N;
  out->proto = f->proto;
  out->placement = f->place;
  out->lanes = f->lanes;
  out->recv_lanes = f->rlanes;
  out->posted = f->pctl + (size_t)channel * xp::kPostCtlBytes;
  out->ce = f->pump ? f->ce_mem.dev + (size_t)channel * xp::kCeCtlBytes : nullptr;
  out->send_ring = f->pump ? f->send_ring + (size_t)channel * f->ch_stride : nullptr;
  out->recv_ring = f->pump ? f->recv_ring + (size_t)channel * f->ch_stride : nullptr;
  out->discard = discard_on(f) ? 1 : 0;
  return XP_OK;
}

enum { kOpSimple = 0, kOpZeroCopy = 1, kOpPostedCopy = 2, kOpPostedDirect = 3, kOpProxy = 4 };   // p2p_tma_kernel_ptr modes

static xp_status p2p_op(xp_fifo* f, const void* src, void* dst, size_t bytes, xp_stream_t stream, int mode) {
  const bool zero_copy = mode == kOpZeroCopy;
  const bool posted = mode == kOpPostedCopy || mode == kOpPostedDirect;
  if (!f) return fail(XP_ERR_INVALID, "fifo is NULL");
  if (bytes == 0) return XP_OK;
  if (!src || !dst) return fail(XP_ERR_INVALID, "src or dst is NULL");
  if (!aligned16(src) || !aligned16(dst)) return fail(XP_ERR_INVALID, "src and dst must be 16-byte aligned");
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
  if (s0 < d0 + bytes && d0 < s0 + bytes) return fail(XP_ERR_INVALID, "src and dst overlap");
  if (zero_copy && f->proto != XP_PROTO_SIMPLE) return fail(XP_ERR_INVALID, "zero copy needs a SIMPLE FIFO");
  if (posted && (f->proto != XP_PROTO_SIMPLE || f->place != XP_PLACE_DEVICE))
    return fail(XP_ERR_INVALID, "posted transfers need a SIMPLE FIFO in device memory");
  if (mode == kOpProxy && !f->pump) return fail(XP_ERR_INVALID, "the proxy mode is not enabled (xp_fifo_enable_ce)");
  if (f->proto != XP_PROTO_SIMPLE && bytes % 8)
    return fail(XP_ERR_INVALID, "LL and LL128 move whole 8-byte words: bytes %% 8 != 0");
  xp_status s = check_device(f->cm);
  if (s != XP_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  xp::P2pParams p = {};
  p.ctl = f->ctl;
  p.arr = f->arr;
  p.stats = f->stats;
  p.pctl = f->pctl;
  p.ce = f->ce_mem.dev;
  p.send_ring = f->send_ring;
  p.recv_ring = f->recv_ring;
  p.hops = f->hops;
  p.discard = discard_on(f) ? 1 : 0;
  p.slots = f->slots;
  p.ch_stride = f->ch_stride;
  p.src = static_cast<const char*>(src);
  p.dst = static_cast<char*>(dst);
  p.nbytes = bytes;
  p.nchannels = f->C;
  p.nslots = f->N;
  p.slot_bytes = (unsigned)f->S;
  p.status = f->cm.status;
  p.abort_word = g_abort_dev;
  p.timeout_ns = g_timeout_ns.load();
  const void* kernel;
  int csize, block, smem = 0;
  if (f->proto != XP_PROTO_SIMPLE) {
    kernel = f->proto == XP_PROTO_LL ? xp::ll_kernel_ptr() : xp::ll128_kernel_ptr();
    // LL: one cluster of a sender and a receiver CTA per channel; LL128: the
    // channel's sender lanes, then its receiver lanes
    p.lanes = f->proto == XP_PROTO_LL ? 1 : f->lanes;
    p.rlanes = f->proto == XP_PROTO_LL ? 1 : f->rlanes;
    csize = p.lanes + p.rlanes;
    block = f->proto == XP_PROTO_LL ? xp::kLLThreads : xp::ll128_threads();
    if (f->proto == XP_PROTO_LL128) smem = xp::ll128_smem();
  } else {
    p.lanes = f->lanes;
    p.rlanes = (zero_copy || mode == kOpPostedDirect) ? 1 : f->rlanes;
    csize = p.lanes + p.rlanes;
    if (f->place == XP_PLACE_DEVICE || mode == kOpProxy) {
      // HBM FIFO (or the proxy mode's device rings): bulk copies through shared memory
      kernel = xp::p2p_tma_kernel_ptr(mode);
      block = xp::p2p_tma_threads();
      smem = xp::p2p_tma_smem();
    } else {
      // mapped host FIFO: 16-byte vector loads and stores from every warp
      kernel = xp::p2p_kernel_ptr(zero_copy);
      block = xp::kP2pThreads;
    }
  }
  p.csize = csize;
  // The bulk-copy and LL128 kernels need the sender and receiver CTAs of a
  // channel resident together: a cooperative grid when all of it fits at
  // once (no cluster placement limits), else one cluster per channel.  The
  // other kernels always use clusters.
  int launch_csize = csize;
  if ((kernel == xp::p2p_tma_kernel_ptr(mode) || kernel == xp::ll128_kernel_ptr()) &&
      f->C * csize <= resident_ctas(kernel, block, smem))
    launch_csize = 0;
  if (launch_csize > xp::kMaxCluster)
    return fail(XP_ERR_INVALID, "%d channels x %d CTAs neither fit on the GPU at once nor form clusters of at most 16",
                f->C, csize);
  p.op = ++f->cm.ops;
  const int grid = f->C * csize;
  if ((s = launch(kernel, grid, block, launch_csize, &p, st, smem)) != XP_OK) return s;
  if (mode == kOpProxy) xp::pump_kick(f->pump);
  return record_done(f->cm, st);
}

xp_status xp_send_recv(xp_fifo* f, const void* src, void* dst, size_t bytes, xp_stream_t stream) {
  return p2p_op(f, src, dst, bytes, stream, kOpSimple);
}

xp_status xp_send_recv_zero_copy(xp_fifo* f, const void* src, void* dst, size_t bytes, xp_stream_t stream) {
  return p2p_op(f, src, dst, bytes, stream, kOpZeroCopy);
}

xp_status xp_send_recv_posted(xp_fifo* f, const void* src, void* dst, size_t bytes, int direct, xp_stream_t stream) {
  return p2p_op(f, src, dst, bytes, stream, direct ? kOpPostedDirect : kOpPostedCopy);
}

xp_status xp_send_recv_ce(xp_fifo* f, const void* src, void* dst, size_t bytes, xp_stream_t stream) {
  return p2p_op(f, src, dst, bytes, stream, kOpProxy);
}

xp_status xp_send_recv_staged(xp_fifo* f, const void* host_src, void* host_dst, void* dev_src, void* dev_dst,
                              size_t bytes, size_t chunk_bytes, xp_stream_t stream) {
  if (!f) return fail(XP_ERR_INVALID, "fifo is NULL");
  if (bytes == 0) return XP_OK;
  if (!host_src || !host_dst || !dev_src || !dev_dst) return fail(XP_ERR_INVALID, "a buffer is NULL");
  if (chunk_bytes == 0) chunk_bytes = (size_t)64 << 20;
  if (chunk_bytes % 16) return fail(XP_ERR_INVALID, "chunk_bytes %zu is not a multiple of 16", chunk_bytes);
  if (f->proto != XP_PROTO_SIMPLE && bytes % 8)
    return fail(XP_ERR_INVALID, "LL and LL128 move whole 8-byte words: bytes %% 8 != 0");
  xp_status s = check_device(f->cm);
  if (s != XP_OK) return s;
  if (!f->s_in) {
    XP_CUDA(cudaStreamCreateWithFlags(&f->s_in, cudaStreamNonBlocking));
    XP_CUDA(cudaStreamCreateWithFlags(&f->s_out, cudaStreamNonBlocking));
    for (cudaEvent_t& e : f->ev) XP_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // everything starts after the work already on `stream`
  XP_CUDA(cudaEventRecord(f->ev[0], st));
  XP_CUDA(cudaStreamWaitEvent(f->s_in, f->ev[0], 0));
  XP_CUDA(cudaStreamWaitEvent(f->s_out, f->ev[0], 0));
  const char* hs = static_cast<const char*>(host_src);
  char* hd = static_cast<char*>(host_dst);
  char* ds = static_cast<char*>(dev_src);
  char* dd = static_cast<char*>(dev_dst);
  for (size_t off = 0; off < bytes; off += chunk_bytes) {
    const size_t n = bytes - off < chunk_bytes ? bytes - off : chunk_bytes;
    // chunk i: copy in on s_in | transfer on `stream` | copy out on s_out;
    // each event is waited on right after it is recorded, so two suffice
    XP_CUDA(cudaMemcpyAsync(ds + off, hs + off, n, cudaMemcpyHostToDevice, f->s_in));
    XP_CUDA(cudaEventRecord(f->ev[1], f->s_in));
    XP_CUDA(cudaStreamWaitEvent(st, f->ev[1], 0));
    if ((s = p2p_op(f, ds + off, dd + off, n, stream, kOpSimple)) != XP_OK) return s;
    XP_CUDA(cudaEventRecord(f->ev[2], st));
    XP_CUDA(cudaStreamWaitEvent(f->s_out, f->ev[2], 0));
    XP_CUDA(cudaMemcpyAsync(hd + off, dd + off, n, cudaMemcpyDeviceToHost, f->s_out));
  }
  XP_CUDA(cudaEventRecord(f->ev[0], f->s_out));
  XP_CUDA(cudaStreamWaitEvent(st, f->ev[0], 0));
  return record_done(f->cm, st);
}

xp_status xp_fifo_status(xp_fifo* f, int sync, xp_report* report) {
  if (!f) return fail(XP_ERR_INVALID, "fifo is NULL");
  const xp_status s = read_status(f->cm, sync, report);
  if (const char* e = xp::pump_error(f->pump)) xp::set_last_error(e);
  return s;
}

xp_status xp_fifo_stats(xp_fifo* f, int channel, xp_channel_stats* out) {
  if (!f || !out) return fail(XP_ERR_INVALID, "NULL argument");
  if (channel < 0 || channel >= f->C) return fail(XP_ERR_INVALID, "channel %d out of range", channel);
  if (f->cm.used) XP_CUDA(cudaEventSynchronize(f->cm.done));
  xp::ChanStats h;
  XP_CUDA(cudaMemcpyAsync(&h, f->stats + channel, sizeof h, cudaMemcpyDeviceToHost, f->cm.query));
  XP_CUDA(cudaStreamSynchronize(f->cm.query));
  out->steps = h.steps;
  out->t_start_ns = h.t_start;
  out->t_end_ns = h.t_end;
  out->send_polls = h.send_polls;
  out->recv_polls = h.recv_polls;
  return XP_OK;
}

xp_status xp_fifo_reset(xp_fifo* f) {
  if (!f) return fail(XP_ERR_INVALID, "fifo is NULL");
  if (f->cm.used) XP_CUDA(cudaEventSynchronize(f->cm.done));
  XP_CUDA(cudaMemsetAsync(f->cm.status, 0, sizeof(DevStatus), f->cm.query));
  XP_CUDA(cudaMemsetAsync(f->arr, 0, (size_t)f->C * xp::kArrBytes, f->cm.query));
  XP_CUDA(cudaStreamSynchronize(f->cm.query));
  if (f->pump) {
    // restart the pump on zeroed proxy counters
    xp::pump_stop(f->pump);
    f->pump = nullptr;
    memset(f->ce_mem.host, 0, f->ce_mem.bytes);
    std::string err;
    f->pump = xp::pump_start(pump_config(f), &err);
    if (!f->pump) return fail(XP_ERR_CUDA, "%s", err.c_str());
  }
  return mem_init(f->mem, f->C, f->cm.query);
}

xp_status xp_ll_pingpong(xp_fifo* ab, xp_fifo* ba, int iters, uint64_t* elapsed_ns, xp_stream_t stream) {
  if (!ab || !ba || !elapsed_ns) return fail(XP_ERR_INVALID, "NULL argument");
  if (ab == ba) return fail(XP_ERR_INVALID, "ping-pong needs two FIFOs");
  if (ab->proto != XP_PROTO_LL || ba->proto != XP_PROTO_LL) return fail(XP_ERR_INVALID, "ping-pong needs LL FIFOs");
  if (iters < 1 || iters > 10000000) return fail(XP_ERR_INVALID, "iters %d not in [1, 1e7]", iters);
  xp_status s = check_device(ab->cm);
  if (s != XP_OK) return s;
  if ((s = check_device(ba->cm)) != XP_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  xp::PingParams p = {};
  p.ctl_ab = ab->ctl;
  p.slots_ab = ab->slots;
  p.ctl_ba = ba->ctl;
  p.slots_ba = ba->slots;
  p.nslots_ab = ab->N;
  p.nslots_ba = ba->N;
  p.slot_bytes_ab = (unsigned)ab->S;
  p.slot_bytes_ba = (unsigned)ba->S;
  p.iters = iters;
  p.elapsed = &ab->cm.status->elapsed;
  p.status = ab->cm.status;
  p.abort_word = g_abort_dev;
  p.timeout_ns = g_timeout_ns.load();
  p.op = ++ab->cm.ops;
  ++ba->cm.ops;
  if ((s = launch(xp::ll_pingpong_kernel_ptr(), 2, 32, 2, &p, st)) != XP_OK) return s;
  XP_CUDA(cudaEventRecord(ab->cm.done, st));
  XP_CUDA(cudaEventRecord(ba->cm.done, st));
  ab->cm.used = ba->cm.used = true;
  XP_CUDA(cudaEventSynchronize(ab->cm.done));
  DevStatus h;
  XP_CUDA(cudaMemcpyAsync(&h, ab->cm.status, sizeof h, cudaMemcpyDeviceToHost, ab->cm.query));
  XP_CUDA(cudaStreamSynchronize(ab->cm.query));
  if ((h.claim >> 32) == (p.op & 0xffffffffull) && (uint32_t)h.claim != XP_OK)
    return static_cast<xp_status>((uint32_t)h.claim);
  *elapsed_ns = h.elapsed;
  return XP_OK;
}

xp_status xp_ring_create(int nranks, int nchannels, int nslots, size_t slot_bytes, xp_placement place, xp_ring** out) {
  if (!out) return fail(XP_ERR_INVALID, "out is NULL");
  if (nranks < 2 || nranks > xp::kMaxRanks) return fail(XP_ERR_INVALID, "nranks %d not in [2, 16]", nranks);
  if (nchannels < 1 || nchannels > xp::kMaxChannels) return fail(XP_ERR_INVALID, "nchannels %d not in [1, 64]", nchannels);
  if (nslots < 2 || nslots > xp::kMaxSlots) return fail(XP_ERR_INVALID, "the ring needs 2 <= nslots <= 64, got %d", nslots);
  if (slot_bytes == 0 || slot_bytes % 16 || slot_bytes > (1ull << 31))
    return fail(XP_ERR_INVALID, "slot_bytes %zu must be a non-zero multiple of 16, at most 2^31", slot_bytes);
  if (place != XP_PLACE_DEVICE && place != XP_PLACE_HOST_MAPPED) return fail(XP_ERR_INVALID, "unknown placement %d", (int)place);
  if ((unsigned long long)nranks * nchannels * nslots * slot_bytes > (1ull << 40)) return fail(XP_ERR_INVALID, "FIFOs larger than 2^40 bytes");
  xp_status s = ensure_abort_word();
  if (s != XP_OK) return s;
  xp_ring* r = new xp_ring();
  r->P = nranks;
  r->C = nchannels;
  r->N = nslots;
  r->S = slot_bytes;
  r->place = place;
  const int nf = nranks * nchannels;
  r->ctl_region = round_up((size_t)nf * xp::kRingMaxLanes * xp::kCtlBytes, 4096);
  r->fifo_stride = round_up((size_t)nslots * slot_bytes, 4096);
  if ((s = common_init(r->cm)) != XP_OK || (s = mem_alloc(r->mem, r->ctl_region + nf * r->fifo_stride, place)) != XP_OK ||
      (s = mem_init(r->mem, nf * xp::kRingMaxLanes, r->cm.query)) != XP_OK) {
    common_free(r->cm);
    mem_free(r->mem);
    delete r;
    return s;
  }
  r->ctl = r->mem.dev;
  r->slots = r->mem.dev + r->ctl_region;
  *out = r;
  return XP_OK;
}

xp_status xp_ring_destroy(xp_ring* r) {
  if (!r) return XP_OK;
  cudaDeviceSynchronize();
  common_free(r->cm);
  mem_free(r->mem);
  delete r;
  return XP_OK;
}

xp_status xp_ring_set_lanes(xp_ring* r, int lanes) {
  if (!r) return fail(XP_ERR_INVALID, "ring is NULL");
  if (lanes < 0 || lanes > xp::kRingMaxLanes) return fail(XP_ERR_INVALID, "lanes %d not in [0, 8]", lanes);
  if (r->place != XP_PLACE_DEVICE && r->P * lanes > xp::kMaxCluster)
    return fail(XP_ERR_INVALID, "host-placed rings need nranks * lanes <= 16");
  r->lanes = lanes;
  return XP_OK;
}

xp_status xp_ring_allreduce_virtual(xp_ring* r, const void* const* send_bufs, void* const* recv_bufs, size_t count,
                                    xp_dtype dt, xp_stream_t stream) {
  if (!r) return fail(XP_ERR_INVALID, "ring is NULL");
  if (dt != XP_F32 && dt != XP_I32) return fail(XP_ERR_INVALID, "the ring reduces XP_F32 or XP_I32 only");
  if (count == 0) return XP_OK;
  if (!send_bufs || !recv_bufs) return fail(XP_ERR_INVALID, "buffer arrays are NULL");
  if (count > (1ull << 38)) return fail(XP_ERR_INVALID, "count too large");
  for (int i = 0; i < r->P; ++i) {
    if (!send_bufs[i] || !recv_bufs[i]) return fail(XP_ERR_INVALID, "rank %d buffer is NULL", i);
    if (!aligned16(send_bufs[i]) || !aligned16(recv_bufs[i])) return fail(XP_ERR_INVALID, "rank %d buffer not 16-byte aligned", i);
  }
  xp_status s = check_device(r->cm);
  if (s != XP_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  xp::RingParams p = {};
  p.ctl = r->ctl;
  p.slots = r->slots;
  p.fifo_stride = r->fifo_stride;
  for (int i = 0; i < r->P; ++i) {
    p.send[i] = static_cast<const char*>(send_bufs[i]);
    p.recv[i] = static_cast<char*>(recv_bufs[i]);
  }
  p.count = count;
  p.nranks = r->P;
  p.nchannels = r->C;
  p.nslots = r->N;
  // lanes 0: HBM rings run their channels in groups whose live FIFO data
  // (about half of every FIFO: a chunk is N/2 slots and each hop lags one
  // chunk) fits in kRingLiveBytes, one launch per group, each group with the
  // most lanes whose whole grid is resident at once (a cooperative launch),
  // at least one; host-placed rings take one lane and one launch.  Explicit
  // lanes run every channel in one launch.
  int lanes = r->lanes, group = r->C;
  if (lanes == 0) {
    lanes = 1;
    if (r->place == XP_PLACE_DEVICE) {
      const size_t live = (size_t)r->P * (size_t)(r->N / 2) * r->S;   // per channel
      group = (int)(kRingLiveBytes / live);
      if (group < 1) group = 1;
      if (group > r->C) group = r->C;
      const int fit = ring_tma_resident();
      while (lanes < xp::kRingMaxLanes && group * (lanes + 1) * r->P <= fit) ++lanes;
    }
  }
  p.lanes = lanes;
  p.dtype = dt;
  p.slot_bytes = (unsigned)r->S;
  p.status = r->cm.status;
  p.abort_word = g_abort_dev;
  p.timeout_ns = g_timeout_ns.load();
  p.op = ++r->cm.ops;
  if (r->place == XP_PLACE_DEVICE) {
    // HBM FIFOs: bulk copies through shared memory, every lane with its own
    // counters.  The ranks a lane's ring waits on must be resident together:
    // a cooperative grid when the whole grid fits on the GPU at once (no
    // cluster placement limits), else one cluster of P CTAs per (channel, lane).
    for (int c0 = 0; c0 < r->C && s == XP_OK; c0 += group) {
      p.c_first = c0;
      const int grid = (r->C - c0 < group ? r->C - c0 : group) * lanes * r->P;
      s = launch(xp::ring_tma_kernel_ptr(dt), grid, xp::ring_tma_threads(), grid <= ring_tma_resident() ? 0 : r->P, &p,
                 st, xp::ring_tma_smem());
    }
  } else {
    // mapped host FIFOs: 16-byte vector loads and stores from every warp; one
    // cluster of P * lanes CTAs per channel, lanes sharing the counters
    const int csize = r->P * lanes;
    s = launch(xp::ring_kernel_ptr(dt), r->C * csize, xp::kRingThreads, csize, &p, st);
  }
  if (s != XP_OK) return s;
  return record_done(r->cm, st);
}

xp_status xp_ring_status(xp_ring* r, int sync, xp_report* report) {
  if (!r) return fail(XP_ERR_INVALID, "ring is NULL");
  return read_status(r->cm, sync, report);
}

xp_status xp_ring_reset(xp_ring* r) {
  if (!r) return fail(XP_ERR_INVALID, "ring is NULL");
  if (r->cm.used) XP_CUDA(cudaEventSynchronize(r->cm.done));
  XP_CUDA(cudaMemsetAsync(r->cm.status, 0, sizeof(DevStatus), r->cm.query));
  return mem_init(r->mem, r->P * r->C * xp::kRingMaxLanes, r->cm.query);
}

}  // extern "C"
