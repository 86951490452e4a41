// xp_send_recv_noalloc: a SIMPLE transfer whose FIFO lives in a fixed
// device array that this library owns, so the call allocates nothing.
//
// Who needs it: callers that must not allocate device memory while they run,
// such as code inside a memory pool or allocator hook (a cudaMalloc there can
// recurse into the allocator), code that runs under a strict device-memory
// budget, or code that must never block on the driver's allocation lock.
// They still allocate their own src and dst; the FIFO (control blocks, slots
// and status) comes from kNoallocBytes of device memory that every GPU which
// loads this library reserves until the process exits.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "xp_internal.h"

namespace xp {
void set_last_error(const char* msg);
void* p2p_tma_kernel_ptr(int mode);
int p2p_tma_threads();
int p2p_tma_smem();
}  // namespace xp

namespace {

constexpr int kNoallocMaxChannels = 16;
constexpr size_t kNoallocSlotBytes = 8u << 20;   // every channel's slots together
constexpr size_t kNoallocStatusOff = 0;
constexpr size_t kNoallocCtlOff = 256;
constexpr size_t kNoallocArrOff = kNoallocCtlOff + (size_t)kNoallocMaxChannels * xp::kCtlBytes;
constexpr size_t kNoallocSlotsOff = kNoallocArrOff + (size_t)kNoallocMaxChannels * xp::kArrBytes;
constexpr size_t kNoallocBytes = kNoallocSlotsOff + kNoallocSlotBytes;
constexpr unsigned long long kNoallocTimeoutNs = 2000000000ull;

// The scratch memory: status block, control blocks, slots.  In host code
// this name is a host-side stand-in; its device address comes from
// cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

std::mutex g_noalloc_mu;
bool g_noalloc_ready[64] = {};   // per device: the kernel's shared-memory attribute is set

size_t round_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

xp_status invalid(const char* msg) {
  xp::set_last_error(msg);
  return XP_ERR_INVALID;
}
xp_status cuda_failed(const char* what, cudaError_t e) {
  static thread_local char buf[256];
  snprintf(buf, sizeof buf, "xp_send_recv_noalloc: %s: %s", what, cudaGetErrorString(e));
  xp::set_last_error(buf);
  return XP_ERR_CUDA;
}

}  // namespace

extern "C" xp_status xp_send_recv_noalloc(const void* src, void* dst, size_t bytes, int nchannels, int nslots,
                                          size_t slot_bytes, int32_t* dev_status, xp_stream_t stream) {
  if (nchannels < 1 || nchannels > kNoallocMaxChannels)
    return invalid("xp_send_recv_noalloc: nchannels must be in [1, 16]");
  if (nslots < 1 || nslots > xp::kMaxSlots) return invalid("xp_send_recv_noalloc: nslots must be in [1, 64]");
  if (slot_bytes == 0 || slot_bytes % 16 || slot_bytes > (1ull << 31))
    return invalid("xp_send_recv_noalloc: slot_bytes must be a non-zero multiple of 16");
  const size_t ch_stride = round_up((size_t)nslots * slot_bytes, 4096);
  if ((size_t)nchannels * ch_stride > kNoallocSlotBytes)
    return invalid("xp_send_recv_noalloc: nchannels x round_up(nslots x slot_bytes, 4096) exceeds the 8 MiB "
                   "static FIFO; use fewer or smaller slots, or xp_fifo_create + xp_send_recv");
  if (bytes == 0) return XP_OK;
  if (!src || !dst) return invalid("xp_send_recv_noalloc: src or dst is NULL");
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u)
    return invalid("xp_send_recv_noalloc: src and dst must be 16-byte aligned");
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
  if (s0 < d0 + bytes && d0 < s0 + bytes) return invalid("xp_send_recv_noalloc: src and dst overlap");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_failed("cudaGetDevice", e);
  if (dev < 0 || dev >= 64) return invalid("xp_send_recv_noalloc: device index above 63");
  // The array's device address, looked up on every call with this device
  // current (the lookup allocates nothing, and a context created anew, say
  // after cudaDeviceReset, maps the array at a new address).
  void* ptr = nullptr;
  if ((e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch)) != cudaSuccess) return cuda_failed("cudaGetSymbolAddress", e);
  if (!ptr) return invalid("xp_send_recv_noalloc: no device address for the static FIFO");
  unsigned char* base = static_cast<unsigned char*>(ptr);
  {
    // once per device: let the kernel use its dynamic shared memory
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ready[dev]) {
      const void* kern = xp::p2p_tma_kernel_ptr(0);
      if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, xp::p2p_tma_smem())) != cudaSuccess)
        return cuda_failed("cudaFuncSetAttribute", e);
      g_noalloc_ready[dev] = true;
    }
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  xp::DevStatus* status = reinterpret_cast<xp::DevStatus*>(base + kNoallocStatusOff);
  // status, counters, ptrExchange, step base and lane arrival counters start
  // at zero on every call
  if ((e = cudaMemsetAsync(base, 0, kNoallocSlotsOff, st)) != cudaSuccess) return cuda_failed("cudaMemsetAsync", e);

  xp::P2pParams p = {};
  p.ctl = reinterpret_cast<char*>(base + kNoallocCtlOff);
  p.discard = 1;
  p.arr = reinterpret_cast<unsigned long long*>(base + kNoallocArrOff);
  p.slots = reinterpret_cast<char*>(base + kNoallocSlotsOff);
  p.ch_stride = ch_stride;
  p.src = static_cast<const char*>(src);
  p.dst = static_cast<char*>(dst);
  p.nbytes = bytes;
  p.nchannels = nchannels;
  p.nslots = nslots;
  p.lanes = 1;
  p.rlanes = 1;
  p.csize = 2;
  p.slot_bytes = (unsigned)slot_bytes;
  p.status = status;
  p.abort_word = nullptr;
  p.timeout_ns = kNoallocTimeoutNs;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * nchannels, 1, 1);
  cfg.blockDim = dim3(xp::p2p_tma_threads(), 1, 1);
  cfg.dynamicSmemBytes = (size_t)xp::p2p_tma_smem();
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  void* args[] = {&p};
  if ((e = cudaLaunchKernelExC(&cfg, xp::p2p_tma_kernel_ptr(0), args)) != cudaSuccess)
    return cuda_failed("cudaLaunchKernelExC", e);
  // the claim word's low half is the failure code (the operation id, in the
  // high half, is 0 here: the status block starts at zero on every call)
  if (dev_status &&
      (e = cudaMemcpyAsync(dev_status, &status->claim, sizeof(int32_t), cudaMemcpyDeviceToDevice, st)) != cudaSuccess)
    return cuda_failed("cudaMemcpyAsync", e);
  return XP_OK;
}
