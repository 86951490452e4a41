// Host pump of the proxy (copy-engine) mode; see xp_proxy.cu.
#pragma once

#include <cstddef>
#include <string>

#include "xp_internal.h"

namespace xp {

struct PumpConfig {
  int device = 0;
  int nchannels = 0;
  int nslots = 0;
  size_t slot_bytes = 0;
  size_t ch_stride = 0;              // bytes between channels in every ring
  int hops = 1;                      // copies per slot-step (1 or 2)
  char* ce_host = nullptr;           // host view of the nchannels proxy-mode blocks
  char* rings[kCeMaxHops + 1] = {};  // ring h, channel c at rings[h] + c * ch_stride
};

struct Pump;

// Starts the pump thread; nullptr (and *err) on failure.
Pump* pump_start(const PumpConfig& cfg, std::string* err);
// Stops and joins the thread, waits for its copies, frees it.  NULL-safe.
void pump_stop(Pump* p);
// Asks the pump to spin (not sleep) for the next few milliseconds.
void pump_kick(Pump* p);
// The error that stopped the pump, or nullptr.
const char* pump_error(const Pump* p);

}  // namespace xp
