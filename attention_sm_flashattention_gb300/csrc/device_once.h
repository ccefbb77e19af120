// Per-device "done once" flags for host-side set-up such as kernel function
// attributes.  cudaFuncSetAttribute applies to the device that is current when
// it is called, so a launcher that raises a kernel's shared-memory limit must
// do so once on every device it launches on, not once per process.
//
// Host-only and free of CUDA types, so that the bookkeeping can be built and
// tested without a GPU.
#pragma once

#include <atomic>

namespace fa {

constexpr int kMaxFlagDevices = 64;

// One flag per device index; a zero-initialised static array of these starts
// with every device "not done".
using DeviceOnceFlags = std::atomic<bool>[kMaxFlagDevices];

// Runs `setup()` for device `dev` unless an earlier call for that device
// succeeded.  `setup` returns 0 on success; on failure the flag stays clear,
// so the next call retries.  Two host threads racing on the same device may
// both run `setup` (it must be idempotent); neither sees a flag set before
// its set-up finished.  Returns 0, the failing set-up's code, or -1 for a
// device index outside [0, kMaxFlagDevices).
template <typename F>
int once_per_device(DeviceOnceFlags& flags, int dev, F&& setup) {
  if (dev < 0 || dev >= kMaxFlagDevices) return -1;
  if (flags[dev].load(std::memory_order_acquire)) return 0;
  const int rc = setup();
  if (rc != 0) return rc;
  flags[dev].store(true, std::memory_order_release);
  return 0;
}

}  // namespace fa
