// Bounded device-side waits shared by the kernels.  Every wait gives up
// after kWaitNs of %globaltimer, sets the workspace status word to
// "timeout" and raises the CTA's abort flag; the caller then stops taking
// work, lets its own copies drain and returns, so the context stays usable
// and snapkv_get_status reports the timeout.
#pragma once
#include <cstdint>

#include "plan.h"

namespace snapkv {
namespace tc {

constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

struct Ctl {
  volatile int* abort;  // CTA-wide abort flag (shared memory)
  int* status;          // device status word
};

__device__ __forceinline__ void raise_timeout(const Ctl& c) {
  *c.abort = 1;
  atomicExch(c.status, kDevTimeout);
}

// Bounded wait until *ctr >= target (device-scope acquire).
__device__ __forceinline__ bool wait_counter(const int* ctr, int target, const Ctl& c) {
  const uint64_t t0 = global_ns();
  for (;;) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    if (*c.abort) return false;
    if (global_ns() - t0 > kWaitNs) {
      raise_timeout(c);
      return false;
    }
    __nanosleep(128);
  }
}

}  // namespace tc
}  // namespace snapkv
