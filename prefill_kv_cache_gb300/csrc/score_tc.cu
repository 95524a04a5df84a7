// Tensor-core (tcgen05 / TMA) observation-window score kernel.  Placeholder
// that declines every problem until the kernel lands; the caller then runs
// the CUDA-core path.
#include <cuda_runtime.h>

#include "plan.h"

namespace snapkv {

int launch_score_tc(const Plan&, void*, bool* taken) {
  *taken = false;
  return cudaSuccess;
}

}  // namespace snapkv
