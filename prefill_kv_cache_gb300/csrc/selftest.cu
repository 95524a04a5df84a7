// Self-test of the bounded-wait mechanism that every cross-CTA wait in the
// kernels uses (wait.cuh): one thread waits on a device flag with the same
// wait_counter the score kernel uses for its queue counters.  With
// set_flag = 0 nothing ever sets the flag, the wait runs out after its limit,
// the status word becomes "timeout" and the kernel returns normally, so the
// context stays usable; with set_flag = 1 the kernel sets the flag first and
// the wait succeeds.  No counterpart on the SnapKV pages: it exists so the
// failure path can be tested without faulting or hanging a GPU.
#include <cuda_runtime.h>

#include "plan.h"
#include "snapkv.h"
#include "wait.cuh"

namespace snapkv {

__global__ void selftest_wait_kernel(int* status, int* flag, int set_flag) {
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  if (set_flag) atomicExch(flag, 1);
  const tc::Ctl ctl{&abort_flag, status};
  tc::wait_counter(flag, 1, ctl);
}

}  // namespace snapkv

int snapkv_selftest_wait(void* workspace, size_t workspace_bytes, int32_t set_flag, void* stream) {
  if (!workspace || workspace_bytes < 512 || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return SNAPKV_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  if (cudaMemsetAsync(ws, 0, 512, st) != cudaSuccess) return SNAPKV_ERR_CUDA;  // status, flag
  snapkv::selftest_wait_kernel<<<1, 32, 0, st>>>(reinterpret_cast<int*>(ws),
                                                 reinterpret_cast<int*>(ws + 256), set_flag ? 1 : 0);
  if (cudaGetLastError() != cudaSuccess) return SNAPKV_ERR_CUDA;
  snapkv::count_launches(1);
  return SNAPKV_OK;
}
