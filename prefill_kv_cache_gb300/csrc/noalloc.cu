// snapkv_compress_noalloc: the compression with library-owned scratch.
//
// Some callers cannot call cudaMalloc: a plugin running inside a serving
// engine that owns all device memory through its own pool and hands plugins
// no allocator, or a latency-critical path where cudaMalloc's implicit
// device-wide synchronisation is not acceptable.  For them this entry point
// takes its workspace from a fixed array that lives in the library's device
// image instead of from the caller.  It is the same compression as
// snapkv_compress (same kernels, same results); only where the scratch comes
// from differs.
#include <cuda_runtime.h>

#include "snapkv.h"

namespace snapkv {
namespace {

// Largest workspace this entry point can serve.  Every GPU that loads the
// library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_scratch[kNoAllocScratchBytes];

// Device address of g_scratch in the calling thread's current context.  In
// host code the array's name is only a stand-in for the symbol, never a
// device address.  Each CUDA context has its own copy of the array, so the
// address is looked up on every call rather than cached: a cached value would
// go stale after cudaDeviceReset or point into another context when the
// caller switches contexts.  The lookup allocates nothing; the first one in a
// context may load the library's device code.
cudaError_t scratch_in_current_context(void** out) {
  return cudaGetSymbolAddress(out, g_scratch);
}

}  // namespace
}  // namespace snapkv

extern "C" int snapkv_compress_noalloc(const snapkv_shape* shape, const void* q_win,
                                       const void* k, const void* v,
                                       const int32_t* seqlens_host, int32_t W,
                                       int32_t kernel_size, int32_t pool_type, int32_t C,
                                       void* out_k, void* out_v, int32_t* out_idx,
                                       void* stream) {
  using namespace snapkv;
  const size_t need = snapkv_workspace_size(shape, seqlens_host, W, C);
  if (need == 0) {  // invalid or unsupported problem: report which
    size_t a = 0, b = 0, c = 0;
    const int rc = snapkv_score_offsets(shape, seqlens_host, W, C, &a, &b, &c);
    return rc != SNAPKV_OK ? rc : SNAPKV_ERR_INVALID_ARG;
  }
  if (need > kNoAllocScratchBytes) return SNAPKV_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_in_current_context(&scratch) != cudaSuccess) return SNAPKV_ERR_CUDA;
  // The status word and the work-queue counters at the start of the scratch
  // are cleared on the stream by snapkv_compress; every other region is fully
  // written before it is read, so the previous call's contents do not matter.
  return snapkv_compress(shape, q_win, k, v, seqlens_host, W, kernel_size, pool_type, C, out_k,
                         out_v, out_idx, scratch, kNoAllocScratchBytes, stream);
}

extern "C" int snapkv_noalloc_get_status(void* stream) {
  using namespace snapkv;
  // the status word sits at the start of the scratch, where the workspace
  // layout puts it
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SNAPKV_ERR_CUDA;
  int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_scratch, sizeof(int), 0, cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return SNAPKV_ERR_CUDA;
  return word == 0 ? SNAPKV_OK : SNAPKV_ERR_TIMEOUT;
}
