// C ABI of libsnapkv: argument checks, workspace layout, launch planning.
//
// Every entry point is declared, with its contract, in include/snapkv.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "plan.h"
#include "snapkv.h"

namespace snapkv {

// counter_off: next unused int of the call's zeroed counter region (in/out)
int launch_score_tc(const Plan& p, void* stream, bool* taken, int* counter_off);

static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

static std::atomic<uint64_t> g_score_launches[2];
void count_score_launches(int path, int n) {
  g_score_launches[path].fetch_add((uint64_t)n, std::memory_order_relaxed);
}

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
DeviceInfo g_dev_info[kMaxDevices];
bool g_dev_known[kMaxDevices] = {};
}  // namespace

const DeviceInfo* current_device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (!g_dev_known[dev]) {
    DeviceInfo d{};
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        d.sms <= 0 || d.smem_optin <= 0)
      return nullptr;
    g_dev_info[dev] = d;
    g_dev_known[dev] = true;
  }
  return &g_dev_info[dev];
}

namespace {

constexpr size_t kAlign = 256;
constexpr int kChunkKeys = 1024;    // keys per score piece, at most
constexpr int kMinChunkKeys = 256;  // and at least
constexpr int kTargetPieces = 4 * 152;  // pieces per pass a call aims for

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  size_t status = 0;  // int status word
  size_t counters = 0;  // kCounterInts ints
  size_t raw = 0, pooled = 0, stats = 0, lse = 0;
  size_t score_count = 0;  // floats in raw (and in pooled)
  size_t total = 0;
};

// Checks shared by every entry point; SNAPKV_OK when the problem is valid
// and supported.
int check_problem(const snapkv_shape* sh, const int32_t* seqlens, int W, int C) {
  if (!sh || !seqlens) return SNAPKV_ERR_INVALID_ARG;
  if (sh->batch < 1 || sh->batch > kMaxBatch) return SNAPKV_ERR_INVALID_ARG;
  if (sh->num_q_heads < 1 || sh->num_kv_heads < 1) return SNAPKV_ERR_INVALID_ARG;
  if (sh->num_q_heads % sh->num_kv_heads) return SNAPKV_ERR_INVALID_ARG;
  if (sh->dtype != SNAPKV_BF16 && sh->dtype != SNAPKV_FP32) return SNAPKV_ERR_INVALID_ARG;
  if (W < 1 || C < W) return SNAPKV_ERR_INVALID_ARG;
  for (int b = 0; b < sh->batch; ++b)
    if (seqlens[b] < 1) return SNAPKV_ERR_INVALID_ARG;
  if (sh->head_dim != 64 && sh->head_dim != 128) return SNAPKV_ERR_UNSUPPORTED;
  const long long Wp = (long long)W * (sh->num_q_heads / sh->num_kv_heads);
  if (Wp > kMaxRows) return SNAPKV_ERR_UNSUPPORTED;
  return SNAPKV_OK;
}

// Flags of the _ex entry points: known bits only; per-query-head selection
// needs groups of at most 8 query heads.
int check_flags(const snapkv_shape* sh, int32_t flags) {
  if (!sh) return SNAPKV_ERR_INVALID_ARG;
  if (flags & ~SNAPKV_PER_QUERY_HEAD) return SNAPKV_ERR_INVALID_ARG;
  if ((flags & SNAPKV_PER_QUERY_HEAD) && sh->num_kv_heads > 0 &&
      sh->num_q_heads / sh->num_kv_heads > 8)
    return SNAPKV_ERR_UNSUPPORTED;
  return SNAPKV_OK;
}

// Keys per score piece (the unit of work of both scoring paths): 1024 for
// the tensor-core kernel; for the CUDA-core kernels, whose blocks each take
// one piece, less when the call has too few pieces to give every SM of a
// GB300 (152) several of them, so that short prompts still spread over the
// GPU.  A function of the problem only, so that the workspace size and the
// launch agree.
int chunk_keys_for(const snapkv_shape* sh, const int32_t* seqlens, int W, int C) {
  int ck = kChunkKeys;
  const int Wp = W * (sh->num_q_heads / sh->num_kv_heads);
  if (sh->dtype == SNAPKV_BF16 && (sh->head_dim == 64 || sh->head_dim == 128) &&
      (Wp == 128 || Wp == 256))
    return ck;
  for (; ck > kMinChunkKeys; ck /= 2) {
    long long pieces = 0;
    for (int b = 0; b < sh->batch; ++b)
      if (seqlens[b] > C) pieces += (long long)sh->num_kv_heads * ((seqlens[b] + ck - 1) / ck);
    if (pieces >= kTargetPieces) break;
  }
  return ck;
}

int chunks_for(int L, int ck) { return (L + ck - 1) / ck; }

Layout layout_for(const snapkv_shape* sh, const int32_t* seqlens, int W, int C,
                  bool per_q = false) {
  Layout lay;
  const int H = sh->num_kv_heads;
  const int Wp = W * (sh->num_q_heads / H);
  size_t scores = 0, max_pieces = 0, max_units = 0;
  const int ck = chunk_keys_for(sh, seqlens, W, C);
  for (int g0 = 0; g0 < sh->batch; g0 += kGroupSeqs) {
    const int g1 = std::min(sh->batch, g0 + kGroupSeqs);
    size_t pieces = 0;
    for (int b = g0; b < g1; ++b) {
      if (seqlens[b] > C) {
        scores += (size_t)(per_q ? sh->num_q_heads : H) * (seqlens[b] - W);
        pieces += (size_t)H * chunks_for(seqlens[b], ck);
      }
    }
    max_pieces = std::max(max_pieces, pieces);
    max_units = std::max(max_units, (size_t)(g1 - g0) * H);
  }
  size_t off = 0;
  lay.status = off;
  off += kAlign;
  lay.counters = off;
  off = align_up(off + kCounterInts * sizeof(int));
  lay.raw = off;
  off = align_up(off + scores * sizeof(float));
  lay.pooled = off;
  off = align_up(off + scores * sizeof(float));
  // 512 partial (max, sum) statistics per piece: the tensor-core kernel's
  // consumer groups publish theirs separately (2 per row at W * g = 256, 4 at
  // 128); the CUDA-core kernels use one per row (W * g <= 256 of them)
  lay.stats = off;
  off = align_up(off + max_pieces * 512 * sizeof(float2));
  lay.lse = off;
  off = align_up(off + max_units * Wp * sizeof(float));
  lay.score_count = scores;
  lay.total = off;
  return lay;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace snapkv

using namespace snapkv;

extern "C" {

const char* snapkv_status_string(int status) {
  switch (status) {
    case SNAPKV_OK: return "ok";
    case SNAPKV_ERR_INVALID_ARG: return "invalid argument";
    case SNAPKV_ERR_UNSUPPORTED: return "unsupported shape or type";
    case SNAPKV_ERR_WORKSPACE: return "workspace too small";
    case SNAPKV_ERR_CUDA: return "CUDA error";
    case SNAPKV_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

int snapkv_version(void) { return 0x000401; }

size_t snapkv_workspace_size(const snapkv_shape* shape, const int32_t* seqlens_host, int32_t W,
                             int32_t C) {
  if (check_problem(shape, seqlens_host, W, C) != SNAPKV_OK) return 0;
  return layout_for(shape, seqlens_host, W, C).total;
}

size_t snapkv_workspace_size_ex(const snapkv_shape* shape, const int32_t* seqlens_host,
                                int32_t W, int32_t C, int32_t flags) {
  if (check_flags(shape, flags) != SNAPKV_OK) return 0;
  if (check_problem(shape, seqlens_host, W, C) != SNAPKV_OK) return 0;
  return layout_for(shape, seqlens_host, W, C, flags & SNAPKV_PER_QUERY_HEAD).total;
}

int snapkv_score_offsets(const snapkv_shape* shape, const int32_t* seqlens_host, int32_t W,
                         int32_t C, size_t* raw_offset, size_t* pooled_offset, size_t* count) {
  return snapkv_score_offsets_ex(shape, seqlens_host, W, C, 0, raw_offset, pooled_offset, count);
}

int snapkv_score_offsets_ex(const snapkv_shape* shape, const int32_t* seqlens_host, int32_t W,
                            int32_t C, int32_t flags, size_t* raw_offset, size_t* pooled_offset,
                            size_t* count) {
  int rc = check_flags(shape, flags);
  if (rc != SNAPKV_OK) return rc;
  rc = check_problem(shape, seqlens_host, W, C);
  if (rc != SNAPKV_OK) return rc;
  if (!raw_offset || !pooled_offset || !count) return SNAPKV_ERR_INVALID_ARG;
  const Layout lay = layout_for(shape, seqlens_host, W, C, flags & SNAPKV_PER_QUERY_HEAD);
  *raw_offset = lay.raw;
  *pooled_offset = lay.pooled;
  *count = lay.score_count;
  return SNAPKV_OK;
}

namespace {

// Shared by snapkv_compress (score_only = false) and snapkv_score.
int enqueue(const snapkv_shape* shape, const void* q_win, const void* k, const void* v,
            const int32_t* seqlens_host, int32_t W, int32_t kernel_size, int32_t pool_type,
            int32_t C, void* out_k, void* out_v, int32_t* out_idx, void* workspace,
            size_t workspace_bytes, void* stream, bool score_only, const float* lse_in,
            bool per_q = false, const void* q_all = nullptr, const float* lse_all = nullptr,
            bool v_zero_copy = false, int* status_word = nullptr, int gpu_share = 1) {
  int rc = check_problem(shape, seqlens_host, W, C);
  if (rc == SNAPKV_ERR_INVALID_ARG) return rc;
  if (!q_win || !k || !workspace) return SNAPKV_ERR_INVALID_ARG;
  if (!aligned(q_win, 16) || !aligned(k, 16) || !aligned(workspace, kAlign))
    return SNAPKV_ERR_INVALID_ARG;
  if (!score_only) {
    if (!v || !out_k || !out_v || !out_idx) return SNAPKV_ERR_INVALID_ARG;
    if (kernel_size < 1 || kernel_size % 2 == 0) return SNAPKV_ERR_INVALID_ARG;
    if (pool_type != SNAPKV_POOL_AVG && pool_type != SNAPKV_POOL_MAX)
      return SNAPKV_ERR_INVALID_ARG;
    if (!aligned(v, 16) || !aligned(out_k, 16) || !aligned(out_v, 16) || !aligned(out_idx, 16))
      return SNAPKV_ERR_INVALID_ARG;
  }
  if (rc != SNAPKV_OK) return rc;
  const Layout lay = layout_for(shape, seqlens_host, W, C, per_q);
  if (workspace_bytes < lay.total) return SNAPKV_ERR_WORKSPACE;

  char* ws = static_cast<char*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // one memset per call: the status word and the work-queue counters, which
  // sit together at the start of the workspace (the counters alone when the
  // caller keeps a status word of its own across several calls)
  static_assert(sizeof(int) * kCounterInts % 4 == 0, "counter region");
  const size_t clear0 = status_word ? lay.counters : lay.status;
  if (cudaMemsetAsync(ws + clear0, 0, lay.counters + sizeof(int) * kCounterInts - clear0, st) !=
      cudaSuccess)
    return SNAPKV_ERR_CUDA;
  int counter_off = 0;

  const int H = shape->num_kv_heads;
  Plan p;
  std::memset(&p, 0, sizeof p);
  p.H_q = shape->num_q_heads;
  p.H_kv = H;
  p.g = p.H_q / H;
  p.d = shape->head_dim;
  p.W = W;
  p.Wp = W * p.g;
  p.C = C;
  p.n = C - W;
  p.kp = kernel_size;
  p.pool = pool_type;
  p.dtype = shape->dtype;
  p.scale = (float)(1.0 / std::sqrt((double)p.d));
  p.log2e_scale = (float)(1.4426950408889634 / std::sqrt((double)p.d));
  p.chunk_keys = chunk_keys_for(shape, seqlens_host, W, C);
  p.q = q_win;
  p.k = k;
  p.v = v;
  p.out_k = out_k;
  p.out_v = out_v;
  p.out_idx = out_idx;
  p.raw = reinterpret_cast<float*>(ws + lay.raw);
  p.pooled = reinterpret_cast<float*>(ws + lay.pooled);
  p.stats = reinterpret_cast<float2*>(ws + lay.stats);
  p.lse = reinterpret_cast<float*>(ws + lay.lse);
  p.lse_in = lse_in;
  p.q_all = q_all;
  p.lse_all = lse_all;
  p.v_zero_copy = v_zero_copy ? 1 : 0;
  p.gpu_share = gpu_share;
  p.out_heads = per_q ? p.H_q : H;
  p.head_div = per_q ? p.g : 1;
  p.status = status_word ? status_word : reinterpret_cast<int*>(ws + lay.status);
  p.counters = reinterpret_cast<int*>(ws + lay.counters);
  p.batch = shape->batch;
  p.total_rows = 0;
  for (int b = 0; b < shape->batch; ++b) p.total_rows += seqlens_host[b];

  long long row0 = 0, score0 = 0;
  for (int g0 = 0; g0 < shape->batch; g0 += kGroupSeqs) {
    const int g1 = std::min(shape->batch, g0 + kGroupSeqs);
    p.nseq = g1 - g0;
    int piece = 0;
    for (int b = g0; b < g1; ++b) {
      SeqInfo& S = p.seq[b - g0];
      S.b = b;
      S.L = seqlens_host[b];
      S.P = S.L - W;
      S.scored = S.L > C;
      S.row0 = row0;
      S.score0 = score0;
      S.piece0 = piece;
      S.chunks = S.scored ? chunks_for(S.L, p.chunk_keys) : 0;
      piece += S.chunks * H;
      if (S.scored) score0 += (long long)p.out_heads * S.P;
      row0 += S.L;
    }
    p.total_pieces = piece;
    if (piece > 0 && q_all) {
      if (launch_score_allq(p, stream) != cudaSuccess) return SNAPKV_ERR_CUDA;
    } else if (piece > 0) {
      bool taken = false;
      if (launch_score_tc(p, stream, &taken, &counter_off) != cudaSuccess) return SNAPKV_ERR_CUDA;
      if (!taken && launch_score_simt(p, stream) != cudaSuccess) return SNAPKV_ERR_CUDA;
    }
    if (!score_only && launch_select_gather(p, stream) != cudaSuccess) return SNAPKV_ERR_CUDA;
  }
  return SNAPKV_OK;
}

}  // namespace

int snapkv_compress(const snapkv_shape* shape, const void* q_win, const void* k, const void* v,
                    const int32_t* seqlens_host, int32_t W, int32_t kernel_size,
                    int32_t pool_type, int32_t C, void* out_k, void* out_v, int32_t* out_idx,
                    void* workspace, size_t workspace_bytes, void* stream) {
  return enqueue(shape, q_win, k, v, seqlens_host, W, kernel_size, pool_type, C, out_k, out_v,
                 out_idx, workspace, workspace_bytes, stream, false, nullptr);
}

size_t snapkv_workspace_size_layers(const snapkv_shape* shape, const int32_t* seqlens_host,
                                    int32_t W, int32_t C, int32_t n_streams) {
  if (check_problem(shape, seqlens_host, W, C) != SNAPKV_OK) return 0;
  if (n_streams < 1 || n_streams > SNAPKV_MAX_LAYER_STREAMS) return 0;
  return (size_t)n_streams * align_up(layout_for(shape, seqlens_host, W, C).total);
}

int snapkv_compress_layers(const snapkv_shape* shape, int32_t n_layers,
                           const void* const* q_win, const void* const* k, const void* const* v,
                           const float* const* lse_win, const int32_t* seqlens_host, int32_t W,
                           int32_t kernel_size, int32_t pool_type, int32_t C,
                           void* const* out_k, void* const* out_v,
                           int32_t* const* out_idx, void* workspace, size_t workspace_bytes,
                           void* stream, int32_t n_streams, void* const* layer_streams,
                           void* const* events) {
  int rc = check_problem(shape, seqlens_host, W, C);
  if (rc != SNAPKV_OK) return rc;
  if (n_layers < 1 || !q_win || !k || !v || !out_k || !out_v || !out_idx || !workspace ||
      !aligned(workspace, kAlign) || n_streams < 1 || n_streams > SNAPKV_MAX_LAYER_STREAMS ||
      !layer_streams || !events)
    return SNAPKV_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l)
    if (!q_win[l] || !k[l] || !v[l] || !out_k[l] || !out_v[l] || !out_idx[l] ||
        (lse_win && (!lse_win[l] || !aligned(lse_win[l], 4))))
      return SNAPKV_ERR_INVALID_ARG;
  for (int i = 0; i < n_streams; ++i) {
    if (!layer_streams[i]) return SNAPKV_ERR_INVALID_ARG;
    for (int j = 0; j < i; ++j)
      if (layer_streams[i] == layer_streams[j]) return SNAPKV_ERR_INVALID_ARG;
  }
  for (int e = 0; e <= n_streams; ++e)
    if (!events[e]) return SNAPKV_ERR_INVALID_ARG;
  const size_t part = align_up(layout_for(shape, seqlens_host, W, C).total);
  if (workspace_bytes < (size_t)n_streams * part) return SNAPKV_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaEvent_t fork = static_cast<cudaEvent_t>(events[0]);
  char* ws = static_cast<char*>(workspace);
  int* status = reinterpret_cast<int*>(ws);  // the first part's status word serves the call
  // clear it, then fork the layer streams off the caller's stream
  if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess ||
      cudaEventRecord(fork, st) != cudaSuccess)
    return SNAPKV_ERR_CUDA;
  for (int i = 0; i < n_streams; ++i)
    if (cudaStreamWaitEvent(static_cast<cudaStream_t>(layer_streams[i]), fork, 0) != cudaSuccess)
      return SNAPKV_ERR_CUDA;
  // layer l runs on stream l % n_streams in workspace part l % n_streams: a
  // layer's selection overlaps the next layers' scoring on the other streams,
  // and each layer's score kernel takes 1/n_streams of the SMs, so that the
  // layers' latency-bound pass-1 -> merge -> pass-2 chains run side by side
  const int share = std::min<int>(n_streams, n_layers);  // launches that can run side by side
  int first_err = SNAPKV_OK;
  for (int l = 0; l < n_layers && first_err == SNAPKV_OK; ++l) {
    const int h = l % n_streams;
    first_err = enqueue(shape, q_win[l], k[l], v[l], seqlens_host, W, kernel_size, pool_type, C,
                        out_k[l], out_v[l], out_idx[l], ws + h * part, part, layer_streams[h],
                        false, lse_win ? lse_win[l] : nullptr, false, nullptr, nullptr, false,
                        status, share);
  }
  // join, whatever happened above: the caller's stream waits for every one
  for (int i = 0; i < n_streams; ++i) {
    cudaEvent_t join = static_cast<cudaEvent_t>(events[1 + i]);
    if (cudaEventRecord(join, static_cast<cudaStream_t>(layer_streams[i])) != cudaSuccess ||
        cudaStreamWaitEvent(st, join, 0) != cudaSuccess)
      return SNAPKV_ERR_CUDA;
  }
  return first_err;
}

int snapkv_score(const snapkv_shape* shape, const void* q_win, const void* k,
                 const int32_t* seqlens_host, int32_t W, int32_t C, void* workspace,
                 size_t workspace_bytes, void* stream) {
  return enqueue(shape, q_win, k, nullptr, seqlens_host, W, 1, SNAPKV_POOL_AVG, C, nullptr,
                 nullptr, nullptr, workspace, workspace_bytes, stream, true, nullptr);
}

int snapkv_compress_ex(const snapkv_shape* shape, const void* q_win, const void* k, const void* v,
                       const int32_t* seqlens_host, int32_t W, int32_t kernel_size,
                       int32_t pool_type, int32_t C, void* out_k, void* out_v, int32_t* out_idx,
                       void* workspace, size_t workspace_bytes, void* stream, int32_t flags) {
  const int rc = check_flags(shape, flags);
  if (rc != SNAPKV_OK) return rc;
  return enqueue(shape, q_win, k, v, seqlens_host, W, kernel_size, pool_type, C, out_k, out_v,
                 out_idx, workspace, workspace_bytes, stream, false, nullptr,
                 (flags & SNAPKV_PER_QUERY_HEAD) != 0);
}

int snapkv_compress_all_queries(const snapkv_shape* shape, const void* q_all, const void* k,
                                const void* v, const float* lse_all,
                                const int32_t* seqlens_host, int32_t W, int32_t kernel_size,
                                int32_t pool_type, int32_t C, void* out_k, void* out_v,
                                int32_t* out_idx, void* workspace, size_t workspace_bytes,
                                void* stream) {
  if (!q_all || !lse_all || !aligned(q_all, 16) || !aligned(lse_all, 4))
    return SNAPKV_ERR_INVALID_ARG;
  // q_all stands in for q_win in the argument checks; only q_all is read
  return enqueue(shape, q_all, k, v, seqlens_host, W, kernel_size, pool_type, C, out_k, out_v,
                 out_idx, workspace, workspace_bytes, stream, false, nullptr, false, q_all,
                 lse_all);
}

int snapkv_compress_with_lse(const snapkv_shape* shape, const void* q_win, const void* k,
                             const void* v, const float* lse_win, const int32_t* seqlens_host,
                             int32_t W, int32_t kernel_size, int32_t pool_type, int32_t C,
                             void* out_k, void* out_v, int32_t* out_idx, void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (!lse_win || !aligned(lse_win, 4)) return SNAPKV_ERR_INVALID_ARG;
  return enqueue(shape, q_win, k, v, seqlens_host, W, kernel_size, pool_type, C, out_k, out_v,
                 out_idx, workspace, workspace_bytes, stream, false, lse_win);
}

int snapkv_score_with_lse(const snapkv_shape* shape, const void* q_win, const void* k,
                          const float* lse_win, const int32_t* seqlens_host, int32_t W, int32_t C,
                          void* workspace, size_t workspace_bytes, void* stream) {
  if (!lse_win || !aligned(lse_win, 4)) return SNAPKV_ERR_INVALID_ARG;
  return enqueue(shape, q_win, k, nullptr, seqlens_host, W, 1, SNAPKV_POOL_AVG, C, nullptr,
                 nullptr, nullptr, workspace, workspace_bytes, stream, true, lse_win);
}

uint64_t snapkv_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

uint64_t snapkv_score_path_launches(int32_t path) {
  if (path != SNAPKV_SCORE_PATH_TENSOR_CORES && path != SNAPKV_SCORE_PATH_CUDA_CORES) return 0;
  return g_score_launches[path].load(std::memory_order_relaxed);
}

int snapkv_get_status(const void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < sizeof(int)) return SNAPKV_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return SNAPKV_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SNAPKV_ERR_CUDA;
  return word == kDevOk ? SNAPKV_OK : SNAPKV_ERR_TIMEOUT;
}

// Host-buffer variant: staging holds q, k, v, out_k, out_v, out_idx, workspace.
namespace {
struct HostLayout {
  size_t q, k, v, ok, ov, oi, ws, ws_bytes, total;
  size_t q_bytes, kv_bytes, out_bytes, idx_bytes;
};

HostLayout host_layout(const snapkv_shape* sh, const int32_t* seqlens, int W, int C) {
  HostLayout h{};
  const size_t esz = sh->dtype == SNAPKV_BF16 ? 2 : 4;
  long long T = 0;
  for (int b = 0; b < sh->batch; ++b) T += seqlens[b];
  h.q_bytes = (size_t)sh->batch * W * sh->num_q_heads * sh->head_dim * esz;
  h.kv_bytes = (size_t)T * sh->num_kv_heads * sh->head_dim * esz;
  h.out_bytes = (size_t)sh->batch * C * sh->num_kv_heads * sh->head_dim * esz;
  h.idx_bytes = (size_t)sh->batch * sh->num_kv_heads * C * sizeof(int32_t);
  size_t off = 0;
  h.q = off; off = align_up(off + h.q_bytes);
  h.k = off; off = align_up(off + h.kv_bytes);
  h.v = off; off = align_up(off + h.kv_bytes);
  h.ok = off; off = align_up(off + h.out_bytes);
  h.ov = off; off = align_up(off + h.out_bytes);
  h.oi = off; off = align_up(off + h.idx_bytes);
  h.ws = off;
  h.ws_bytes = layout_for(sh, seqlens, W, C).total;
  h.total = off + h.ws_bytes;
  return h;
}
}  // namespace

size_t snapkv_host_staging_size(const snapkv_shape* shape, const int32_t* seqlens_host,
                                int32_t W, int32_t C) {
  if (check_problem(shape, seqlens_host, W, C) != SNAPKV_OK) return 0;
  return host_layout(shape, seqlens_host, W, C).total;
}

int snapkv_compress_host(const snapkv_shape* shape, const void* q_win_host, const void* k_host,
                         const void* v_host, const int32_t* seqlens_host, int32_t W,
                         int32_t kernel_size, int32_t pool_type, int32_t C, void* out_k_host,
                         void* out_v_host, int32_t* out_idx_host, void* staging,
                         size_t staging_bytes, void* stream) {
  int rc = check_problem(shape, seqlens_host, W, C);
  if (rc != SNAPKV_OK) return rc;
  if (!q_win_host || !k_host || !v_host || !out_k_host || !out_v_host || !out_idx_host ||
      !staging || !aligned(staging, kAlign))
    return SNAPKV_ERR_INVALID_ARG;
  const HostLayout h = host_layout(shape, seqlens_host, W, C);
  if (staging_bytes < h.total) return SNAPKV_ERR_WORKSPACE;
  char* base = static_cast<char*>(staging);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Only the kept V rows are ever read: page-locked V stays on the host and
  // the gather reads those rows in place, instead of uploading all of V.
  const void* v_dev = base + h.v;
  bool v_zero_copy = false;
  {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, v_host) == cudaSuccess && at.type == cudaMemoryTypeHost &&
        at.devicePointer != nullptr && aligned(at.devicePointer, 16)) {
      v_dev = at.devicePointer;
      v_zero_copy = true;
    }
    cudaGetLastError();  // a pageable pointer is not an error here
  }
  if (cudaMemcpyAsync(base + h.q, q_win_host, h.q_bytes, cudaMemcpyHostToDevice, st) ||
      cudaMemcpyAsync(base + h.k, k_host, h.kv_bytes, cudaMemcpyHostToDevice, st) ||
      (!v_zero_copy &&
       cudaMemcpyAsync(base + h.v, v_host, h.kv_bytes, cudaMemcpyHostToDevice, st)))
    return SNAPKV_ERR_CUDA;
  rc = enqueue(shape, base + h.q, base + h.k, v_dev, seqlens_host, W, kernel_size, pool_type, C,
               base + h.ok, base + h.ov, reinterpret_cast<int32_t*>(base + h.oi), base + h.ws,
               h.ws_bytes, stream, false, nullptr, false, nullptr, nullptr, v_zero_copy);
  if (rc != SNAPKV_OK) return rc;
  if (cudaMemcpyAsync(out_k_host, base + h.ok, h.out_bytes, cudaMemcpyDeviceToHost, st) ||
      cudaMemcpyAsync(out_v_host, base + h.ov, h.out_bytes, cudaMemcpyDeviceToHost, st) ||
      cudaMemcpyAsync(out_idx_host, base + h.oi, h.idx_bytes, cudaMemcpyDeviceToHost, st))
    return SNAPKV_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SNAPKV_ERR_CUDA;
  return SNAPKV_OK;
}

size_t snapkv_host_staging_size_layers(const snapkv_shape* shape, const int32_t* seqlens_host,
                                       int32_t W, int32_t C) {
  if (check_problem(shape, seqlens_host, W, C) != SNAPKV_OK) return 0;
  return 2 * align_up(host_layout(shape, seqlens_host, W, C).total);
}

int snapkv_compress_host_layers(const snapkv_shape* shape, int32_t n_layers,
                                const void* const* q_win_host, const void* const* k_host,
                                const void* const* v_host, const int32_t* seqlens_host, int32_t W,
                                int32_t kernel_size, int32_t pool_type, int32_t C,
                                void* const* out_k_host, void* const* out_v_host,
                                int32_t* const* out_idx_host, void* staging, size_t staging_bytes,
                                void* stream, void* copy_stream, void* const* events) {
  int rc = check_problem(shape, seqlens_host, W, C);
  if (rc != SNAPKV_OK) return rc;
  if (n_layers < 1 || !q_win_host || !k_host || !v_host || !out_k_host || !out_v_host ||
      !out_idx_host || !staging || !aligned(staging, kAlign) || !events)
    return SNAPKV_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l)
    if (!q_win_host[l] || !k_host[l] || !v_host[l] || !out_k_host[l] || !out_v_host[l] ||
        !out_idx_host[l])
      return SNAPKV_ERR_INVALID_ARG;
  for (int e = 0; e < 4; ++e)
    if (!events[e]) return SNAPKV_ERR_INVALID_ARG;
  const HostLayout h = host_layout(shape, seqlens_host, W, C);
  const size_t slot = align_up(h.total);
  if (staging_bytes < 2 * slot) return SNAPKV_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStream_t cs = static_cast<cudaStream_t>(copy_stream);
  cudaEvent_t uploaded[2] = {static_cast<cudaEvent_t>(events[0]),
                             static_cast<cudaEvent_t>(events[1])};
  cudaEvent_t done[2] = {static_cast<cudaEvent_t>(events[2]), static_cast<cudaEvent_t>(events[3])};
  // two staging slots: layer l + 1's inputs upload on the copy stream while
  // layer l compresses on the compute stream; a slot is refilled only after
  // the compression that read it and the copy of its outputs have finished
  for (int l = 0; l < n_layers; ++l) {
    const int sl = l & 1;
    char* base = static_cast<char*>(staging) + sl * slot;
    const void* v_dev = base + h.v;
    bool v_zero_copy = false;
    {
      cudaPointerAttributes at{};
      if (cudaPointerGetAttributes(&at, v_host[l]) == cudaSuccess &&
          at.type == cudaMemoryTypeHost && at.devicePointer != nullptr &&
          aligned(at.devicePointer, 16)) {
        v_dev = at.devicePointer;
        v_zero_copy = true;
      }
      cudaGetLastError();  // a pageable pointer is not an error here
    }
    if (l >= 2 && cudaStreamWaitEvent(cs, done[sl], 0) != cudaSuccess) return SNAPKV_ERR_CUDA;
    if (cudaMemcpyAsync(base + h.q, q_win_host[l], h.q_bytes, cudaMemcpyHostToDevice, cs) ||
        cudaMemcpyAsync(base + h.k, k_host[l], h.kv_bytes, cudaMemcpyHostToDevice, cs) ||
        (!v_zero_copy &&
         cudaMemcpyAsync(base + h.v, v_host[l], h.kv_bytes, cudaMemcpyHostToDevice, cs)) ||
        cudaEventRecord(uploaded[sl], cs) || cudaStreamWaitEvent(st, uploaded[sl], 0))
      return SNAPKV_ERR_CUDA;
    rc = enqueue(shape, base + h.q, base + h.k, v_dev, seqlens_host, W, kernel_size, pool_type,
                 C, base + h.ok, base + h.ov, reinterpret_cast<int32_t*>(base + h.oi),
                 base + h.ws, h.ws_bytes, stream, false, nullptr, false, nullptr, nullptr,
                 v_zero_copy);
    if (rc != SNAPKV_OK) return rc;
    if (cudaMemcpyAsync(out_k_host[l], base + h.ok, h.out_bytes, cudaMemcpyDeviceToHost, st) ||
        cudaMemcpyAsync(out_v_host[l], base + h.ov, h.out_bytes, cudaMemcpyDeviceToHost, st) ||
        cudaMemcpyAsync(out_idx_host[l], base + h.oi, h.idx_bytes, cudaMemcpyDeviceToHost, st) ||
        cudaEventRecord(done[sl], st))
      return SNAPKV_ERR_CUDA;
  }
  if (cudaStreamSynchronize(st) != cudaSuccess || cudaStreamSynchronize(cs) != cudaSuccess)
    return SNAPKV_ERR_CUDA;
  return SNAPKV_OK;
}

}  // extern "C"
