// Scissorhands decode-time KV-cache eviction: one decode step of one layer
// (abeam.tech summary of "Scissorhands: Exploiting the Persistence of
// Importance Hypothesis for LLM KV Cache Compression at Test Time", 技術の仕組み:
// a per-head token budget; when the new token takes the cache past it, drop
// a batch of the tokens whose attention weight was below average most often
// over the last w steps, never the r newest; attend over what remains).
//
// Kernels of one step, in stream order (all state on the device, so the step
// can be captured in a CUDA graph):
//
//   sh_append_evict  grid (H_kv, B), 256 threads.  Writes the new token's K
//                    and V rows, position and cleared history into slot n of
//                    its head.  Where that makes budget + 1 rows: counts each
//                    candidate's history bits (popcount), finds the count
//                    threshold of the `evict` largest with a histogram over
//                    the count values, ranks equal counts by slot (the older
//                    token goes first) with block scans, and compacts K, V,
//                    positions and history in place -- sources are read a
//                    chunk at a time in slot order before any of the chunk is
//                    written, and a kept slot only ever moves down, so no
//                    unread source is overwritten.
//   decode_chunk, decode_combine (decode.cu, Scissorhands instantiation):
//                    attention over the rows that remain, keeping every logit
//                    and each query head's (max, sum).
//   sh_mark          grid (slot blocks, H_kv, B).  For each cached row, the
//                    group's weights relative to the average, sum_x n e_x / Z_x,
//                    against g decides the row's history bit for this step;
//                    the last CTA to finish advances every sequence's state.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <vector>

#include "pdl.cuh"
#include "plan.h"
#include "scissorhands.h"
#include "sh_attention.h"

namespace snapkv {
namespace sh {

constexpr int kThreads = 256;
constexpr int kMaxBudget = 16383;
constexpr int kMaxHistory = 1024;
constexpr uint16_t kGone = 0xffff;

struct Args {
  int B, H_q, H_kv, rowb;  // rowb: bytes of one K (or V) row of one head, d * element size
  int cap, budget, recent, history, evict, hw;
  const void* k_new;
  const void* v_new;
  void* k;
  void* v;
  int* pos;
  uint32_t* hist;
  int* state;
  const float* logits;
  const float2* ml;
  unsigned* done;
  // init only
  const void* k0;
  const void* v0;
  const int* pos0;
  int C0;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Exclusive prefix sum over the CTA of one int per thread; also the total.
// Every thread of the CTA must call it.
__device__ __forceinline__ int block_scan(int x, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int before = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const int t = warp_tot[w];
    if (w < warp) before += t;
    total += t;
  }
  __syncthreads();  // warp_tot may be reused by the next call
  return before + incl - x;
}

// Moves slot j's 32-bit entry of one per-slot array to dest[j], chunk by chunk.
__device__ void compact_words(uint32_t* base, const uint16_t* dest, int n1) {
  for (int c0 = 0; c0 < n1; c0 += kThreads) {
    const int j = c0 + threadIdx.x;
    int dj = -1;
    uint32_t x = 0;
    if (j < n1) {
      const int d = dest[j];
      if (d != kGone && d != j) {
        x = base[j];
        dj = d;
      }
    }
    __syncthreads();
    if (dj >= 0) base[dj] = x;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kThreads) sh_append_evict(const __grid_constant__ Args a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int warp_tot[kThreads / 32];
  __shared__ int s_thr, s_need;
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();  // the previous step's state and history are written
  if (b == 0 && h == 0 && tid == 0) *a.done = 0;  // sh_mark's completion count
  const int n = a.state[b * 4], np = a.state[b * 4 + 2];
  if (n < 0 || n > a.budget) return;  // a cache that was never initialised
  const int pieces = a.rowb / 16;
  const size_t slot_stride = (size_t)a.H_kv * a.rowb;
  char* kb = static_cast<char*>(a.k) + ((size_t)b * a.cap * a.H_kv + h) * a.rowb;
  char* vb = static_cast<char*>(a.v) + ((size_t)b * a.cap * a.H_kv + h) * a.rowb;
  const uint4* kn = reinterpret_cast<const uint4*>(static_cast<const char*>(a.k_new) +
                                                   ((size_t)b * a.H_kv + h) * a.rowb);
  const uint4* vn = reinterpret_cast<const uint4*>(static_cast<const char*>(a.v_new) +
                                                   ((size_t)b * a.H_kv + h) * a.rowb);
  int* pos = a.pos + ((size_t)b * a.H_kv + h) * a.cap;
  uint32_t* hist = a.hist + ((size_t)b * a.H_kv + h) * a.hw * a.cap;  // [hw][cap]

  // append at slot n (n <= budget < cap)
  for (int i = tid; i < 2 * pieces; i += kThreads) {
    const bool isv = i >= pieces;
    const int pc = isv ? i - pieces : i;
    reinterpret_cast<uint4*>((isv ? vb : kb) + (size_t)n * slot_stride)[pc] = (isv ? vn : kn)[pc];
  }
  if (tid == 0) pos[n] = np;
  for (int w = tid; w < a.hw; w += kThreads) hist[(size_t)w * a.cap + n] = 0;
  const int n1 = n + 1;
  if (n1 <= a.budget) return;  // uniform over the CTA
  __syncthreads();             // the appended row is visible to the whole CTA

  // ---- batch eviction of `evict` slots among the n1 - recent oldest ----
  const int cap_pad = (a.cap + 7) & ~7;
  uint16_t* cnt = reinterpret_cast<uint16_t*>(smem);  // [cap]
  uint16_t* dest = cnt + cap_pad;                     // [cap]
  int* bins = reinterpret_cast<int*>(dest + cap_pad);  // [history + 1]
  const int cand = n1 - a.recent;
  for (int v = tid; v <= a.history; v += kThreads) bins[v] = 0;
  __syncthreads();
  // the history words hold exactly the steps t - w .. t - 1 (bit t mod w is
  // rewritten at every step and a slot's words start at zero)
  for (int j = tid; j < cand; j += kThreads) {
    int c = 0;
    for (int w = 0; w < a.hw; ++w) c += __popc(hist[(size_t)w * a.cap + j]);
    c = min(c, a.history);  // only bits below `history` are ever set
    cnt[j] = (uint16_t)c;
    atomicAdd(&bins[c], 1);
  }
  __syncthreads();
  if (tid == 0) {
    // largest counts first: every slot above thr goes, plus the `need`
    // oldest at thr (thr = 0 when fewer than `evict` have a count at all)
    int acc = 0, v = a.history;
    for (; v > 0; --v) {
      if (acc + bins[v] >= a.evict) break;
      acc += bins[v];
    }
    s_thr = v;
    s_need = a.evict - acc;
  }
  __syncthreads();
  const int thr = s_thr, need = s_need;
  int eq_seen = 0, kept_seen = 0;
  for (int c0 = 0; c0 < n1; c0 += kThreads) {
    const int j = c0 + tid;
    int cj = -1;
    if (j < cand) cj = cnt[j];
    const int eq = cj == thr ? 1 : 0;
    int eq_tot, kept_tot;
    const int eq_before = eq_seen + block_scan(eq, warp_tot, eq_tot);
    const bool gone = j < cand && (cj > thr || (eq && eq_before < need));
    const int keep = (j < n1 && !gone) ? 1 : 0;
    const int kept_before = kept_seen + block_scan(keep, warp_tot, kept_tot);
    if (j < n1) dest[j] = keep ? (uint16_t)kept_before : kGone;
    eq_seen += eq_tot;
    kept_seen += kept_tot;
  }
  __syncthreads();

  // K and V rows: 4 * kThreads 16-byte pieces per chunk
  const int per_slot = 2 * pieces;
  const int chunk = 4 * kThreads / per_slot;
  for (int c0 = 0; c0 < n1; c0 += chunk) {
    uint4 reg[4];
    int dst[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = u * kThreads + tid;
      const int j = c0 + i / per_slot, pc = i % per_slot;
      dst[u] = -1;
      if (j < n1) {
        const int dj = dest[j];
        if (dj != kGone && dj != j) {
          const bool isv = pc >= pieces;
          reg[u] = reinterpret_cast<const uint4*>((isv ? vb : kb) +
                                                  (size_t)j * slot_stride)[isv ? pc - pieces : pc];
          dst[u] = dj;
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (dst[u] < 0) continue;
      const int pc = (u * kThreads + tid) % per_slot;
      const bool isv = pc >= pieces;
      reinterpret_cast<uint4*>((isv ? vb : kb) + (size_t)dst[u] * slot_stride)[isv ? pc - pieces : pc] =
          reg[u];
    }
    __syncthreads();
  }
  compact_words(reinterpret_cast<uint32_t*>(pos), dest, n1);
  for (int w = 0; w < a.hw; ++w) compact_words(hist + (size_t)w * a.cap, dest, n1);
}

template <int G>
__global__ void __launch_bounds__(kThreads) sh_mark(const __grid_constant__ Args a) {
  __shared__ float2 sml[G];
  __shared__ bool last;
  const int b = blockIdx.z, h = blockIdx.y, tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();  // the logits and each query head's (max, sum) are written
  int n = a.state[b * 4] + 1;
  if (n > a.budget) n -= a.evict;
  n = min(max(n, 0), a.cap);
  const unsigned t = (unsigned)a.state[b * 4 + 1];
  if (tid < G) sml[tid] = a.ml[(size_t)b * a.H_q + h * G + tid];
  __syncthreads();
  const int j = blockIdx.x * kThreads + tid;
  if (j < n) {
    const float* lg = a.logits + (((size_t)b * a.H_kv + h) * a.cap + j) * G;
    const float fn = (float)n;
    float rel = 0.f;  // n times the group-mean weight, times g
#pragma unroll
    for (int x = 0; x < G; ++x) rel += __fdiv_rn(fn * ex2(lg[x] - sml[x].x), sml[x].y);
    const unsigned u = t % (unsigned)a.history;
    uint32_t* wp = a.hist + (((size_t)b * a.H_kv + h) * a.hw + u / 32) * a.cap + j;
    const uint32_t bit = 1u << (u % 32);
    const uint32_t old = *wp;
    *wp = rel < (float)G ? (old | bit) : (old & ~bit);
  }
  // the last CTA to finish advances the state (every CTA has read it by then)
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned total = gridDim.x * gridDim.y * gridDim.z;
    last = atomicAdd(a.done, 1u) == total - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int s = tid; s < a.B; s += kThreads) {
    int* st = a.state + s * 4;
    int nn = st[0] + 1;
    if (nn > a.budget) nn -= a.evict;
    st[0] = nn;
    st[1] += 1;
    st[2] += 1;
  }
}

// Grid (H_kv, B): loads the prefix rows, positions, and zero history.
__global__ void __launch_bounds__(kThreads) sh_init(const __grid_constant__ Args a) {
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int n = a.state[b * 4];
  const int pieces = a.rowb / 16;
  const size_t slot_stride = (size_t)a.H_kv * a.rowb;
  char* kb = static_cast<char*>(a.k) + ((size_t)b * a.cap * a.H_kv + h) * a.rowb;
  char* vb = static_cast<char*>(a.v) + ((size_t)b * a.cap * a.H_kv + h) * a.rowb;
  for (int i = tid; i < n * 2 * pieces; i += kThreads) {
    const int s = i / (2 * pieces), pc = i % (2 * pieces);
    const bool isv = pc >= pieces;
    const char* src = static_cast<const char*>(isv ? a.v0 : a.k0) +
                      (((size_t)b * a.C0 + s) * a.H_kv + h) * a.rowb;
    reinterpret_cast<uint4*>((isv ? vb : kb) + (size_t)s * slot_stride)[isv ? pc - pieces : pc] =
        reinterpret_cast<const uint4*>(src)[isv ? pc - pieces : pc];
  }
  int* pos = a.pos + ((size_t)b * a.H_kv + h) * a.cap;
  for (int s = tid; s < n; s += kThreads)
    pos[s] = a.pos0 ? a.pos0[((size_t)b * a.H_kv + h) * a.C0 + s] : s;
  uint32_t* hist = a.hist + ((size_t)b * a.H_kv + h) * a.hw * a.cap;
  for (size_t i = tid; i < (size_t)a.hw * a.cap; i += kThreads) hist[i] = 0;
}

int check(const snapkv_shape* sh, const scissorhands_params* pr) {
  if (!sh || !pr) return SNAPKV_ERR_INVALID_ARG;
  if (sh->batch < 1 || sh->batch > kMaxBatch) return SNAPKV_ERR_INVALID_ARG;
  if (sh->num_q_heads < 1 || sh->num_kv_heads < 1 || sh->num_q_heads % sh->num_kv_heads)
    return SNAPKV_ERR_INVALID_ARG;
  if (sh->dtype != SNAPKV_BF16 && sh->dtype != SNAPKV_FP32) return SNAPKV_ERR_INVALID_ARG;
  if (pr->budget < 1 || pr->budget > kMaxBudget) return SNAPKV_ERR_INVALID_ARG;
  if (pr->recent < 1 || pr->recent > pr->budget) return SNAPKV_ERR_INVALID_ARG;
  if (pr->history < 1 || pr->history > kMaxHistory) return SNAPKV_ERR_INVALID_ARG;
  if (pr->evict < 1 || pr->evict > pr->budget + 1 - pr->recent) return SNAPKV_ERR_INVALID_ARG;
  if (sh->head_dim != 64 && sh->head_dim != 128) return SNAPKV_ERR_UNSUPPORTED;
  const int g = sh->num_q_heads / sh->num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16) return SNAPKV_ERR_UNSUPPORTED;
  return SNAPKV_OK;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct WsLayout {
  size_t done, part_o, part_ml, logits, ml, total;
};

WsLayout ws_layout(const snapkv_shape* sh, const scissorhands_params* pr) {
  const int cap = pr->budget + 1, g = sh->num_q_heads / sh->num_kv_heads;
  const size_t units = sh_attention_units(sh->batch, cap, sh->num_kv_heads);
  WsLayout w;
  w.done = 0;
  w.part_o = 256;
  w.part_ml = w.part_o + align256(units * g * sh->head_dim * sizeof(float));
  w.logits = w.part_ml + align256(units * g * sizeof(float2));
  w.ml = w.logits + align256((size_t)sh->batch * sh->num_q_heads * cap * sizeof(float));
  w.total = w.ml + align256((size_t)sh->batch * sh->num_q_heads * sizeof(float2));
  return w;
}

bool aligned(const void* p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

Args base_args(const snapkv_shape* sh, const scissorhands_params* pr, const scissorhands_cache* c) {
  Args a{};
  a.B = sh->batch;
  a.H_q = sh->num_q_heads;
  a.H_kv = sh->num_kv_heads;
  a.rowb = sh->head_dim * (sh->dtype == SNAPKV_BF16 ? 2 : 4);
  a.cap = pr->budget + 1;
  a.budget = pr->budget;
  a.recent = pr->recent;
  a.history = pr->history;
  a.evict = pr->evict;
  a.hw = (pr->history + 31) / 32;
  a.k = c->k;
  a.v = c->v;
  a.pos = c->pos;
  a.hist = c->hist;
  a.state = c->state;
  return a;
}

bool cache_ok(const scissorhands_cache* c) {
  return c && c->k && c->v && c->pos && c->hist && c->state && aligned(c->k, 16) &&
         aligned(c->v, 16) && aligned(c->pos, 16) && aligned(c->hist, 16) &&
         aligned(c->state, 16);
}

}  // namespace sh
}  // namespace snapkv

using namespace snapkv;

size_t scissorhands_buffer_bytes(const snapkv_shape* shape, const scissorhands_params* params,
                                 int32_t which) {
  if (sh::check(shape, params) != SNAPKV_OK) return 0;
  const size_t B = shape->batch, H_kv = shape->num_kv_heads, cap = params->budget + 1;
  const size_t e = shape->dtype == SNAPKV_BF16 ? 2 : 4;
  switch (which) {
    case SCISSORHANDS_BUF_K:
    case SCISSORHANDS_BUF_V: return B * cap * H_kv * shape->head_dim * e;
    case SCISSORHANDS_BUF_POS: return B * H_kv * cap * sizeof(int32_t);
    case SCISSORHANDS_BUF_HIST: return B * H_kv * ((params->history + 31) / 32) * cap * 4;
    case SCISSORHANDS_BUF_STATE: return B * 4 * sizeof(int32_t);
    default: return 0;
  }
}

size_t scissorhands_workspace_size(const snapkv_shape* shape, const scissorhands_params* params) {
  if (sh::check(shape, params) != SNAPKV_OK) return 0;
  return sh::ws_layout(shape, params).total;
}

int scissorhands_init(const snapkv_shape* shape, const scissorhands_params* params,
                      const scissorhands_cache* cache, const void* k0, const void* v0,
                      int32_t C0, const int32_t* pos0, const int32_t* lens0_host,
                      const int32_t* next_pos0_host, void* stream) {
  const int rc = sh::check(shape, params);
  if (rc != SNAPKV_OK) return rc;
  if (!sh::cache_ok(cache) || !lens0_host || !next_pos0_host) return SNAPKV_ERR_INVALID_ARG;
  bool any_rows = false;
  for (int b = 0; b < shape->batch; ++b) {
    if (lens0_host[b] < 0 || lens0_host[b] > params->budget || lens0_host[b] > C0 ||
        next_pos0_host[b] < 0)
      return SNAPKV_ERR_INVALID_ARG;
    any_rows |= lens0_host[b] > 0;
  }
  if (any_rows && (!k0 || !v0 || !sh::aligned(k0, 16) || !sh::aligned(v0, 16)))
    return SNAPKV_ERR_INVALID_ARG;
  std::vector<int32_t> st(4 * (size_t)shape->batch, 0);
  for (int b = 0; b < shape->batch; ++b) {
    st[4 * b] = lens0_host[b];
    st[4 * b + 2] = next_pos0_host[b];
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // from pageable memory: returns once the source has been staged
  if (cudaMemcpyAsync(cache->state, st.data(), st.size() * sizeof(int32_t),
                      cudaMemcpyHostToDevice, s) != cudaSuccess)
    return SNAPKV_ERR_CUDA;
  sh::Args a = sh::base_args(shape, params, cache);
  a.k0 = k0;
  a.v0 = v0;
  a.pos0 = pos0;
  a.C0 = C0;
  sh::sh_init<<<dim3(a.H_kv, a.B), sh::kThreads, 0, s>>>(a);
  if (cudaGetLastError() != cudaSuccess) return SNAPKV_ERR_CUDA;
  count_launches(1);
  return SNAPKV_OK;
}

int scissorhands_step(const snapkv_shape* shape, const scissorhands_params* params,
                      const scissorhands_cache* cache, const void* q, const void* k_new,
                      const void* v_new, float* out, void* workspace, size_t workspace_bytes,
                      void* stream) {
  const int rc = sh::check(shape, params);
  if (rc != SNAPKV_OK) return rc;
  if (!sh::cache_ok(cache) || !q || !k_new || !v_new || !out || !workspace)
    return SNAPKV_ERR_INVALID_ARG;
  if (!sh::aligned(q, 16) || !sh::aligned(k_new, 16) || !sh::aligned(v_new, 16) ||
      !sh::aligned(out, 16) || !sh::aligned(workspace, 256))
    return SNAPKV_ERR_INVALID_ARG;
  const sh::WsLayout w = sh::ws_layout(shape, params);
  if (workspace_bytes < w.total) return SNAPKV_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  sh::Args a = sh::base_args(shape, params, cache);
  a.k_new = k_new;
  a.v_new = v_new;
  a.logits = reinterpret_cast<const float*>(ws + w.logits);
  a.ml = reinterpret_cast<const float2*>(ws + w.ml);
  a.done = reinterpret_cast<unsigned*>(ws + w.done);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  const size_t smem = 2 * (size_t)((a.cap + 7) & ~7) * sizeof(uint16_t) +
                      (size_t)(a.history + 1) * sizeof(int);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(sh::sh_append_evict, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return SNAPKV_ERR_CUDA;
  if (launch_pdl(sh::sh_append_evict, dim3(a.H_kv, a.B), dim3(sh::kThreads), smem, s, a) !=
          cudaSuccess ||
      cudaGetLastError() != cudaSuccess)
    return SNAPKV_ERR_CUDA;

  ShAttention at{};
  at.B = a.B;
  at.H_q = a.H_q;
  at.H_kv = a.H_kv;
  at.d = shape->head_dim;
  at.dtype = shape->dtype;
  at.cap = a.cap;
  at.budget = a.budget;
  at.evict = a.evict;
  at.q = q;
  at.k = cache->k;
  at.v = cache->v;
  at.state = cache->state;
  at.out = out;
  at.part_o = reinterpret_cast<float*>(ws + w.part_o);
  at.part_ml = reinterpret_cast<float2*>(ws + w.part_ml);
  at.logits = reinterpret_cast<float*>(ws + w.logits);
  at.ml = reinterpret_cast<float2*>(ws + w.ml);
  if (launch_sh_attention(at, stream) != cudaSuccess) return SNAPKV_ERR_CUDA;

  const dim3 grid((a.cap + sh::kThreads - 1) / sh::kThreads, a.H_kv, a.B);
  cudaError_t e;
  switch (a.H_q / a.H_kv) {
    case 1: e = launch_pdl(sh::sh_mark<1>, grid, dim3(sh::kThreads), 0, s, a); break;
    case 2: e = launch_pdl(sh::sh_mark<2>, grid, dim3(sh::kThreads), 0, s, a); break;
    case 4: e = launch_pdl(sh::sh_mark<4>, grid, dim3(sh::kThreads), 0, s, a); break;
    case 8: e = launch_pdl(sh::sh_mark<8>, grid, dim3(sh::kThreads), 0, s, a); break;
    default: e = launch_pdl(sh::sh_mark<16>, grid, dim3(sh::kThreads), 0, s, a); break;
  }
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return SNAPKV_ERR_CUDA;
  count_launches(2);
  return SNAPKV_OK;
}
