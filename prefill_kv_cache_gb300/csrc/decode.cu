// One decode step of attention over a KV cache: the full prompt cache or the
// compressed one that snapkv_compress emits.
//
// After compression the generation (decode) phase attends over the compressed
// cache (jisaku.com glossary "SnapKV", "SnapKVの仕組み", algorithm flow step
// 4); a smaller cache relieves the memory-bandwidth bound of decoding
// (glossary FAQ Q2; hotpaper.ai summary of "SnapKV: LLM Knows What You are
// Looking for Before Generation", "주요 결과": 3.6x generation speed at 16K).
// Per sequence b and query head hq (KV head h = hq / g):
//
//   o[b, hq] = sum_j softmax_j(q[b, hq] . k[b, j, h] / sqrt(d)) v[b, j, h]
//
// over the sequence's n_b cached rows.  The step reads every cached K and V
// byte once and does ~2 multiply-adds per byte: it is HBM-bound, so it runs
// on the CUDA cores (split-K "flash decoding"):
//
//   decode_chunk   grid (key chunks of all sequences, H_kv), 8 warps.  A
//                  warp takes blocks of 32 keys: each lane computes its key's
//                  logits for the g query heads of the group from a whole K
//                  row (16-byte loads), the warp updates the running max and
//                  sum of exp2, then walks the block's keys broadcasting their
//                  weights while each lane accumulates its d/32 columns of
//                  the V rows (coalesced).  The CTA merges its warps and
//                  writes (max, sum, unnormalised output) per query head.
//   decode_combine grid (B, H_q): merges the chunks of each sequence.
//
// The Scissorhands instantiation (SH = true) serves one step of the
// decode-time eviction in scissorhands.cu: the rows of each sequence come from
// the device-side cache state (the step's append and eviction already ran),
// every logit is also stored for the history marks, and the combine stores
// each query head's final (max, sum).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "plan.h"
#include "sh_attention.h"
#include "snapkv.h"

namespace snapkv {
namespace dec {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kGroup = 512;        // sequences per launch (kernel-parameter table)
constexpr int kMinChunk = 128;     // keys per CTA, bounds
constexpr int kMaxChunk = 2048;
constexpr int kVUnroll = 8;        // V rows loaded ahead of their multiply-adds

struct Seq {
  long long row0;  // first cache row of the sequence (a row = H_kv * d elements)
  int n;           // cached rows
  int chunk0;      // first chunk of the sequence in this launch
};

struct Params {
  int nseq, H_q, H_kv, g, d, dtype, chunk, total_chunks;
  float c2;  // log2(e) / sqrt(d)
  const void* q;
  const void* k;
  const void* v;
  float* out;       // [B, H_q, d]
  float* part_o;    // [total_chunks, H_kv, g, d]
  float2* part_ml;  // [total_chunks, H_kv, g]: (max of log2-scaled logits, sum of exp2)
  int b0;           // batch index of seq[0]
  // Scissorhands step only
  const int* sh_state;  // [B, 4]: rows before the step's append, ...
  int sh_budget, sh_evict, sh_cap;
  float* sh_logits;     // [B, H_kv, cap, g]: log2-scaled logits
  float2* sh_ml;        // [B, H_q]: final (max, sum of exp2)
  Seq seq[kGroup];
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// 8 consecutive elements of a row as fp32
template <typename T>
__device__ __forceinline__ void load8(const T* p, float* f);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float* f) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float* f) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// this lane's DL = D / 32 consecutive columns of a V row as fp32
template <typename T, int DL>
__device__ __forceinline__ void load_cols(const T* p, float* f);
template <>
__device__ __forceinline__ void load_cols<__nv_bfloat16, 4>(const __nv_bfloat16* p, float* f) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  f[0] = __uint_as_float(u.x << 16);
  f[1] = __uint_as_float(u.x & 0xffff0000u);
  f[2] = __uint_as_float(u.y << 16);
  f[3] = __uint_as_float(u.y & 0xffff0000u);
}
template <>
__device__ __forceinline__ void load_cols<__nv_bfloat16, 2>(const __nv_bfloat16* p, float* f) {
  const uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(p));
  f[0] = __uint_as_float(u << 16);
  f[1] = __uint_as_float(u & 0xffff0000u);
}
template <>
__device__ __forceinline__ void load_cols<float, 4>(const float* p, float* f) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
}
template <>
__device__ __forceinline__ void load_cols<float, 2>(const float* p, float* f) {
  const float2 a = __ldg(reinterpret_cast<const float2*>(p));
  f[0] = a.x; f[1] = a.y;
}

template <typename T, int D, int G, bool SH>
__global__ void __launch_bounds__(kThreads) decode_chunk(const __grid_constant__ Params p) {
  constexpr int DL = D / 32;
  extern __shared__ __align__(16) float sm[];
  float* qs = sm;                        // [G][D], pre-scaled by log2(e)/sqrt(d)
  float* wml = qs + G * D;               // [kWarps][G][2]
  float* wacc = wml + kWarps * G * 2;    // [kWarps][G][D]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // persistent: units (chunk, KV head), the heads of a chunk side by side
  for (int unit_i = blockIdx.x; unit_i < p.total_chunks * p.H_kv; unit_i += gridDim.x) {
  const int ch = unit_i / p.H_kv, h = unit_i % p.H_kv;
  // the sequence of this chunk
  int lo = 0, hi = p.nseq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.seq[mid].chunk0 <= ch) lo = mid; else hi = mid - 1;
  }
  const Seq& S = p.seq[lo];
  const int b = p.b0 + lo;
  const int j0 = (ch - S.chunk0) * p.chunk;
  int rows = S.n;
  if constexpr (SH) {  // the rows after this step's append and eviction
    rows = p.sh_state[b * 4] + 1;
    if (rows > p.sh_budget) rows -= p.sh_evict;
    rows = min(max(rows, 0), p.sh_cap);
  }
  const int j1 = min(rows, j0 + p.chunk);
  __syncthreads();  // the previous unit's shared-memory readers are done

  const T* qb = static_cast<const T*>(p.q) + ((size_t)b * p.H_q + (size_t)h * G) * D;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    float f;
    if constexpr (sizeof(T) == 2)
      f = __bfloat162float(qb[i]);
    else
      f = qb[i];
    qs[i] = f * p.c2;
  }
  __syncthreads();

  const size_t row_elems = (size_t)p.H_kv * D;
  const T* kbase = static_cast<const T*>(p.k) + (size_t)S.row0 * row_elems + (size_t)h * D;
  const T* vbase = static_cast<const T*>(p.v) + (size_t)S.row0 * row_elems + (size_t)h * D;

  float m[G], l[G], acc[G][DL];
#pragma unroll
  for (int x = 0; x < G; ++x) {
    m[x] = -INFINITY;
    l[x] = 0.f;
#pragma unroll
    for (int c = 0; c < DL; ++c) acc[x][c] = 0.f;
  }
  // this warp's keys: a contiguous share of the chunk, in blocks of 32
  const int per = (p.chunk + kWarps - 1) / kWarps;
  const int wj0 = j0 + warp * per, wj1 = min(j1, wj0 + per);
  for (int base = wj0; base < wj1; base += 32) {
    const int j = base + lane;
    const bool live = j < wj1;
    float s[G];
#pragma unroll
    for (int x = 0; x < G; ++x) s[x] = 0.f;
    if (live) {
      const T* kr = kbase + (size_t)j * row_elems;
#pragma unroll
      for (int c = 0; c < D; c += 8) {  // all of the row's loads in flight at once
        float kf[8];
        load8<T>(kr + c, kf);
#pragma unroll
        for (int x = 0; x < G; ++x) {
          const float4 qa = *reinterpret_cast<const float4*>(qs + x * D + c);
          const float4 qc = *reinterpret_cast<const float4*>(qs + x * D + c + 4);
          s[x] = fmaf(qa.x, kf[0], s[x]);
          s[x] = fmaf(qa.y, kf[1], s[x]);
          s[x] = fmaf(qa.z, kf[2], s[x]);
          s[x] = fmaf(qa.w, kf[3], s[x]);
          s[x] = fmaf(qc.x, kf[4], s[x]);
          s[x] = fmaf(qc.y, kf[5], s[x]);
          s[x] = fmaf(qc.z, kf[6], s[x]);
          s[x] = fmaf(qc.w, kf[7], s[x]);
        }
      }
    }
    if constexpr (SH) {
      if (live) {
        float* lg = p.sh_logits + (((size_t)b * p.H_kv + h) * p.sh_cap + j) * G;
        if constexpr (G % 4 == 0) {
#pragma unroll
          for (int x = 0; x < G; x += 4)
            *reinterpret_cast<float4*>(lg + x) = make_float4(s[x], s[x + 1], s[x + 2], s[x + 3]);
        } else {
#pragma unroll
          for (int x = 0; x < G; ++x) lg[x] = s[x];
        }
      }
    }
    float pw[G];
#pragma unroll
    for (int x = 0; x < G; ++x) {
      const float bm = warp_max(live ? s[x] : -INFINITY);
      const float mn = fmaxf(m[x], bm);
      pw[x] = live ? ex2(s[x] - mn) : 0.f;
      const float sc = ex2(m[x] - mn);  // 0 on the first block (m = -inf)
      l[x] = l[x] * sc + warp_sum(pw[x]);
#pragma unroll
      for (int c = 0; c < DL; ++c) acc[x][c] *= sc;
      m[x] = mn;
    }
    const int nk = min(32, wj1 - base);
    for (int j8 = 0; j8 < nk; j8 += kVUnroll) {
      float vf[kVUnroll][DL];  // kVUnroll rows' loads in flight
#pragma unroll
      for (int u = 0; u < kVUnroll; ++u) {
        const int jj = min(j8 + u, nk - 1);  // past the block end: a row already loaded, weight 0
        load_cols<T, DL>(vbase + (size_t)(base + jj) * row_elems + lane * DL, vf[u]);
      }
#pragma unroll
      for (int u = 0; u < kVUnroll; ++u) {
#pragma unroll
        for (int x = 0; x < G; ++x) {
          float w = __shfl_sync(0xffffffffu, pw[x], (j8 + u) & 31);
          if (j8 + u >= nk) w = 0.f;
#pragma unroll
          for (int c = 0; c < DL; ++c) acc[x][c] = fmaf(w, vf[u][c], acc[x][c]);
        }
      }
    }
  }
  // merge the warps
#pragma unroll
  for (int x = 0; x < G; ++x) {
    if (lane == 0) {
      wml[(warp * G + x) * 2] = m[x];
      wml[(warp * G + x) * 2 + 1] = l[x];
    }
#pragma unroll
    for (int c = 0; c < DL; ++c) wacc[(warp * G + x) * D + lane * DL + c] = acc[x][c];
  }
  __syncthreads();
  const size_t unit = (size_t)unit_i;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int x = i / D, c = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wml[(w * G + x) * 2]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mw = wml[(w * G + x) * 2];
        if (mw == -INFINITY) continue;
        const float f = ex2(mw - M);
        L += wml[(w * G + x) * 2 + 1] * f;
        O += wacc[(w * G + x) * D + c] * f;
      }
    }
    p.part_o[unit * G * D + i] = O;
    if (c == 0) p.part_ml[unit * G + x] = make_float2(M, L);
  }
  }
}

// Grid (nseq, H_q), D threads: merges the chunks of one sequence and head.
template <bool SH>
__global__ void decode_combine(const __grid_constant__ Params p) {
  const int s = blockIdx.x, hq = blockIdx.y, c = threadIdx.x;
  const Seq& S = p.seq[s];
  const int h = hq / p.g, x = hq % p.g;
  const int nch = (S.n + p.chunk - 1) / p.chunk;
  float M = -INFINITY;
  for (int k = 0; k < nch; ++k)
    M = fmaxf(M, p.part_ml[((size_t)(S.chunk0 + k) * p.H_kv + h) * p.g + x].x);
  float L = 0.f, O = 0.f;
  for (int k = 0; k < nch; ++k) {
    const size_t unit = (size_t)(S.chunk0 + k) * p.H_kv + h;
    const float2 ml = p.part_ml[unit * p.g + x];
    if (ml.x == -INFINITY) continue;
    const float f = ex2(ml.x - M);
    L += ml.y * f;
    O += p.part_o[(unit * p.g + x) * p.d + c] * f;
  }
  p.out[((size_t)(p.b0 + s) * p.H_q + hq) * p.d + c] = O / L;
  if constexpr (SH) {
    if (c == 0) p.sh_ml[(size_t)(p.b0 + s) * p.H_q + hq] = make_float2(M, L);
  }
}

int sm_count() {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  return sms;
}

template <typename T, int D, bool SH = false>
cudaError_t launch_typed(const Params& p, cudaStream_t st) {
  const size_t smem = ((size_t)p.g * D + kWarps * p.g * 2 + (size_t)kWarps * p.g * D) * sizeof(float);
  const int units = p.total_chunks * p.H_kv;
  cudaError_t e = cudaSuccess;
  auto go = [&](auto kern) {
    if (smem > 48 * 1024)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    int per_sm = 0;
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e == cudaSuccess) {
      const int grid = std::max(1, std::min(units, sm_count() * std::max(per_sm, 1)));
      kern<<<grid, kThreads, smem, st>>>(p);
      e = cudaGetLastError();
    }
  };
  switch (p.g) {
    case 1: go(decode_chunk<T, D, 1, SH>); break;
    case 2: go(decode_chunk<T, D, 2, SH>); break;
    case 4: go(decode_chunk<T, D, 4, SH>); break;
    case 8: go(decode_chunk<T, D, 8, SH>); break;
    case 16: go(decode_chunk<T, D, 16, SH>); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  decode_combine<SH><<<dim3(p.nseq, p.H_q), D, 0, st>>>(p);
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(2);
  return e;
}

// Keys per unit: about eight units per SM over the launch (the persistent
// CTAs then finish within a fraction of a unit of each other), a multiple of
// 32 in [kMinChunk, kMaxChunk].
int chunk_for(long long total_rows, int H_kv, int sms) {
  const long long want = (total_rows * H_kv + 8LL * sms - 1) / (8LL * sms);
  const long long c = (want + 31) / 32 * 32;
  return (int)std::min<long long>(kMaxChunk, std::max<long long>(kMinChunk, c));
}

int check(const snapkv_shape* sh, const int32_t* lens, int32_t layout, int32_t C) {
  if (!sh || !lens) return SNAPKV_ERR_INVALID_ARG;
  if (sh->batch < 1 || sh->batch > kMaxBatch) return SNAPKV_ERR_INVALID_ARG;
  if (sh->num_q_heads < 1 || sh->num_kv_heads < 1 || sh->num_q_heads % sh->num_kv_heads)
    return SNAPKV_ERR_INVALID_ARG;
  if (sh->dtype != SNAPKV_BF16 && sh->dtype != SNAPKV_FP32) return SNAPKV_ERR_INVALID_ARG;
  if (layout != SNAPKV_CACHE_PACKED && layout != SNAPKV_CACHE_SLOTS) return SNAPKV_ERR_INVALID_ARG;
  if (layout == SNAPKV_CACHE_SLOTS && C < 1) return SNAPKV_ERR_INVALID_ARG;
  for (int b = 0; b < sh->batch; ++b) {
    if (lens[b] < 1) return SNAPKV_ERR_INVALID_ARG;
    if (layout == SNAPKV_CACHE_SLOTS && lens[b] > C) return SNAPKV_ERR_INVALID_ARG;
  }
  if (sh->head_dim != 64 && sh->head_dim != 128) return SNAPKV_ERR_UNSUPPORTED;
  const int g = sh->num_q_heads / sh->num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16) return SNAPKV_ERR_UNSUPPORTED;
  return SNAPKV_OK;
}

// Worst-case chunks of one launch group (the smallest chunk size).
size_t max_units(const snapkv_shape* sh, const int32_t* lens) {
  size_t best = 0;
  for (int g0 = 0; g0 < sh->batch; g0 += kGroup) {
    size_t ch = 0;
    for (int b = g0; b < std::min(sh->batch, g0 + kGroup); ++b)
      ch += (size_t)(lens[b] + kMinChunk - 1) / kMinChunk;
    best = std::max(best, ch);
  }
  return best * (size_t)sh->num_kv_heads;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace dec

size_t sh_attention_units(int B, int cap, int H_kv) {
  const size_t per = (size_t)(cap + dec::kMinChunk - 1) / dec::kMinChunk;
  return (size_t)std::min(B, dec::kGroup) * per * H_kv;
}

int launch_sh_attention(const ShAttention& a, void* stream) {
  dec::Params* pp = new dec::Params;
  dec::Params& p = *pp;
  std::memset(&p, 0, sizeof p);
  p.H_q = a.H_q;
  p.H_kv = a.H_kv;
  p.g = a.H_q / a.H_kv;
  p.d = a.d;
  p.dtype = a.dtype;
  p.c2 = (float)(1.4426950408889634 / std::sqrt((double)a.d));
  p.q = a.q;
  p.k = a.k;
  p.v = a.v;
  p.out = a.out;
  p.part_o = a.part_o;
  p.part_ml = a.part_ml;
  p.sh_state = a.state;
  p.sh_budget = a.budget;
  p.sh_evict = a.evict;
  p.sh_cap = a.cap;
  p.sh_logits = a.logits;
  p.sh_ml = a.ml;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int sms = dec::sm_count();
  cudaError_t e = cudaSuccess;
  for (int g0 = 0; g0 < a.B && e == cudaSuccess; g0 += dec::kGroup) {
    const int g1 = std::min(a.B, g0 + dec::kGroup);
    p.nseq = g1 - g0;
    p.b0 = g0;
    // chunks sized for the full cache: the rows in use are only known on the device
    p.chunk = dec::chunk_for((long long)p.nseq * a.cap, a.H_kv, sms);
    const int per = (a.cap + p.chunk - 1) / p.chunk;
    for (int s = 0; s < p.nseq; ++s) {
      p.seq[s].row0 = (long long)(g0 + s) * a.cap;
      p.seq[s].n = a.cap;
      p.seq[s].chunk0 = s * per;
    }
    p.total_chunks = p.nseq * per;
    if (p.dtype == SNAPKV_BF16)
      e = a.d == 64 ? dec::launch_typed<__nv_bfloat16, 64, true>(p, st)
                    : dec::launch_typed<__nv_bfloat16, 128, true>(p, st);
    else
      e = a.d == 64 ? dec::launch_typed<float, 64, true>(p, st)
                    : dec::launch_typed<float, 128, true>(p, st);
  }
  delete pp;
  return e;
}
}  // namespace snapkv

using namespace snapkv;

size_t snapkv_decode_workspace_size(const snapkv_shape* shape, const int32_t* lens_host,
                                    int32_t layout, int32_t C) {
  if (dec::check(shape, lens_host, layout, C) != SNAPKV_OK) return 0;
  const size_t units = dec::max_units(shape, lens_host);
  const int g = shape->num_q_heads / shape->num_kv_heads;
  const size_t o_bytes = units * g * shape->head_dim * sizeof(float);
  const size_t ml_bytes = units * g * sizeof(float2);
  return ((o_bytes + 255) & ~(size_t)255) + ((ml_bytes + 255) & ~(size_t)255);
}

int snapkv_decode_attention(const snapkv_shape* shape, const void* q, const void* k_cache,
                            const void* v_cache, int32_t layout, const int32_t* lens_host,
                            int32_t C, float* out, void* workspace, size_t workspace_bytes,
                            void* stream) {
  const int rc = dec::check(shape, lens_host, layout, C);
  if (rc != SNAPKV_OK) return rc;
  if (!q || !k_cache || !v_cache || !out || !workspace) return SNAPKV_ERR_INVALID_ARG;
  if (!dec::aligned16(q) || !dec::aligned16(k_cache) || !dec::aligned16(v_cache) ||
      !dec::aligned16(out) || !dec::aligned16(workspace))
    return SNAPKV_ERR_INVALID_ARG;
  const size_t need = snapkv_decode_workspace_size(shape, lens_host, layout, C);
  if (workspace_bytes < need) return SNAPKV_ERR_WORKSPACE;

  const int H_kv = shape->num_kv_heads, d = shape->head_dim;
  const int g = shape->num_q_heads / H_kv;
  const size_t units_max = dec::max_units(shape, lens_host);
  dec::Params* pp = new dec::Params;  // ~8 KB table: keep it off the host stack
  dec::Params& p = *pp;
  std::memset(&p, 0, sizeof p);
  p.H_q = shape->num_q_heads;
  p.H_kv = H_kv;
  p.g = g;
  p.d = d;
  p.dtype = shape->dtype;
  p.c2 = (float)(1.4426950408889634 / std::sqrt((double)d));
  p.q = q;
  p.k = k_cache;
  p.v = v_cache;
  p.out = out;
  char* ws = static_cast<char*>(workspace);
  p.part_o = reinterpret_cast<float*>(ws);
  p.part_ml = reinterpret_cast<float2*>(
      ws + ((units_max * g * d * sizeof(float) + 255) & ~(size_t)255));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int sms = dec::sm_count();
  long long packed_row = 0;
  int result = SNAPKV_OK;
  for (int g0 = 0; g0 < shape->batch && result == SNAPKV_OK; g0 += dec::kGroup) {
    const int g1 = std::min(shape->batch, g0 + dec::kGroup);
    long long rows = 0;
    for (int b = g0; b < g1; ++b) rows += lens_host[b];
    p.nseq = g1 - g0;
    p.b0 = g0;
    p.chunk = dec::chunk_for(rows, H_kv, sms);
    int chunks = 0;
    for (int b = g0; b < g1; ++b) {
      dec::Seq& S = p.seq[b - g0];
      S.n = lens_host[b];
      S.row0 = layout == SNAPKV_CACHE_PACKED ? packed_row : (long long)b * C;
      S.chunk0 = chunks;
      chunks += (S.n + p.chunk - 1) / p.chunk;
      packed_row += S.n;
    }
    p.total_chunks = chunks;
    cudaError_t e;
    if (p.dtype == SNAPKV_BF16)
      e = d == 64 ? dec::launch_typed<__nv_bfloat16, 64>(p, st)
                  : dec::launch_typed<__nv_bfloat16, 128>(p, st);
    else
      e = d == 64 ? dec::launch_typed<float, 64>(p, st) : dec::launch_typed<float, 128>(p, st);
    if (e != cudaSuccess) result = SNAPKV_ERR_CUDA;
  }
  delete pp;
  return result;
}
