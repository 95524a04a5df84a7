// Observation-window scores on CUDA cores (FFMA), for any element type.
//
// This is the path for fp32 inputs (where tensor cores would round the
// operands) and for shapes the tensor-core kernel does not take.  It computes
// the window attention scores exactly as defined: softmax(q.k / sqrt(d)) of
// each window row over its causally visible keys, summed over the window rows
// for every prefix key and averaged over the query heads of the KV group
// (jisaku.com glossary "SnapKV", "SnapKVの仕組み"; hotpaper.ai summary of
// "SnapKV: LLM Knows What You are Looking for Before Generation",
// "핵심 아이디어").  Without storing the W x L probability matrix, it runs in
// two passes over K:
//
//   pass 1: per key chunk, the running max and sum of exp of each window
//           row (online softmax statistics), written per chunk;
//   merge:  per row, the log-sum-exp over chunks;
//   pass 2: per prefix key, sum over rows of exp(logit - lse) / g.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "plan.h"

namespace snapkv {

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Sequence owning score piece `piece`: the last one whose piece0 <= piece
// (sequences that are not scored own no pieces and share the next piece0).
__device__ __forceinline__ int piece_seq(const Plan& p, int piece) {
  int lo = 0, hi = p.nseq - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (p.seq[mid].piece0 <= piece) lo = mid; else hi = mid - 1;
  }
  return lo;
}

constexpr int kSimtThreads = 256;
constexpr int kSimtTileKeys = 32;

// Pass 1.  Grid: (total_pieces, ceil(Wp / 256)).  Thread = (row, key split).
template <typename T, int D>
__global__ void __launch_bounds__(kSimtThreads)
score_pass1_simt(const __grid_constant__ Plan p) {
  __shared__ float ks[kSimtTileKeys][D];
  __shared__ float2 red[kSimtThreads];
  const int piece = blockIdx.x;
  const int s = piece_seq(p, piece);
  const SeqInfo& S = p.seq[s];
  const int local = piece - S.piece0;
  const int h = local / S.chunks;
  const int c = local % S.chunks;
  const int key_begin = c * p.chunk_keys;
  const int key_end = min(S.L, key_begin + p.chunk_keys);

  const int t = threadIdx.x;
  const int RB = min(p.Wp, kSimtThreads);
  const int nsplit = kSimtThreads / RB;
  const int rloc = t % RB;
  const int split = t / RB;
  const int row = blockIdx.y * kSimtThreads + rloc;
  const bool active = split < nsplit && row < p.Wp;

  const int i = row / p.g;       // window row
  const int member = row % p.g;  // query head within the group
  float q[D];
  if (active) {
    const T* qp = static_cast<const T*>(p.q) +
                  ((size_t)(S.b * p.W + i) * p.H_q + (size_t)h * p.g + member) * D;
#pragma unroll
    for (int e = 0; e < D; ++e) q[e] = to_f(qp[e]);
  }
  const int limit = S.P + i;  // last key this row sees (causal)
  const T* kbase = static_cast<const T*>(p.k);
  float m = -INFINITY, z = 0.f;
  for (int tile = key_begin; tile < key_end; tile += kSimtTileKeys) {
    __syncthreads();
    for (int e = t; e < kSimtTileKeys * D; e += kSimtThreads) {
      const int kk = e / D, cc = e % D;
      const int j = tile + kk;
      ks[kk][cc] = (j < key_end)
                       ? to_f(kbase[((size_t)(S.row0 + j) * p.H_kv + h) * D + cc])
                       : 0.f;
    }
    __syncthreads();
    if (active) {
      for (int kk = split; kk < kSimtTileKeys; kk += nsplit) {
        const int j = tile + kk;
        if (j >= key_end || j > limit) break;
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < D; ++e) dot = fmaf(q[e], ks[kk][e], dot);
        const float x = dot * p.scale;
        if (x > m) {
          z = z * expf(m - x) + 1.f;
          m = x;
        } else {
          z += expf(x - m);
        }
      }
    }
  }
  red[t] = make_float2(m, z);
  __syncthreads();
  if (active && split == 0) {
    for (int sp = 1; sp < nsplit; ++sp) {
      const float2 o = red[sp * RB + rloc];
      if (o.x == -INFINITY) continue;
      if (o.x > m) {
        z = z * expf(m - o.x) + o.y;
        m = o.x;
      } else {
        z += o.y * expf(o.x - m);
      }
    }
    p.stats[(size_t)piece * p.Wp + row] = make_float2(m, z);
  }
}

// Merge of the per-chunk statistics: lse = M + log(sum_c z_c exp(m_c - M)).
// Grid: nseq * H_kv blocks.
__global__ void __launch_bounds__(kSimtThreads) lse_merge(const __grid_constant__ Plan p) {
  const int unit = blockIdx.x;
  const int s = unit / p.H_kv, h = unit % p.H_kv;
  const SeqInfo& S = p.seq[s];
  if (!S.scored) return;
  const float2* st = p.stats + (size_t)(S.piece0 + h * S.chunks) * p.Wp;
  for (int row = threadIdx.x; row < p.Wp; row += blockDim.x) {
    float M = -INFINITY;
    for (int c = 0; c < S.chunks; ++c) M = fmaxf(M, st[(size_t)c * p.Wp + row].x);
    float Z = 0.f;
    for (int c = 0; c < S.chunks; ++c) {
      const float2 v = st[(size_t)c * p.Wp + row];
      if (v.x != -INFINITY) Z += v.y * expf(v.x - M);
    }
    p.lse[(size_t)unit * p.Wp + row] = M + logf(Z);
  }
}

// Pass 2.  Grid: total_pieces.  Thread = prefix key; loops over all rows.
template <typename T, int D>
__global__ void __launch_bounds__(kSimtThreads)
score_pass2_simt(const __grid_constant__ Plan p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  T* qs = reinterpret_cast<T*>(smem_raw);
  float* lse_s = reinterpret_cast<float*>(smem_raw + (size_t)p.Wp * D * sizeof(T));
  const int piece = blockIdx.x;
  const int s = piece_seq(p, piece);
  const SeqInfo& S = p.seq[s];
  const int local = piece - S.piece0;
  const int h = local / S.chunks;
  const int c = local % S.chunks;
  const int key_begin = c * p.chunk_keys;
  const int key_end = min(S.P, key_begin + p.chunk_keys);
  if (key_begin >= key_end) return;

  const T* qb = static_cast<const T*>(p.q);
  for (int e = threadIdx.x; e < p.Wp * D; e += blockDim.x) {
    const int row = e / D, cc = e % D;
    const int i = row / p.g, member = row % p.g;
    qs[e] = qb[((size_t)(S.b * p.W + i) * p.H_q + (size_t)h * p.g + member) * D + cc];
  }
  if (p.lse_in) {  // the caller's LSE, row = i * g + member
    for (int row = threadIdx.x; row < p.Wp; row += blockDim.x)
      lse_s[row] = p.lse_in[(size_t)(S.b * p.W + row / p.g) * p.H_q + (size_t)h * p.g + row % p.g];
  } else {
    const float* lse = p.lse + (size_t)(s * p.H_kv + h) * p.Wp;
    for (int row = threadIdx.x; row < p.Wp; row += blockDim.x) lse_s[row] = lse[row];
  }
  __syncthreads();

  const T* kbase = static_cast<const T*>(p.k);
  if (p.out_heads != p.H_kv) {
    // every query head keeps its own sum (member m = row % g), no group mean
    float* rawq = p.raw + S.score0 + (size_t)h * p.g * S.P;
    for (int j = key_begin + threadIdx.x; j < key_end; j += blockDim.x) {
      float kr[D];
      const T* kp = kbase + ((size_t)(S.row0 + j) * p.H_kv + h) * D;
#pragma unroll
      for (int e = 0; e < D; ++e) kr[e] = to_f(kp[e]);
      float accm[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int row = 0; row < p.Wp; ++row) {
        const T* qr = qs + (size_t)row * D;
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < D; ++e) dot = fmaf(to_f(qr[e]), kr[e], dot);
        const float v = expf(dot * p.scale - lse_s[row]);
        const int m = row % p.g;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (k == m) accm[k] += v;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k < p.g) rawq[(size_t)k * S.P + j] = accm[k];
    }
    return;
  }
  float* raw = p.raw + S.score0 + (size_t)h * S.P;
  for (int j = key_begin + threadIdx.x; j < key_end; j += blockDim.x) {
    float kr[D];
    const T* kp = kbase + ((size_t)(S.row0 + j) * p.H_kv + h) * D;
#pragma unroll
    for (int e = 0; e < D; ++e) kr[e] = to_f(kp[e]);
    float acc = 0.f;
    for (int row = 0; row < p.Wp; ++row) {
      const T* qr = qs + (size_t)row * D;
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < D; ++e) dot = fmaf(to_f(qr[e]), kr[e], dot);
      acc += expf(dot * p.scale - lse_s[row]);
    }
    raw[j] = acc / (float)p.g;
  }
}

template <typename T, int D>
static int launch_simt_typed(const Plan& p, cudaStream_t st) {
  cudaError_t e;
  if (!p.lse_in) {  // pass 1 and the merge make the LSE; a caller's LSE replaces both
    dim3 g1(p.total_pieces, (p.Wp + kSimtThreads - 1) / kSimtThreads);
    score_pass1_simt<T, D><<<g1, kSimtThreads, 0, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    lse_merge<<<p.nseq * p.H_kv, kSimtThreads, 0, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launches(2);
  }
  const size_t smem = (size_t)p.Wp * D * sizeof(T) + (size_t)p.Wp * sizeof(float);
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(score_pass2_simt<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
  }
  score_pass2_simt<T, D><<<p.total_pieces, kSimtThreads, smem, st>>>(p);
  count_launches(1);
  count_score_launches(kScorePathCudaCores, 1);
  return cudaGetLastError();
}

int launch_score_simt(const Plan& p, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p.total_pieces == 0) return cudaSuccess;
  const bool bf = p.dtype == 0;
  if (p.d == 64) return bf ? launch_simt_typed<__nv_bfloat16, 64>(p, st)
                           : launch_simt_typed<float, 64>(p, st);
  return bf ? launch_simt_typed<__nv_bfloat16, 128>(p, st) : launch_simt_typed<float, 128>(p, st);
}

}  // namespace snapkv
