// All-query ("heavy hitter") scoring, a SnapKV scoring variant: every prompt
// query votes, not only the observation window -- the accumulated attention
// that H2O uses, the method the SnapKV summary compares against (hotpaper.ai
// summary of "SnapKV: LLM Knows What You are Looking for Before
// Generation", "주요 결과").  For prefix key j < P = L - W of KV head h:
//
//   raw[j] = (1/g) sum_{hq in group} sum_{i = j}^{L-1} exp(q_i . k_j / sqrt(d) - lse_i)
//
// with lse_i the natural-log normaliser of query row i over the keys it sees
// (j <= i), which the caller's prefill attention has already computed (the
// scoring rides along with prefill: jisaku.com glossary "SnapKV", FAQ Q3).
// The work is ~L^2/2 * H_q * d multiply-adds per layer -- quadratic in the
// prompt, which is why SnapKV looks only at a window; it runs on the CUDA
// cores: one thread per prefix key holds its K row in registers while the
// CTA streams the query rows i >= its keys through shared memory.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "plan.h"

namespace snapkv {
namespace allq {

constexpr int kKeys = 128;   // prefix keys per CTA (one per thread)
constexpr int kRowsPos = 8;  // query positions staged per step

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// CTA -> (sequence, KV head, key chunk): chunks of 128 prefix keys, in
// sequence order, the heads of a sequence side by side.
__device__ __forceinline__ bool locate(const Plan& p, int cta, int& s, int& h, int& j0) {
  int base = 0;
  for (s = 0; s < p.nseq; ++s) {
    const SeqInfo& S = p.seq[s];
    if (!S.scored) continue;
    const int per = (S.P + kKeys - 1) / kKeys;
    if (cta < base + per * p.H_kv) {
      const int local = cta - base;
      h = local / per;
      j0 = (local % per) * kKeys;
      return true;
    }
    base += per * p.H_kv;
  }
  return false;
}

template <typename T, int D>
__global__ void __launch_bounds__(kKeys) score_allq_kernel(const __grid_constant__ Plan p) {
  extern __shared__ __align__(16) float sq[];  // [kRowsPos * g][D] queries, then [kRowsPos * g] lse2
  int s, h, j0;
  if (!locate(p, blockIdx.x, s, h, j0)) return;
  const SeqInfo& S = p.seq[s];
  const int g = p.g;
  float* lse2 = sq + (size_t)kRowsPos * g * D;
  const int j = j0 + threadIdx.x;
  const bool live = j < S.P;
  float kr[D];
  const T* kp = static_cast<const T*>(p.k) + ((size_t)(S.row0 + (live ? j : j0)) * p.H_kv + h) * D;
#pragma unroll
  for (int e = 0; e < D; ++e) kr[e] = to_f(kp[e]);
  const T* qa = static_cast<const T*>(p.q_all);
  float acc = 0.f;
  // query rows i >= j0 (rows below a thread's own key are skipped per thread)
  for (int i0 = j0; i0 < S.L; i0 += kRowsPos) {
    const int ni = min(kRowsPos, S.L - i0);
    __syncthreads();  // the previous step's readers are done
    for (int x = threadIdx.x; x < ni * g * D; x += blockDim.x) {
      const int r = x / D, c = x % D;  // r = position offset * g + member
      const int i = i0 + r / g, m = r % g;
      sq[x] = to_f(qa[((size_t)(S.row0 + i) * p.H_q + (size_t)h * g + m) * D + c]) *
              p.log2e_scale;
    }
    for (int x = threadIdx.x; x < ni * g; x += blockDim.x) {
      const int i = i0 + x / g, m = x % g;
      lse2[x] = p.lse_all[(size_t)(S.row0 + i) * p.H_q + (size_t)h * g + m] * 1.4426950408889634f;
    }
    __syncthreads();
    if (!live) continue;
    for (int r = 0; r < ni * g; ++r) {
      if (i0 + r / g < j) continue;  // row i sees keys <= i only
      const float* q = sq + (size_t)r * D;
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < D; e += 4) {
        const float4 q4 = *reinterpret_cast<const float4*>(q + e);
        dot = fmaf(q4.x, kr[e], dot);
        dot = fmaf(q4.y, kr[e + 1], dot);
        dot = fmaf(q4.z, kr[e + 2], dot);
        dot = fmaf(q4.w, kr[e + 3], dot);
      }
      acc += ex2(dot - lse2[r]);
    }
  }
  if (live) p.raw[S.score0 + (size_t)h * S.P + j] = acc / (float)g;
}

template <typename T, int D>
int launch_typed(const Plan& p, cudaStream_t st, int ctas) {
  const size_t smem = ((size_t)kRowsPos * p.g * D + (size_t)kRowsPos * p.g) * sizeof(float);
  cudaError_t e = cudaSuccess;
  if (smem > 48 * 1024)
    e = cudaFuncSetAttribute(score_allq_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
  if (e != cudaSuccess) return e;
  score_allq_kernel<T, D><<<ctas, kKeys, smem, st>>>(p);
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(1);
  return e;
}

}  // namespace allq

int launch_score_allq(const Plan& p, void* stream) {
  int ctas = 0;
  for (int s = 0; s < p.nseq; ++s)
    if (p.seq[s].scored) ctas += (p.seq[s].P + allq::kKeys - 1) / allq::kKeys * p.H_kv;
  if (ctas == 0) return cudaSuccess;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool bf = p.dtype == 0;
  if (p.d == 64)
    return bf ? allq::launch_typed<__nv_bfloat16, 64>(p, st, ctas)
              : allq::launch_typed<float, 64>(p, st, ctas);
  return bf ? allq::launch_typed<__nv_bfloat16, 128>(p, st, ctas)
            : allq::launch_typed<float, 128>(p, st, ctas);
}

}  // namespace snapkv
