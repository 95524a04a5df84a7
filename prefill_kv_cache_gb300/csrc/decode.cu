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
// on the CUDA cores (split-K "flash decoding"), with the cache streamed
// through shared memory by the bulk-copy (TMA) engine:
//
//   decode_chunk   persistent, one CTA of up to 8 warps per SM; work units
//                  are (key chunk, KV head), the chunk length chosen so the
//                  CTA with the most units does the least work.  Each warp
//                  owns a contiguous share of a unit's rows and streams it in
//                  blocks of 32 rows through its own shared-memory slots --
//                  two for K, one for V: lane 0 issues the TMA tensor copies
//                  (boxes of 32 rows x 128 bytes of one head, 128-byte
//                  swizzle) that complete on each slot's mbarrier; the next
//                  block's K is in flight while the current block is
//                  computed, its V while the next block's logits are (blocks
//                  of the next unit included).  The swizzle puts the 16-byte
//                  pieces of 8 consecutive rows in distinct banks, so the
//                  per-lane row reads of the logit phase are conflict-free.
//                  Lane i computes row i's logits for the g query heads of
//                  the group; the warp updates its running max and sum of
//                  exp2; each lane then accumulates its d/32 columns over the
//                  block's V rows (packed fp32x2 FMAs in both phases).  The
//                  CTA merges its warps and writes (max, sum, unnormalised
//                  output) per query head.
//   decode_combine grid (B, H_q): merges the chunks of each sequence.
//
// Both are launched with programmatic dependent launch (pdl.cuh).
//
// The Scissorhands instantiation (SH = true) serves one step of the
// decode-time eviction in scissorhands.cu: the rows of each sequence come from
// the device-side cache state (the step's append and eviction already ran),
// every logit is also stored for the history marks, and the combine stores
// each query head's final (max, sum).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "pdl.cuh"
#include "plan.h"
#include "sh_attention.h"
#include "snapkv.h"

namespace snapkv {
namespace dec {

constexpr int kGroup = 512;        // sequences per launch (kernel-parameter table)
constexpr int kMinChunk = 128;     // keys per unit, bounds
constexpr int kMaxChunk = 16384;
constexpr int kRows = 32;          // rows per block: one per lane
constexpr int kMaxWarps = 8;
constexpr uint64_t kWaitNs = 2000000000ull;  // a stage that has not landed in 2 s
constexpr int kBoxBytes = kRows * 128;       // one TMA box: 32 rows x 128 bytes

struct Seq {
  long long row0;  // first cache row of the sequence (a row = H_kv * d elements)
  int n;           // cached rows
  int chunk0;      // first chunk of the sequence in this launch
};

struct Params {
  int nseq, H_q, H_kv, g, d, dtype, chunk, total_chunks;
  int warps, stages, nbw;  // warps per CTA, stages per warp, blocks per warp per unit
  float c2;  // log2(e) / sqrt(d)
  const void* q;
  const void* k;
  const void* v;
  float* out;       // [B, H_q, d]
  float* part_o;    // [total_chunks, H_kv, g, d]
  float2* part_ml;  // [total_chunks, H_kv, g]: (max of log2-scaled logits, sum of exp2)
  int b0;           // batch index of seq[0]
  long long rows_total;  // rows of the k / v arrays (the tensor maps' extent)
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

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ bool bar_test(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred q;\n mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n"
      " selp.b32 %0, 1, 0, q;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait for a stage; false once the CTA is aborting (its flag was
// already up, or this wait ran out and raised it).
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (bar_test(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (bar_test(bar, parity)) return true;
    if ((it & 31) == 0) {
      if (*abort) return false;
      if (global_ns() - t0 > kWaitNs) {
        *abort = 1;
        return false;
      }
    }
  }
}

// 8 consecutive elements of a row in shared memory as fp32
template <typename T>
__device__ __forceinline__ void lds8(const unsigned char* p, float* f);
template <>
__device__ __forceinline__ void lds8<__nv_bfloat16>(const unsigned char* p, float* f) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// DL consecutive elements of a row in shared memory as fp32
template <typename T, int DL>
__device__ __forceinline__ void lds_cols(const unsigned char* p, float* f) {
  if constexpr (sizeof(T) == 2 && DL == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    f[0] = __uint_as_float(u.x << 16);
    f[1] = __uint_as_float(u.x & 0xffff0000u);
    f[2] = __uint_as_float(u.y << 16);
    f[3] = __uint_as_float(u.y & 0xffff0000u);
  } else if constexpr (sizeof(T) == 2 && DL == 2) {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    f[0] = __uint_as_float(u << 16);
    f[1] = __uint_as_float(u & 0xffff0000u);
  } else if constexpr (DL == 4) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  } else {
    const float2 a = *reinterpret_cast<const float2*>(p);
    f[0] = a.x; f[1] = a.y;
  }
}

// Shared-memory bytes of one slot: 32 K (or V) rows as 128-byte wide boxes
// (a row of D * esize bytes spans D * esize / 128 boxes).
__host__ __device__ constexpr int boxes(int D, int esize) { return D * esize / 128; }
__host__ __device__ constexpr int slot_bytes(int D, int esize) {
  return boxes(D, esize) * kBoxBytes;
}
// Byte address of byte o of row r within a 128-byte-swizzled K or V block:
// 16-byte piece c of row r sits at piece c ^ (r mod 8) of its 128-byte line.
__device__ __forceinline__ int swz(int r, int o) {
  return (o >> 7) * kBoxBytes + r * 128 + ((((o >> 4) & 7) ^ (r & 7)) << 4) + (o & 15);
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// Where the unit's rows of one sequence start and end.
struct UnitRows {
  int seq, h, j0, j1;
};

template <bool SH>
__device__ __forceinline__ UnitRows unit_rows(const Params& p, int unit_i) {
  const int ch = unit_i / p.H_kv;
  UnitRows u;
  u.h = unit_i % p.H_kv;
  int lo = 0, hi = p.nseq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.seq[mid].chunk0 <= ch) lo = mid; else hi = mid - 1;
  }
  u.seq = lo;
  const Seq& S = p.seq[lo];
  int rows = S.n;
  if constexpr (SH) {  // the rows after this step's append and eviction
    rows = p.sh_state[(p.b0 + lo) * 4] + 1;
    if (rows > p.sh_budget) rows -= p.sh_evict;
    rows = min(max(rows, 0), p.sh_cap);
  }
  u.j0 = (ch - S.chunk0) * p.chunk;
  u.j1 = min(rows, u.j0 + p.chunk);
  return u;
}

template <typename T, int D, int G, bool SH>
__global__ void __launch_bounds__(kMaxWarps * 32, 1)
    decode_chunk(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v) {
  constexpr int DL = D / 32;
  constexpr int NB = boxes(D, (int)sizeof(T));
  constexpr int SLOT = slot_bytes(D, (int)sizeof(T));
  constexpr int EPB = 128 / (int)sizeof(T);  // elements per box row
  extern __shared__ __align__(1024) unsigned char sm_raw[];
  // the swizzle pattern repeats every 1024 bytes: boxes start on such a boundary
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // per warp: NS K slots and one V slot (the next block's V is fetched while
  // its logits are computed)
  const int warps = p.warps, NS = p.stages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* kslots = sm + (size_t)warp * (NS + 1) * SLOT;
  unsigned char* vslot = kslots + (size_t)NS * SLOT;
  uint64_t* bars0 = reinterpret_cast<uint64_t*>(sm + (size_t)warps * (NS + 1) * SLOT);
  uint64_t* kbars = bars0 + warp * (NS + 1);
  uint64_t* vbar = kbars + NS;
  float* qs = reinterpret_cast<float*>(bars0 + warps * (NS + 1));  // [G][D], pre-scaled
  float* pwb = qs + G * D + warp * kRows * G;        // this warp's [32][G] weights
  float* wml = qs + G * D + warps * kRows * G;       // [warps][G][2]
  float* wacc = wml + warps * G * 2;                 // [warps][G][D]
  volatile int* abort = reinterpret_cast<volatile int*>(wacc + warps * G * D);

  const int nunits = p.total_chunks * p.H_kv;
  const int my_units =
      (int)blockIdx.x < nunits ? (nunits - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int total = my_units * p.nbw;  // blocks in this warp's stream
  if (threadIdx.x == 0) *abort = 0;
  if (lane == 0)
    for (int s = 0; s <= NS; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&kbars[s])) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  pdl_trigger();
  __syncthreads();
  pdl_wait();  // the cache, the queries and the cache state are written

  // the rows [first, first + count) of block n of this warp's stream
  auto block_rows = [&](int n, int& seq, int& h, int& first, int& count) {
    const int k = n / p.nbw, m = n % p.nbw;
    const UnitRows u = unit_rows<SH>(p, (int)blockIdx.x + k * (int)gridDim.x);
    seq = u.seq;
    h = u.h;
    first = u.j0 + (warp * p.nbw + m) * kRows;
    count = min(kRows, u.j1 - first);
    if (count < 0) count = 0;
  };
  // lane 0 copies block n's K (or V) boxes into a slot (rows past the end of
  // the cache arrive as zeros and are not used)
  int k_issued = 0, k_landed = 0, v_issued = 0, v_landed = 0;  // blocks, in order
  auto issue = [&](int n, bool is_v) {
    const int stop = __shfl_sync(0xffffffffu, *abort, 0);  // one decision for the warp
    if (n >= total || stop) return;
    (is_v ? v_issued : k_issued) = n + 1;
    if (lane != 0) return;
    int seq, h, first, count;
    block_rows(n, seq, h, first, count);
    const uint32_t bar = saddr(is_v ? vbar : &kbars[n % NS]);
    if (count > 0) {
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                   "r"(SLOT)
                   : "memory");
      const uint32_t dst = saddr(is_v ? vslot : kslots + (size_t)(n % NS) * SLOT);
      const int row = (int)(p.seq[seq].row0 + first);
#pragma unroll
      for (int bx = 0; bx < NB; ++bx)
        tma_load_3d(dst + bx * kBoxBytes, is_v ? &tm_v : &tm_k, bar, bx * EPB, h, row);
    } else {
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
    }
  };

  // Swizzled offsets depend on a row only through row mod 8: this lane's
  // K row (logit phase) and its V columns in rows 8i + u (output phase).
  int koff[8], voff[8];
  {
    const int vo = lane * DL * (int)sizeof(T);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      koff[u] = lane * 128 + ((u ^ (lane & 7)) << 4);
      voff[u] = (vo >> 7) * kBoxBytes + u * 128 + ((((vo >> 4) & 7) ^ u) << 4) + (vo & 15);
    }
  }

  for (int n = 0; n < NS; ++n) issue(n, false);
  issue(0, true);
  int n = 0;
  for (int k = 0; k < my_units; ++k) {
    const int unit_i = (int)blockIdx.x + k * (int)gridDim.x;
    const UnitRows u = unit_rows<SH>(p, unit_i);
    const int b = p.b0 + u.seq, h = u.h;
    __syncthreads();  // the previous unit's merge has read wml / wacc
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

    // packed fp32 pairs (fma.rn.f32x2): this lane's columns 2i, 2i + 1
    float m[G], l[G];
    float2 acc[G][DL / 2];
#pragma unroll
    for (int x = 0; x < G; ++x) {
      m[x] = -INFINITY;
      l[x] = 0.f;
#pragma unroll
      for (int c = 0; c < DL / 2; ++c) acc[x][c] = make_float2(0.f, 0.f);
    }
    for (int mb = 0; mb < p.nbw; ++mb, ++n) {
      const int s = n % NS;
      const int first = u.j0 + (warp * p.nbw + mb) * kRows;
      const int count = max(0, min(kRows, u.j1 - first));
      // every lane polls; the block is used only if all of them saw it land
      const bool ready =
          __all_sync(0xffffffffu, bar_wait(saddr(&kbars[s]), (uint32_t)(n / NS) & 1u, abort));
      if (ready) k_landed = n + 1;
      const unsigned char* kst = kslots + (size_t)s * SLOT;
      const unsigned char* vst = vslot;
      if (ready && count > 0) {
        const bool live = lane < count;
        float sc[G];
#pragma unroll
        for (int x = 0; x < G; ++x) sc[x] = 0.f;
        if (live) {
          // two packed partial sums per query head: four independent pairs
          float2 pa[G], pb[G];
#pragma unroll
          for (int x = 0; x < G; ++x) {
            pa[x] = make_float2(0.f, 0.f);
            pb[x] = make_float2(0.f, 0.f);
          }
#pragma unroll
          for (int c = 0; c < D; c += 8) {
            float kf[8];
            if constexpr (sizeof(T) == 2) {  // piece c / 8 of the row
              lds8<T>(kst + (c >> 6) * kBoxBytes + koff[(c >> 3) & 7], kf);
            } else {  // 8 floats span pieces c / 4 and c / 4 + 1
              const float4 a =
                  *reinterpret_cast<const float4*>(kst + (c >> 5) * kBoxBytes + koff[(c >> 2) & 7]);
              const float4 b2 = *reinterpret_cast<const float4*>(
                  kst + ((c + 4) >> 5) * kBoxBytes + koff[((c + 4) >> 2) & 7]);
              kf[0] = a.x; kf[1] = a.y; kf[2] = a.z; kf[3] = a.w;
              kf[4] = b2.x; kf[5] = b2.y; kf[6] = b2.z; kf[7] = b2.w;
            }
#pragma unroll
            for (int x = 0; x < G; ++x) {
              const float4 qa = *reinterpret_cast<const float4*>(qs + x * D + c);
              const float4 qc = *reinterpret_cast<const float4*>(qs + x * D + c + 4);
              pa[x] = __ffma2_rn(make_float2(qa.x, qa.y), make_float2(kf[0], kf[1]), pa[x]);
              pb[x] = __ffma2_rn(make_float2(qa.z, qa.w), make_float2(kf[2], kf[3]), pb[x]);
              pa[x] = __ffma2_rn(make_float2(qc.x, qc.y), make_float2(kf[4], kf[5]), pa[x]);
              pb[x] = __ffma2_rn(make_float2(qc.z, qc.w), make_float2(kf[6], kf[7]), pb[x]);
            }
          }
#pragma unroll
          for (int x = 0; x < G; ++x) sc[x] = (pa[x].x + pa[x].y) + (pb[x].x + pb[x].y);
          if constexpr (SH) {
            float* lg = p.sh_logits + (((size_t)b * p.H_kv + h) * p.sh_cap + first + lane) * G;
            if constexpr (G % 4 == 0) {
#pragma unroll
              for (int x = 0; x < G; x += 4)
                *reinterpret_cast<float4*>(lg + x) =
                    make_float4(sc[x], sc[x + 1], sc[x + 2], sc[x + 3]);
            } else {
#pragma unroll
              for (int x = 0; x < G; ++x) lg[x] = sc[x];
            }
          }
        }
#pragma unroll
        for (int x = 0; x < G; ++x) {
          const float bm = warp_max(live ? sc[x] : -INFINITY);
          const float mn = fmaxf(m[x], bm);
          const float pw = live ? ex2(sc[x] - mn) : 0.f;
          const float f = ex2(m[x] - mn);  // 0 on the first block (m = -inf)
          l[x] = l[x] * f + warp_sum(pw);
#pragma unroll
          for (int c = 0; c < DL / 2; ++c) acc[x][c] = __fmul2_rn(acc[x][c], make_float2(f, f));
          m[x] = mn;
          pwb[lane * G + x] = pw;
        }
      }
      // the K slot's reads are done: hand it to the copy engine again
      __syncwarp();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(n + NS, false);
      const bool vready =
          __all_sync(0xffffffffu, bar_wait(saddr(vbar), (uint32_t)n & 1u, abort));
      if (vready) v_landed = n + 1;
      if (ready && vready && count > 0) {
        auto vrow = [&](int rr, int off) {
          float vf[DL];
          lds_cols<T, DL>(vst + off, vf);
          const float* w = pwb + rr * G;
#pragma unroll
          for (int x = 0; x < G; ++x) {
            const float2 wx = make_float2(w[x], w[x]);
#pragma unroll
            for (int c = 0; c < DL / 2; ++c)
              acc[x][c] = __ffma2_rn(wx, make_float2(vf[2 * c], vf[2 * c + 1]), acc[x][c]);
          }
        };
        int rr = 0;
        for (; rr + 8 <= count; rr += 8) {
#pragma unroll
          for (int u = 0; u < 8; ++u) vrow(rr + u, rr * 128 + voff[u]);
        }
        for (; rr < count; ++rr) vrow(rr, swz(rr, lane * DL * (int)sizeof(T)));
      }
      // the V slot's reads are done: fetch the next block's V into it
      __syncwarp();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(n + 1, true);
    }
    // merge the warps
#pragma unroll
    for (int x = 0; x < G; ++x) {
      if (lane == 0) {
        wml[(warp * G + x) * 2] = m[x];
        wml[(warp * G + x) * 2 + 1] = l[x];
      }
#pragma unroll
      for (int c = 0; c < DL / 2; ++c)
        *reinterpret_cast<float2*>(wacc + (warp * G + x) * D + lane * DL + 2 * c) = acc[x][c];
    }
    __syncthreads();
    const size_t unit = (size_t)unit_i;
    const bool failed = *abort != 0;
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
      const int x = i / D, c = i % D;
      float M = -INFINITY;
      for (int w = 0; w < warps; ++w) M = fmaxf(M, wml[(w * G + x) * 2]);
      float L = 0.f, O = 0.f;
      if (M != -INFINITY) {
        for (int w = 0; w < warps; ++w) {
          const float mw = wml[(w * G + x) * 2];
          if (mw == -INFINITY) continue;
          const float f = ex2(mw - M);
          L += wml[(w * G + x) * 2 + 1] * f;
          O += wacc[(w * G + x) * D + c] * f;
        }
      }
      if (failed) M = __int_as_float(0x7fc00000);  // a stage never landed: the output reads NaN
      p.part_o[unit * G * D + i] = O;
      if (c == 0) p.part_ml[unit * G + x] = make_float2(M, L);
    }
  }
  // an aborting CTA lets the copies it issued land before it leaves
  for (int r = k_landed; r < k_issued; ++r) {
    const uint64_t t0 = global_ns();
    while (!bar_test(saddr(&kbars[r % NS]), (uint32_t)(r / NS) & 1u) && global_ns() - t0 < kWaitNs) {
    }
  }
  for (int r = v_landed; r < v_issued; ++r) {
    const uint64_t t0 = global_ns();
    while (!bar_test(saddr(vbar), (uint32_t)r & 1u) && global_ns() - t0 < kWaitNs) {
    }
  }
}

// Grid (nseq, H_q), D threads: merges the chunks of one sequence and head.
// Every thread reads every chunk's (max, sum) and its own column of every
// chunk's output, kCombineTile chunks at a time with all loads in flight,
// and merges them online (a running max, sum and output rescaled when the
// max grows), so the block needs no reduction and no barrier: the whole
// merge is about one round trip to memory per tile.
constexpr int kCombineTile = 32;

template <bool SH>
__global__ void decode_combine(const __grid_constant__ Params p) {
  pdl_trigger();
  pdl_wait();  // every chunk's partials are written
  const int s = blockIdx.x, hq = blockIdx.y, c = threadIdx.x;
  const Seq& S = p.seq[s];
  const int h = hq / p.g, x = hq % p.g;
  const int nch = (S.n + p.chunk - 1) / p.chunk;
  const size_t ustride = (size_t)p.H_kv * p.g;                       // between chunks
  const float2* ml = p.part_ml + ((size_t)S.chunk0 * p.H_kv + h) * p.g + x;  // chunk k: ml[k * ustride]
  const float* po = p.part_o + (((size_t)S.chunk0 * p.H_kv + h) * p.g + x) * p.d + c;
  float M = -INFINITY, L = 0.f, O = 0.f;
  for (int k0 = 0; k0 < nch; k0 += kCombineTile) {
    float2 v[kCombineTile];
    float o[kCombineTile];
#pragma unroll
    for (int k = 0; k < kCombineTile; ++k) {
      const bool in = k0 + k < nch;
      v[k] = in ? __ldcg(ml + (size_t)(k0 + k) * ustride) : make_float2(-INFINITY, 0.f);
      o[k] = in ? __ldcg(po + (size_t)(k0 + k) * ustride * p.d) : 0.f;
    }
    float tm = -INFINITY;
#pragma unroll
    for (int k = 0; k < kCombineTile; ++k) tm = fmaxf(tm, v[k].x);
    const float Mn = fmaxf(M, tm);
    if (Mn == -INFINITY) continue;  // no chunk with rows yet
    const float f0 = ex2(M - Mn);   // 0 while M = -inf (L and O are 0 then)
    L *= f0;
    O *= f0;
#pragma unroll
    for (int k = 0; k < kCombineTile; ++k) {
      const float f = v[k].x == -INFINITY ? 0.f : ex2(v[k].x - Mn);
      L = fmaf(v[k].y, f, L);
      O = fmaf(o[k], f, O);
    }
    M = Mn;
  }
  p.out[((size_t)(p.b0 + s) * p.H_q + hq) * p.d + c] = O / L;
  if constexpr (SH) {
    if (c == 0) p.sh_ml[(size_t)(p.b0 + s) * p.H_q + hq] = make_float2(M, L);
  }
}

int sm_count() {
  const DeviceInfo* di = current_device_info();
  return di ? di->sms : 148;
}

int max_smem_optin() {
  const DeviceInfo* di = current_device_info();
  return di ? di->smem_optin : 232448;
}

size_t smem_bytes(int warps, int stages, int D, int esize, int G) {
  return 1024 +  // room to start the slots on a 1024-byte boundary
         (size_t)warps * (stages + 1) * (slot_bytes(D, esize) + 8) +
         ((size_t)G * D + (size_t)warps * kRows * G + (size_t)warps * G * 2 +
          (size_t)warps * G * D) * sizeof(float) + 16;
}

using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiled encoder() {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(ptr);
  }
  return fn;
}

// Tensor map of a cache array [rows, heads, D]: boxes of 32 rows x 128 bytes
// of one head, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int D, int esize, int heads, long long rows) {
  EncodeTiled enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * esize, (cuuint64_t)D * esize * heads};
  cuuint32_t box[3] = {(cuuint32_t)(128 / esize), 1, (cuuint32_t)kRows};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
             const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Warps per CTA and K slots per warp: the most warps (the math, not the
// copies, sets the pace), then the most slots, that one CTA's shared memory
// holds (one CTA per SM).
bool kernel_shape(int D, int esize, int G, int& warps, int& stages) {
  static const int cand[][2] = {{8, 3}, {8, 2}, {6, 2}, {4, 3}, {4, 2}, {2, 3}, {2, 2}, {1, 2}};
  for (const auto& c : cand) {
    if (smem_bytes(c[0], c[1], D, esize, G) <= (size_t)max_smem_optin()) {
      warps = c[0];
      stages = c[1];
      return true;
    }
  }
  return false;
}

// Rows per unit: a multiple of the CTA's 32 * warps rows (whole blocks for
// every warp), at least kMinChunk, chosen so that the CTA with the most units
// does the least work -- ceil(units / grid) * chunk is smallest (ties: the
// longer chunk, fewer merges).
int choose_chunk(const int* n, int nseq, int H_kv, int grid, int gran) {
  int best = 0;
  long long best_cost = -1;
  for (int c = (kMinChunk + gran - 1) / gran * gran; c <= kMaxChunk; c += gran) {
    long long units = 0;
    for (int b = 0; b < nseq; ++b) units += (n[b] + c - 1) / c;
    units *= H_kv;
    const long long cost = (units + grid - 1) / grid * c;
    if (best_cost < 0 || cost <= best_cost) {
      best_cost = cost;
      best = c;
    }
    if (units <= grid) break;  // longer chunks only lengthen every CTA's unit
  }
  return best;
}

// Kernel shape, chunk and the chunk index of every sequence, for row counts n.
bool plan_units(Params& p, const int* n, int esize) {
  if (!kernel_shape(p.d, esize, p.g, p.warps, p.stages)) return false;
  const int gran = p.warps * kRows;
  p.chunk = choose_chunk(n, p.nseq, p.H_kv, sm_count(), gran);
  p.nbw = p.chunk / gran;
  int chunks = 0;
  for (int s = 0; s < p.nseq; ++s) {
    p.seq[s].chunk0 = chunks;
    chunks += (n[s] + p.chunk - 1) / p.chunk;
  }
  p.total_chunks = chunks;
  return true;
}

template <typename T, int D, bool SH = false>
cudaError_t launch_typed(const Params& p, cudaStream_t st) {
  const size_t smem = smem_bytes(p.warps, p.stages, D, (int)sizeof(T), p.g);
  const int units = p.total_chunks * p.H_kv;
  CUtensorMap tm_k, tm_v;
  if (!make_map(&tm_k, p.k, D, (int)sizeof(T), p.H_kv, p.rows_total) ||
      !make_map(&tm_v, p.v, D, (int)sizeof(T), p.H_kv, p.rows_total))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaSuccess;
  auto go = [&](auto kern) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) {
      const int grid = std::max(1, std::min(units, sm_count()));
      e = launch_pdl(kern, dim3(grid), dim3(p.warps * 32), smem, st, p, tm_k, tm_v);
      if (e == cudaSuccess) e = cudaGetLastError();
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
  e = launch_pdl(decode_combine<SH>, dim3(p.nseq, p.H_q), dim3(D), 0, st, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) count_launches(2);
  return e;
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
  p.rows_total = (long long)a.B * a.cap;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  for (int g0 = 0; g0 < a.B && e == cudaSuccess; g0 += dec::kGroup) {
    const int g1 = std::min(a.B, g0 + dec::kGroup);
    p.nseq = g1 - g0;
    p.b0 = g0;
    // chunks sized for the full cache: the rows in use are only known on the device
    int caps[dec::kGroup];
    for (int s = 0; s < p.nseq; ++s) {
      caps[s] = a.cap;
      p.seq[s].row0 = (long long)(g0 + s) * a.cap;
      p.seq[s].n = a.cap;
    }
    if (!dec::plan_units(p, caps, a.dtype == SNAPKV_BF16 ? 2 : 4)) {
      e = cudaErrorInvalidValue;
      break;
    }
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
  p.rows_total = 0;
  for (int b = 0; b < shape->batch; ++b) p.rows_total += lens_host[b];
  if (layout == SNAPKV_CACHE_SLOTS) p.rows_total = (long long)shape->batch * C;
  char* ws = static_cast<char*>(workspace);
  p.part_o = reinterpret_cast<float*>(ws);
  p.part_ml = reinterpret_cast<float2*>(
      ws + ((units_max * g * d * sizeof(float) + 255) & ~(size_t)255));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  long long packed_row = 0;
  int result = SNAPKV_OK;
  for (int g0 = 0; g0 < shape->batch && result == SNAPKV_OK; g0 += dec::kGroup) {
    const int g1 = std::min(shape->batch, g0 + dec::kGroup);
    p.nseq = g1 - g0;
    p.b0 = g0;
    for (int b = g0; b < g1; ++b) {
      dec::Seq& S = p.seq[b - g0];
      S.n = lens_host[b];
      S.row0 = layout == SNAPKV_CACHE_PACKED ? packed_row : (long long)b * C;
      packed_row += S.n;
    }
    if (!dec::plan_units(p, lens_host + g0, shape->dtype == SNAPKV_BF16 ? 2 : 4)) {
      result = SNAPKV_ERR_UNSUPPORTED;
      break;
    }
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
