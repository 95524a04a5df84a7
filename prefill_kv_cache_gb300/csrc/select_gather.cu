// Pooling, top-(C-W) selection and emission of the compressed cache.
//
// One thread-block cluster of kClusterCTAs CTAs handles one (sequence, KV
// head).  The CTAs split the prefix [0, P) into contiguous slices and:
//
//   1. pool the raw scores of their slice (stride 1, k//2 zeros of padding,
//      average divides by k, or maximum) -- jisaku.com glossary "SnapKV",
//      "Pooling for Robustness"; hotpaper.ai summary of "SnapKV: LLM Knows
//      What You are Looking for Before Generation", "기술적 접근법";
//   2. find the exact n-th largest pooled value T by a three-digit radix
//      select over the fp32 bit patterns (scores are >= 0, so the unsigned
//      patterns order like the values); per-digit histograms are merged
//      through distributed shared memory;
//   3. keep every position with a value above T and the lowest-positioned
//      `need` positions equal to T (ties go to the lower position), in
//      ascending order, via per-CTA counts and block prefix scans -- no sort;
//   4. copy the kept K and V rows, then the W window rows, into the
//      compressed cache with 16-byte vector loads and stores
//      (glossary, algorithm flow steps 3-4).
//
// A sequence with L <= C keeps all its rows; its cluster only copies.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math.h>

#include "plan.h"

namespace cg = cooperative_groups;

namespace snapkv {

constexpr int kWarps = kSelectThreads / 32;
static_assert(kMaxRows < kSelectThreads, "window rows are copied in one pass");

__device__ __forceinline__ int block_excl_scan(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int s = wsum[w];
    if (w < warp) before += s;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return before + x - v;
}

__device__ __forceinline__ int block_flag_scan(bool f, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, f);
  if (lane == 0) wsum[warp] = __popc(bal);
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int s = wsum[w];
    if (w < warp) before += s;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return before + __popc(bal & ((1u << lane) - 1u));
}

// Copy `cnt` rows: source position pos[i] of the sequence -> output slot
// slot0 + i (or slot = position when slot0 < 0), K and V, 16 B per access.
__device__ __forceinline__ void copy_rows(const Plan& p, const SeqInfo& S, int h,
                                          const int* pos, int cnt, int slot0, int vecs) {
  const uint4* kin = static_cast<const uint4*>(p.k);
  const uint4* vin = static_cast<const uint4*>(p.v);
  uint4* kout = static_cast<uint4*>(p.out_k);
  uint4* vout = static_cast<uint4*>(p.out_v);
  for (int e = threadIdx.x; e < cnt * vecs; e += blockDim.x) {
    const int it = e / vecs, vv = e % vecs;
    const int src_pos = pos[it];
    const int slot = slot0 < 0 ? src_pos : slot0 + it;
    const size_t src = ((size_t)(S.row0 + src_pos) * p.H_kv + h) * vecs + vv;
    const size_t dst = (((size_t)S.b * p.C + slot) * p.H_kv + h) * vecs + vv;
    kout[dst] = __ldcs(kin + src);
    vout[dst] = __ldcs(vin + src);
  }
}

__global__ void __cluster_dims__(kClusterCTAs, 1, 1) __launch_bounds__(kSelectThreads, 1)
select_gather(const __grid_constant__ Plan p, int cache_floats) {
  extern __shared__ __align__(16) float cache[];
  __shared__ unsigned hist[2048];
  __shared__ unsigned merged[2048];
  __shared__ int wsum[kWarps];
  __shared__ int sel_pos[kSelectThreads];
  __shared__ int sh_digit, sh_above;
  __shared__ int sh_cnt[2];

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int CS = kClusterCTAs;
  const int t = threadIdx.x;
  const int unit = blockIdx.y;
  const int s = unit / p.H_kv, h = unit % p.H_kv;
  const SeqInfo& S = p.seq[s];
  const int vecs = p.d * (p.dtype == 0 ? 2 : 4) / 16;
  int32_t* idx_out = p.out_idx + ((size_t)S.b * p.H_kv + h) * p.C;

  if (!S.scored) {
    // L <= C: slots 0..L-1 take positions 0..L-1, the rest index -1 and zeros.
    const int per = (p.C + CS - 1) / CS;
    const int a = min(p.C, rank * per), e = min(p.C, a + per);
    for (int slot = a + t; slot < e; slot += blockDim.x) idx_out[slot] = slot < S.L ? slot : -1;
    uint4* kout = static_cast<uint4*>(p.out_k);
    uint4* vout = static_cast<uint4*>(p.out_v);
    const uint4* kin = static_cast<const uint4*>(p.k);
    const uint4* vin = static_cast<const uint4*>(p.v);
    for (int x = t; x < (e - a) * vecs; x += blockDim.x) {
      const int slot = a + x / vecs, vv = x % vecs;
      const size_t dst = (((size_t)S.b * p.C + slot) * p.H_kv + h) * vecs + vv;
      if (slot < S.L) {
        const size_t src = ((size_t)(S.row0 + slot) * p.H_kv + h) * vecs + vv;
        kout[dst] = __ldcs(kin + src);
        vout[dst] = __ldcs(vin + src);
      } else {
        kout[dst] = make_uint4(0, 0, 0, 0);
        vout[dst] = make_uint4(0, 0, 0, 0);
      }
    }
    return;
  }

  const int P = S.P, n = p.n, r = p.kp / 2;
  const int Sz = (P + CS - 1) / CS;
  const int j0 = min(P, rank * Sz), j1 = min(P, j0 + Sz);
  const int cnt_local = j1 - j0;
  const bool use_cache = cnt_local <= cache_floats;
  const float* raw = p.raw + S.score0 + (size_t)h * P;
  float* pooled = p.pooled + S.score0 + (size_t)h * P;

  // 1. pooling of this CTA's slice
  for (int j = j0 + t; j < j1; j += blockDim.x) {
    float acc = 0.f, mx = -INFINITY;
    for (int tt = j - r; tt <= j + r; ++tt) {
      const float x = (tt >= 0 && tt < P) ? __ldcg(raw + tt) : 0.f;
      acc += x;
      mx = fmaxf(mx, x);
    }
    const float v = p.pool == 0 ? acc / (float)p.kp : mx;
    pooled[j] = v;
    if (use_cache) cache[j - j0] = v;
  }
  __syncthreads();
  const float* vals = use_cache ? cache : pooled + j0;

  if (n > 0) {
    // 2. radix select of the n-th largest value (digits 11/11/10 bits)
    unsigned prefix = 0, mask = 0;
    int need = n;
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const int nb = pass == 2 ? 1024 : 2048;
      for (int b = t; b < 2048; b += blockDim.x) hist[b] = 0;
      __syncthreads();
      for (int j = t; j < cnt_local; j += blockDim.x) {
        const unsigned u = __float_as_uint(use_cache ? vals[j] : __ldcg(vals + j));
        if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & (nb - 1)], 1u);
      }
      cluster.sync();
      for (int b = t; b < nb; b += blockDim.x) {
        unsigned sum = 0;
        for (int q = 0; q < CS; ++q) sum += cluster.map_shared_rank(hist, q)[b];
        merged[b] = sum;
      }
      cluster.sync();
      // digit D with count(> D) < need <= count(>= D); bins scanned from the top
      int local[4], lsum = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int rb = 4 * t + q;
        local[q] = rb < nb ? (int)merged[nb - 1 - rb] : 0;
        lsum += local[q];
      }
      int total;
      const int excl = block_excl_scan(lsum, wsum, &total);
      if (excl < need && need <= excl + lsum) {
        int cum = excl;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (cum + local[q] >= need) {
            sh_digit = nb - 1 - (4 * t + q);
            sh_above = cum;
            break;
          }
          cum += local[q];
        }
      }
      __syncthreads();
      need -= sh_above;
      prefix |= (unsigned)sh_digit << shift;
      mask |= (unsigned)(nb - 1) << shift;
      __syncthreads();
    }
    const unsigned T = prefix;

    // 3. per-CTA counts above / equal to T, exchanged across the cluster
    int my_gt = 0, my_eq = 0;
    for (int j = t; j < cnt_local; j += blockDim.x) {
      const unsigned u = __float_as_uint(use_cache ? vals[j] : __ldcg(vals + j));
      my_gt += u > T;
      my_eq += u == T;
    }
    int tot_gt, tot_eq;
    block_excl_scan(my_gt, wsum, &tot_gt);
    block_excl_scan(my_eq, wsum, &tot_eq);
    if (t == 0) {
      sh_cnt[0] = tot_gt;
      sh_cnt[1] = tot_eq;
    }
    cluster.sync();
    int eq_before = 0, out_before = 0, eq_acc = 0;
    for (int q = 0; q < CS; ++q) {
      const int* rc = cluster.map_shared_rank(sh_cnt, q);
      const int g_ = rc[0], e_ = rc[1];
      const int take = min(max(need - eq_acc, 0), e_);
      if (q < rank) {
        out_before += g_ + take;
        eq_before += e_;
      }
      eq_acc += e_;
    }
    cluster.sync();  // nobody leaves while others still read its counts

    // ascending compaction of the slice, chunk by chunk, with the row copies
    int running = 0;
    for (int base = 0; base < cnt_local; base += blockDim.x) {
      const int jj = base + t;
      const bool in = jj < cnt_local;
      const unsigned u = in ? __float_as_uint(use_cache ? vals[jj] : __ldcg(vals + jj)) : 0u;
      const bool gt = in && u > T;
      const bool eq = in && u == T;
      int chunk_eq, chunk_sel;
      const int eq_rank = block_flag_scan(eq, wsum, &chunk_eq);
      const bool sel = gt || (eq && eq_before + eq_rank < need);
      const int pos = block_flag_scan(sel, wsum, &chunk_sel);
      // slots past n would belong to the window block: never written from here
      const int room = max(0, min(chunk_sel, n - (out_before + running)));
      if (sel && pos < room) {
        idx_out[out_before + running + pos] = j0 + jj;
        sel_pos[pos] = j0 + jj;
      }
      eq_before += chunk_eq;
      __syncthreads();
      copy_rows(p, S, h, sel_pos, room, out_before + running, vecs);
      running += chunk_sel;
      __syncthreads();
    }
  }

  // 4. the window rows: slots n .. C-1 take positions P .. L-1
  // (W <= kMaxRows < kSelectThreads, so one pass covers the window)
  if (rank == CS - 1) {
    for (int w = t; w < p.W; w += blockDim.x) {
      idx_out[n + w] = P + w;
      sel_pos[w] = P + w;
    }
    __syncthreads();
    copy_rows(p, S, h, sel_pos, p.W, n, vecs);
  }
}

int launch_select_gather(const Plan& p, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int max_slice = 0;
  for (int s = 0; s < p.nseq; ++s)
    if (p.seq[s].scored) max_slice = max(max_slice, (p.seq[s].P + kClusterCTAs - 1) / kClusterCTAs);
  const int cache_floats = min(max_slice, 48 * 1024);
  const size_t smem = (size_t)cache_floats * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(select_gather, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(smem > 0 ? smem : 1));
  if (e != cudaSuccess) return e;
  dim3 grid(kClusterCTAs, p.nseq * p.H_kv);
  select_gather<<<grid, kSelectThreads, smem, st>>>(p, cache_floats);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace snapkv
