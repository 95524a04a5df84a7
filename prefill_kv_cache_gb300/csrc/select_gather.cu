// Pooling, top-(C-W) selection and emission of the compressed cache.
//
// One thread-block cluster handles one (sequence, KV head).  Its size is a
// power of two chosen per launch: large enough that all units together fill
// the GPU and that each CTA's slice fits its shared-memory staging, at most 16
// (8 where the GPU does not allow non-portable cluster sizes).  The CTAs split
// the prefix [0, P) into contiguous slices and:
//
//   1. pool the raw scores of their slice (stride 1, k//2 zeros of padding,
//      average divides by k, or maximum) -- jisaku.com glossary "SnapKV",
//      "Pooling for Robustness"; hotpaper.ai summary of "SnapKV: LLM Knows
//      What You are Looking for Before Generation", "기술적 접근법".  The
//      raw scores are staged in shared memory tile by tile, the pooled slice
//      stays there for the next steps;
//   2. find the exact n-th largest pooled value T by a radix select over the
//      fp32 bit patterns (scores are >= 0, so the unsigned patterns order
//      like the values).  The first digit (11 bits) is histogrammed over the
//      cluster through distributed shared memory: each CTA adds its counts
//      into the owners' bins, then every CTA reads the reduced bins.  The
//      values of the threshold bin are then gathered on rank 0, which
//      finishes the select over them alone (two more digits) and hands every
//      CTA the threshold and its counts; a bin too large to gather takes the
//      two digits over the cluster instead;
//   3. keep every position with a value above T and the lowest-positioned
//      `need` positions equal to T (ties go to the lower position), in
//      ascending order, via per-CTA counts and block prefix scans -- no sort;
//   4. write the kept positions, then the W window positions, to the index
//      output; after a cluster barrier every CTA copies an equal share of
//      the C output rows (K and V) by bulk copies staged in shared memory
//      (glossary, algorithm flow steps 3-4).
//
// A sequence with L <= C keeps all its rows; its cluster only copies.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math.h>

#include <algorithm>
#include <mutex>

#include "pdl.cuh"
#include "plan.h"

namespace cg = cooperative_groups;

namespace snapkv {

constexpr int kWarps = kSelectThreads / 32;
constexpr int kPer = 4;                        // consecutive positions per thread per pass
constexpr int kChunk = kSelectThreads * kPer;  // positions per compaction pass
constexpr int kMaxCluster = 16;
constexpr int kPoolTile = 8192;                // raw scores staged per pooling step
constexpr int kLd = 16;                        // independent global loads in flight per thread
constexpr int kStageFloats = 44 * 1024;         // dynamic shared memory, in floats
// values of the first digit's threshold bin that rank 0 selects from alone
// (one word each, in its raw-staging area, which holds at least kPoolTile)
constexpr int kCandCap = kPoolTile;
// pooled values per CTA below which a smaller cluster costs little latency
constexpr int kShortSlice = 4096;
static_assert(kMaxRows < kChunk, "window rows are copied in one pass");

// Floats of the raw-score staging area for pooling half-width r: the tile,
// its halo, rounded to whole float4 plus one float4 run of slack that the
// vectorised window reads may touch past the last output.
__host__ __device__ constexpr int raw_span(int r) { return ((kPoolTile + 2 * r + 3) & ~3) + 16; }

// Pools m outputs from the staged raw scores: output x covers
// sraw[x .. x + KP - 1] (the tile starts r positions left of its first
// output).  Each thread takes 4 consecutive outputs, reads their KP + 3
// inputs as float4 and sums / maxes them left to right -- the same order,
// hence the same fp32 result, for every output.
template <int KP, bool AVG>
__device__ __forceinline__ void pool_run(const float* sraw, float* spool, float* gout, int m) {
  constexpr int NV = (KP + 3 + 3) / 4;  // float4 reads per 4 outputs
  for (int x = 4 * (int)threadIdx.x; x < m; x += 4 * (int)blockDim.x) {
    float w[4 * NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const float4 f = *reinterpret_cast<const float4*>(sraw + x + 4 * v);
      w[4 * v] = f.x;
      w[4 * v + 1] = f.y;
      w[4 * v + 2] = f.z;
      w[4 * v + 3] = f.w;
    }
    float o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float acc = AVG ? 0.f : -INFINITY;
#pragma unroll
      for (int q = 0; q < KP; ++q) acc = AVG ? acc + w[i + q] : fmaxf(acc, w[i + q]);
      o[i] = AVG ? acc / (float)KP : acc;
    }
    if (x + 3 < m) {
      *reinterpret_cast<float4*>(spool + x) = make_float4(o[0], o[1], o[2], o[3]);
#pragma unroll
      for (int i = 0; i < 4; ++i) gout[x + i] = o[i];
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (x + i < m) {
          spool[x + i] = o[i];
          gout[x + i] = o[i];
        }
    }
  }
}

template <bool AVG>
__device__ bool pool_dispatch(int kp, const float* sraw, float* spool, float* gout, int m) {
  switch (kp) {
    case 1: pool_run<1, AVG>(sraw, spool, gout, m); return true;
    case 3: pool_run<3, AVG>(sraw, spool, gout, m); return true;
    case 5: pool_run<5, AVG>(sraw, spool, gout, m); return true;
    case 7: pool_run<7, AVG>(sraw, spool, gout, m); return true;
    case 9: pool_run<9, AVG>(sraw, spool, gout, m); return true;
    case 11: pool_run<11, AVG>(sraw, spool, gout, m); return true;
    case 13: pool_run<13, AVG>(sraw, spool, gout, m); return true;
    case 15: pool_run<15, AVG>(sraw, spool, gout, m); return true;
    case 17: pool_run<17, AVG>(sraw, spool, gout, m); return true;
    case 19: pool_run<19, AVG>(sraw, spool, gout, m); return true;
    case 21: pool_run<21, AVG>(sraw, spool, gout, m); return true;
    default: return false;
  }
}

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

// Calls f(x, pat(x)) for x = xa .. xb - 1 in order.  Not unrolled: every
// pass of this kernel runs once per CTA, so its code is fetched cold, and
// short loop bodies cost less in instruction fetch than the loads they could
// batch (measured: unrolling by 8 made the selection ~2 us slower).
template <typename Pat, typename F>
__device__ __forceinline__ void walk(Pat pat, int xa, int xb, F f) {
#pragma unroll 1
  for (int x = xa; x < xb; ++x) f(x, pat(x));
}

// Histogram of one radix digit: for x in [xa, xb) with (pat(x) & mask) ==
// prefix, bin (pat(x) >> shift) & (nb - 1) of h gains one.  A thread walks
// consecutive positions and adds each run of equal digits with one atomic
// (neighbouring pooled scores mostly share their leading digit, so this
// avoids most of the same-address conflicts of one atomic per value).
template <typename Pat>
__device__ __forceinline__ void run_hist(Pat pat, int xa, int xb, unsigned prefix, unsigned mask,
                                         int shift, int nb, unsigned* h) {
  int rb = -1;
  unsigned rc = 0;
  walk(pat, xa, xb, [&](int, unsigned u) {
    const int bin = (u & mask) == prefix ? (int)((u >> shift) & (unsigned)(nb - 1)) : -1;
    if (bin != rb) {
      if (rb >= 0) atomicAdd(&h[rb], rc);
      rb = bin;
      rc = 0;
    }
    ++rc;
  });
  if (rb >= 0) atomicAdd(&h[rb], rc);
}

// Exclusive block scans of two values at once; returns a's prefix, writes
// b's prefix and both totals.
__device__ __forceinline__ int block_excl_scan2(int a, int b, int* wsum, int* a_total,
                                                int* b_excl, int* b_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = a, y = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int xa = __shfl_up_sync(0xffffffffu, x, o);
    const int ya = __shfl_up_sync(0xffffffffu, y, o);
    if (lane >= o) {
      x += xa;
      y += ya;
    }
  }
  if (lane == 31) {
    wsum[warp] = x;
    wsum[kWarps + warp] = y;
  }
  __syncthreads();
  int xb = 0, yb = 0, xt = 0, yt = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int sx = wsum[w], sy = wsum[kWarps + w];
    if (w < warp) {
      xb += sx;
      yb += sy;
    }
    xt += sx;
    yt += sy;
  }
  __syncthreads();
  *a_total = xt;
  *b_total = yt;
  *b_excl = yb + y - b;
  return xb + x - a;
}

// The digit D of the nb-bin histogram h with count(> D) < need <= count(>= D),
// bins scanned from the top (4 per thread, nb <= 4 * blockDim.x).  Every
// thread of the block calls it; *digit, *above = count(> D) and *in_bin =
// count(D) are valid in all threads on return.
__device__ __forceinline__ void top_digit(const unsigned* h, int nb, int need, int* wsum, int* digit,
                                          int* above, int* in_bin) {
  const int t = threadIdx.x;
  int local[4], lsum = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int rb = 4 * t + q;
    local[q] = rb < nb ? (int)h[nb - 1 - rb] : 0;
    lsum += local[q];
  }
  int total;
  const int excl = block_excl_scan(lsum, wsum, &total);
  if (excl < need && need <= excl + lsum) {
    int cum = excl;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (cum + local[q] >= need) {
        *digit = nb - 1 - (4 * t + q);
        *above = cum;
        *in_bin = local[q];
        break;
      }
      cum += local[q];
    }
  }
  __syncthreads();
}

// Copy `cnt` rows: source position pos[i] of the sequence (KV head sh) ->
// output slot slot0 + i (output head oh), K and V, 16 B per access.
__device__ __forceinline__ void copy_rows(const Plan& p, const SeqInfo& S, int sh, int oh,
                                          const int* pos, int cnt, int slot0, int vecs) {
  const uint4* kin = static_cast<const uint4*>(p.k);
  const uint4* vin = static_cast<const uint4*>(p.v);
  uint4* kout = static_cast<uint4*>(p.out_k);
  uint4* vout = static_cast<uint4*>(p.out_v);
  // kU independent 16-byte loads of K and of V in flight per thread
  constexpr int kU = 4;
  const int total = cnt * vecs;
  for (int e0 = threadIdx.x; e0 < total; e0 += kU * blockDim.x) {
    uint4 kv[kU], vv_[kU];
    size_t dst[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int e = e0 + u * blockDim.x;
      if (e < total) {
        const int it = e / vecs, vv = e % vecs;
        const size_t src = ((size_t)(S.row0 + pos[it]) * p.H_kv + sh) * vecs + vv;
        dst[u] = (((size_t)S.b * p.C + slot0 + it) * p.out_heads + oh) * vecs + vv;
        kv[u] = __ldcs(kin + src);
        vv_[u] = __ldcs(vin + src);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (e0 + u * blockDim.x < total) {
        kout[dst[u]] = kv[u];
        vout[dst[u]] = vv_[u];
      }
    }
  }
}

// ---- bulk (TMA) row copies through shared memory ----

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Bounded wait for phase `parity` of barrier b (2 s); false on expiry, with
// the status word set.
__device__ bool bar_wait(uint64_t* b, uint32_t parity, int* status) {
  uint64_t t0 = 0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (;;) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred q;\n mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n"
        " selp.b32 %0, 1, 0, q;\n}\n"
        : "=r"(done)
        : "r"(saddr(b)), "r"(parity)
        : "memory");
    if (done) return true;
    uint64_t t1;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
    if (t1 - t0 > 2000000000ull) {
      atomicExch(status, kDevTimeout);
      return false;
    }
  }
}

// Copies the K and V rows of sequence positions pos[0..cnt) (KV head sh) to
// output slots slot0.. of output head oh: batches of rows are fetched into `stage` by bulk
// copies that complete on `bar`, then written out by bulk stores.  Every
// thread of the block calls it.  False if a wait expired.
__device__ bool bulk_copy_rows(const Plan& p, const SeqInfo& S, int sh, int oh, const int* pos, int cnt,
                               int slot0, int row_bytes, unsigned char* stage, int stage_bytes,
                               uint64_t* bar, uint32_t& phase) {
  const int per = stage_bytes / (2 * row_bytes);  // rows per batch (K and V)
  const char* kin = static_cast<const char*>(p.k);
  const char* vin = static_cast<const char*>(p.v);
  char* kout = static_cast<char*>(p.out_k);
  char* vout = static_cast<char*>(p.out_v);
  // the stage held generic-proxy data before: order it before async writes
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  bool ok = true;
  for (int i0 = 0; i0 < cnt && ok; i0 += per) {
    const int m = min(per, cnt - i0);
    if (threadIdx.x == 0)
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)),
                   "r"(2 * m * row_bytes)
                   : "memory");
    __syncthreads();
    for (int i = threadIdx.x; i < 2 * m; i += blockDim.x) {
      const int row = i >> 1;
      const char* src = ((i & 1) ? vin : kin) +
                        ((size_t)(S.row0 + pos[i0 + row]) * p.H_kv + sh) * row_bytes;
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
              "r"(saddr(stage + (size_t)i * row_bytes)),
          "l"(src), "r"(row_bytes), "r"(saddr(bar))
          : "memory");
    }
    ok = __syncthreads_and(bar_wait(bar, phase, p.status));
    if (!ok) {  // give the copies in flight one more bounded wait before leaving
      bar_wait(bar, phase, p.status);
      break;
    }
    phase ^= 1;
    {
      for (int i = threadIdx.x; i < 2 * m; i += blockDim.x) {
        const int row = i >> 1;
        char* dst = ((i & 1) ? vout : kout) +
                    (((size_t)S.b * p.C + slot0 + i0 + row) * p.out_heads + oh) * row_bytes;
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                     "r"(saddr(stage + (size_t)i * row_bytes)), "r"(row_bytes)
                     : "memory");
      }
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // stage reusable
    }
    __syncthreads();
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  return ok;
}

__global__ void __launch_bounds__(kSelectThreads, 2)
select_gather(const __grid_constant__ Plan p, int cap_floats) {
  extern __shared__ __align__(16) float dyn[];  // [raw staging tile + halo][pooled slice]
  // cluster-wide digit histograms, one per radix digit: CTA r holds bins
  // [r * own, (r + 1) * own) of each, and every CTA adds its values' counts
  // into the owners' bins through distributed shared memory
  __shared__ unsigned hb[3][2048];
  __shared__ unsigned hl[2048];  // this CTA's counts of the current digit, then all bins
  __shared__ int wsum[2 * kWarps];
  __shared__ int sel_pos[kChunk];
  __shared__ int sh_digit, sh_above, sh_in_bin, sh_base;
  __shared__ int cl_cnt[2 * kMaxCluster];        // (above, equal) per CTA, on rank 0
  __shared__ int cq[2 * kMaxCluster];            // rank 0: candidates above / equal per CTA
  __shared__ int cand_n;                         // rank 0: candidates gathered
  __shared__ int sel_info[4];                    // T, need, out_before, eq_before from rank 0
  __shared__ __align__(8) uint64_t bulk_bar;

  cg::cluster_group cluster = cg::this_cluster();
  // launched as a programmatic dependent of the score kernel: everything
  // below reads what that kernel wrote
  pdl_wait();
  const int rank = (int)cluster.block_rank();
  const int CS = (int)cluster.num_blocks();
  const int t = threadIdx.x;
  const int unit = blockIdx.y;
  const int s = unit / p.out_heads, oh = unit % p.out_heads;  // output head
  const int h = oh / p.head_div;                                // its KV head
  const SeqInfo& S = p.seq[s];
  const int vecs = p.d * (p.dtype == 0 ? 2 : 4) / 16;
  const int row_bytes = vecs * 16;
  uint32_t bulk_phase = 0;
  if (t == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&bulk_bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  int32_t* idx_out = p.out_idx + ((size_t)S.b * p.out_heads + oh) * p.C;

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
      const size_t dst = (((size_t)S.b * p.C + slot) * p.out_heads + oh) * vecs + vv;
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
  // the digit histograms start at zero in every CTA before any CTA adds to
  // them: zero, arrive on the cluster barrier now, wait after pooling
  for (int b = t; b < 3 * 2048; b += blockDim.x) (&hb[0][0])[b] = 0u;
  if (t < 2 * kMaxCluster) cq[t] = 0;
  if (t == 0) cand_n = 0;
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  const int Sz = (P + CS - 1) / CS;
  const int j0 = min(P, rank * Sz), j1 = min(P, j0 + Sz);
  const int cnt = j1 - j0;
  const float* raw = p.raw + S.score0 + (size_t)oh * P;
  float* pooled = p.pooled + S.score0 + (size_t)oh * P;
  const bool in_smem = raw_span(r) + cnt <= cap_floats;
  float* sraw = dyn;
  float* spool = dyn + raw_span(r);

  // 1. pooling of this CTA's slice (zero padding outside [0, P)), the raw
  //    scores staged in shared memory one tile (plus halo) at a time
  if (in_smem) {
    for (int x0 = 0; x0 < cnt; x0 += kPoolTile) {
      const int m = min(kPoolTile, cnt - x0);
      for (int x1 = t; x1 < m + 2 * r; x1 += kLd * blockDim.x) {  // kLd loads in flight
        float vl[kLd];
#pragma unroll
        for (int u = 0; u < kLd; ++u) {
          const int x = x1 + u * blockDim.x;
          const int jj = j0 + x0 - r + x;
          vl[u] = (x < m + 2 * r && jj >= 0 && jj < P) ? __ldcg(raw + jj) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kLd; ++u)
          if (x1 + u * blockDim.x < m + 2 * r) sraw[x1 + u * blockDim.x] = vl[u];
      }
      __syncthreads();
      const bool done = p.pool == 0
                            ? pool_dispatch<true>(p.kp, sraw, spool + x0, pooled + j0 + x0, m)
                            : pool_dispatch<false>(p.kp, sraw, spool + x0, pooled + j0 + x0, m);
      if (!done) {  // other window sizes
        for (int x = t; x < m; x += blockDim.x) {
          float acc = 0.f, mx = -INFINITY;
          for (int q = 0; q <= 2 * r; ++q) {
            const float v = sraw[x + q];
            acc += v;
            mx = fmaxf(mx, v);
          }
          const float v = p.pool == 0 ? acc / (float)p.kp : mx;
          spool[x0 + x] = v;
          pooled[j0 + x0 + x] = v;
        }
      }
      __syncthreads();
    }
  } else {
    for (int j = j0 + t; j < j1; j += blockDim.x) {
      float acc = 0.f, mx = -INFINITY;
      for (int tt = j - r; tt <= j + r; ++tt) {
        const float v = (tt >= 0 && tt < P) ? __ldcg(raw + tt) : 0.f;
        acc += v;
        mx = fmaxf(mx, v);
      }
      pooled[j] = p.pool == 0 ? acc / (float)p.kp : mx;
    }
  }
  __syncthreads();
  const float* vals = in_smem ? spool : pooled + j0;  // this CTA's pooled slice

  // the cluster barrier armed before pooling: every CTA's histograms are zero
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  // positions per thread for the histogram, counting and compaction passes:
  // an odd stride, so that the threads of a warp reading their i-th
  // positions hit 32 different shared-memory banks
  const int per = ((cnt + (int)blockDim.x - 1) / (int)blockDim.x) | 1;
  const int xa = min(cnt, t * per), xb = min(cnt, xa + per);      // this thread's range
  int out_before = 0, eq_before = 0, need = n;
  unsigned T = 0;
  if (n > 0) {
    auto pat = [&](int x) { return __float_as_uint(vals[x]); };
    // 2. radix select of the n-th largest value over the fp32 patterns:
    //    digits of 11 (bits 31..21), 11 and 10 bits, each histogram summed
    //    over the cluster with one cluster barrier.  After the first digit,
    //    when the threshold bin holds at most kCandCap values, the rest of
    //    the select runs on rank 0 over those candidates alone (2b).
    unsigned prefix = 0, mask = 0;
    bool gathered = false;
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const int nb = pass == 2 ? 1024 : 2048;
      const int own = nb / CS;  // bins held by each CTA
      unsigned* hd = hb[pass];
      for (int b = t; b < nb; b += blockDim.x) hl[b] = 0u;
      __syncthreads();
      run_hist(pat, xa, xb, prefix, mask, shift, nb, hl);
      __syncthreads();
      // this CTA's non-empty bins go to their owners
      for (int b = t; b < nb; b += blockDim.x) {
        const unsigned c = hl[b];
        if (c) atomicAdd(cluster.map_shared_rank(hd, b / own) + b, c);
      }
      cluster.sync();
      for (int b1 = t; b1 < nb; b1 += 4 * blockDim.x) {
        unsigned m4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int b = b1 + u * blockDim.x;
          m4[u] = b < nb ? cluster.map_shared_rank(hd, b / own)[b] : 0u;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (b1 + u * blockDim.x < nb) hl[b1 + u * blockDim.x] = m4[u];
      }
      __syncthreads();
      top_digit(hl, nb, need, wsum, &sh_digit, &sh_above, &sh_in_bin);
      need -= sh_above;
      prefix |= (unsigned)sh_digit << shift;
      mask |= (unsigned)(nb - 1) << shift;
      if (pass == 0 && sh_in_bin <= kCandCap) {  // the same decision in every CTA
        gathered = true;
        // hl (read by top_digit before its closing barrier) starts rank 0's
        // candidate histogram at zero; the second digit uses hb[1], which
        // no CTA touches on this path
        for (int b = t; b < nb; b += blockDim.x) hl[b] = 0u;
        break;
      }
    }

    if (gathered) {
      // 2b. the values of the threshold bin, packed as (CTA rank << 21 | low
      //     21 bits), go to rank 0's raw-staging area (free after pooling);
      //     the values above the bin are counted per CTA
      const unsigned D1 = prefix >> 21;
      unsigned* cand = reinterpret_cast<unsigned*>(sraw);
      int nc = 0, na = 0;
      walk(pat, xa, xb, [&](int, unsigned u) {
        nc += (u >> 21) == D1;
        na += (u >> 21) > D1;
      });
      int tot_c, tot_a, excl_a;
      const int excl_c = block_excl_scan2(nc, na, wsum, &tot_c, &excl_a, &tot_a);
      if (t == 0) {
        sh_base = atomicAdd(cluster.map_shared_rank(&cand_n, 0), tot_c);
        cluster.map_shared_rank(cl_cnt, 0)[2 * rank] = tot_a;
      }
      __syncthreads();
      unsigned* dst = cluster.map_shared_rank(cand, 0) + sh_base + excl_c;
      walk(pat, xa, xb, [&](int, unsigned u) {
        if ((u >> 21) == D1) *dst++ = ((unsigned)rank << 21) | (u & 0x1FFFFFu);
      });
      cluster.sync();
      if (rank == 0) {
        // the last two digits (bits 20..10, 9..0) over the candidates alone
        const int nc_all = cand_n;
        const int cper = ((nc_all + (int)blockDim.x - 1) / (int)blockDim.x) | 1;
        const int ca = min(nc_all, t * cper), cb = min(nc_all, ca + cper);
        auto low = [&](int i) { return cand[i] & 0x1FFFFFu; };
        unsigned p2 = 0, m2 = 0;
        for (int pass = 0; pass < 2; ++pass) {
          const int shift = pass == 0 ? 10 : 0;
          const int nb = pass == 0 ? 2048 : 1024;
          unsigned* hc = pass == 0 ? hl : hb[1];  // both zero here
          run_hist(low, ca, cb, p2, m2, shift, nb, hc);
          __syncthreads();
          top_digit(hc, nb, need, wsum, &sh_digit, &sh_above, &sh_in_bin);
          need -= sh_above;
          p2 |= (unsigned)sh_digit << shift;
          m2 |= (unsigned)(nb - 1) << shift;
        }
        // candidates above / equal to the threshold, per source CTA (runs of
        // one key added at once: a CTA's candidates are contiguous)
        int rk = -1, rc = 0;
        walk([&](int i) { return cand[i]; }, ca, cb, [&](int, unsigned w) {
          const unsigned v = w & 0x1FFFFFu;
          const int key = v > p2 ? 2 * (int)(w >> 21) : (v == p2 ? 2 * (int)(w >> 21) + 1 : -1);
          if (key != rk) {
            if (rk >= 0) atomicAdd(&cq[rk], rc);
            rk = key;
            rc = 0;
          }
          ++rc;
        });
        if (rk >= 0) atomicAdd(&cq[rk], rc);
        __syncthreads();
        if (t < CS) {  // CTA t's kept values before its own, and equal values before its own
          int eq_acc = 0, ob = 0, eb = 0;
          for (int q = 0; q < CS; ++q) {
            const int g_ = cl_cnt[2 * q] + cq[2 * q], e_ = cq[2 * q + 1];
            const int take = min(max(need - eq_acc, 0), e_);
            if (q < t) {
              ob += g_ + take;
              eb += e_;
            }
            eq_acc += e_;
          }
          int* info = cluster.map_shared_rank(sel_info, t);
          info[0] = (int)(prefix | p2);
          info[1] = need;
          info[2] = ob;
          info[3] = eb;
        }
      }
      cluster.sync();
      T = (unsigned)sel_info[0];
      need = sel_info[1];
      out_before = sel_info[2];
      eq_before = sel_info[3];
    } else {
      T = prefix;
    }

    // 3. this thread's values above / equal to T, then across the CTA
    int gt = 0, eq = 0;
    walk(pat, xa, xb, [&](int, unsigned u) {
      gt += u > T;
      eq += u == T;
    });
    int my_gt, my_eq, excl_eq;
    const int excl_gt = block_excl_scan2(gt, eq, wsum, &my_gt, &excl_eq, &my_eq);
    if (!gathered) {
      // the CTA's counts go to rank 0, every CTA reads them all back
      if (t == 0) {
        int* dcl = cluster.map_shared_rank(cl_cnt, 0);
        dcl[2 * rank] = my_gt;
        dcl[2 * rank + 1] = my_eq;
      }
      cluster.sync();
      // every CTA's pair, fetched in parallel (one remote load per thread)
      if (t < 2 * CS) wsum[t] = cluster.map_shared_rank(cl_cnt, 0)[t];
      __syncthreads();
      int eq_acc = 0;
      for (int q = 0; q < CS; ++q) {
        const int g_ = wsum[2 * q], e_ = wsum[2 * q + 1];
        const int take = min(max(need - eq_acc, 0), e_);
        if (q < rank) {
          out_before += g_ + take;
          eq_before += e_;
        }
        eq_acc += e_;
      }
    }

    // 4. ascending compaction: a thread's kept positions go to consecutive
    //    slots after those of lower threads and lower CTAs; equal values are
    //    kept in position order while the cluster still needs them
    int slot = out_before + excl_gt + min(max(need - eq_before, 0), excl_eq);
    int eq_rank = eq_before + excl_eq;
    walk(pat, xa, xb, [&](int x, unsigned u) {
      const bool keep = u > T || (u == T && eq_rank < need);
      eq_rank += u == T;
      if (keep) {
        if (slot < n) idx_out[slot] = j0 + x;  // slots from n on belong to the window
        ++slot;
      }
    });
  }

  // 5. the window rows: slots n .. C-1 take positions P .. L-1
  if (rank == CS - 1)
    for (int w = t; w < p.W; w += blockDim.x) idx_out[n + w] = P + w;

  // 6. every CTA copies an equal share of the C output slots (kept rows
  //    cluster together, so the slices' own kept rows would be unbalanced),
  //    reading the positions back from the index output
  cluster.sync();
  const int share = (p.C + CS - 1) / CS;
  const int s0 = min(p.C, rank * share), s1 = min(p.C, s0 + share);
  // bulk copies read device memory only; host-resident V goes through plain loads
  const bool bulk = !p.v_zero_copy && cap_floats * 4 >= 2 * row_bytes;
  for (int c0 = s0; c0 < s1; c0 += kChunk) {
    const int m = min(kChunk, s1 - c0);
    __syncthreads();  // sel_pos free
    for (int i = t; i < m; i += blockDim.x) sel_pos[i] = __ldcg(idx_out + c0 + i);
    __syncthreads();
    if (bulk) {
      if (!bulk_copy_rows(p, S, h, oh, sel_pos, m, c0, row_bytes, reinterpret_cast<unsigned char*>(dyn),
                          cap_floats * 4, &bulk_bar, bulk_phase))
        break;
    } else {
      copy_rows(p, S, h, oh, sel_pos, m, c0, vecs);
    }
  }
}

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_cluster_mu;
int g_max_cluster[kMaxDevices] = {};  // per device: largest cluster size allowed (16 or 8)

size_t smem_for(int CS, int maxP, int kp) {
  const int slice = (maxP + CS - 1) / CS;
  const int need = raw_span(kp / 2) + slice;
  return (size_t)(need <= kStageFloats ? need : raw_span(kp / 2)) * sizeof(float);
}

// Clusters of CS CTAs (with `smem` dynamic bytes each) that fit on the GPU at once.
int max_active_clusters(int CS, size_t smem) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = CS;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(CS, 1);
  cfg.blockDim = dim3(kSelectThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, select_gather, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace

int launch_select_gather(const Plan& p, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaFuncSetAttribute(select_gather, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kStageFloats * (int)sizeof(float));
  if (e != cudaSuccess) return e;
  const DeviceInfo* di = current_device_info();
  int dev = 0;
  if (!di || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return cudaErrorUnknown;
  const int sms = di->sms;
  int max_cluster = 0;
  {
    std::lock_guard<std::mutex> lock(g_cluster_mu);
    if (g_max_cluster[dev] == 0) {
      int mc = 8;
      if (cudaFuncSetAttribute(select_gather, cudaFuncAttributeNonPortableClusterSizeAllowed,
                               1) == cudaSuccess &&
          max_active_clusters(kMaxCluster, 64 * 1024) > 0)
        mc = kMaxCluster;
      cudaGetLastError();
      g_max_cluster[dev] = mc;
    }
    max_cluster = g_max_cluster[dev];
  }
  // Cluster size: a power of two, large enough that all units together fill
  // the GPU and each slice fits the shared-memory staging, then halved while
  // the clusters would not all be resident at once (one wave).
  const int units = p.nseq * p.out_heads;
  int maxP = 0;
  for (int s = 0; s < p.nseq; ++s)
    if (p.seq[s].scored) maxP = max(maxP, p.seq[s].P);
  const int room = kStageFloats - raw_span(p.kp / 2);
  int CS = 1;
  while (CS < max_cluster && (units * CS < sms || (maxP + CS - 1) / CS > room)) CS *= 2;
  if (p.gpu_share > 1) {
    // several calls share the GPU: clusters only large enough to fill this
    // call's share, as long as every CTA's slice stays short (the selection's
    // passes cost in proportion to it)
    const int fill = std::max(1, sms / p.gpu_share);
    int cs = 1;
    while (cs < CS && (units * cs < fill || (maxP + cs - 1) / cs > kShortSlice)) cs *= 2;
    CS = cs;
  }
  while (CS > 1 && (maxP + CS / 2 - 1) / (CS / 2) <= room &&
         max_active_clusters(CS, smem_for(CS, maxP, p.kp)) < units)
    CS /= 2;
  const size_t smem = smem_for(CS, maxP, p.kp);
  const int cap_floats = (int)(smem / sizeof(float));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = CS;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  // programmatic dependent launch: scheduled while the score kernel drains
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(CS, units);
  cfg.blockDim = dim3(kSelectThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, select_gather, p, cap_floats);
  if (e != cudaSuccess) return e;
  count_launches(1);
  return cudaSuccess;
}

}  // namespace snapkv
