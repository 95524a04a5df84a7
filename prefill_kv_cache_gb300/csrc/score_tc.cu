// Observation-window scores on the 5th-generation tensor cores (tcgen05),
// bf16 inputs, head dim 64 or 128, W*g = 128 or 256 query rows per KV head.
//
// What it computes is the window attention score of every prefix key: the
// softmax(q.k / sqrt(d)) probabilities of the last W prompt queries over
// their causally visible keys, summed over those queries and averaged over
// the query heads of the KV group (jisaku.com glossary "SnapKV",
// "SnapKVの仕組み"; hotpaper.ai summary of "SnapKV: LLM Knows What You are
// Looking for Before Generation", "핵심 아이디어").  The W x L probability
// matrix is never stored: K is swept twice.
//
//   pass 1 (S = Q K^T, query rows on TMEM lanes): per key piece, each
//     thread keeps the running max and sum of exp2 of one query row;
//   merge: per row, the log2-sum-exp2 over the pieces of its KV head;
//   pass 2 (S^T = K Q^T, keys on TMEM lanes): each thread sums
//     exp2(logit * log2e / sqrt(d) - lse2) over all query rows of its key.
//
// Kernel shape: persistent, one CTA per SM (or per SM of the call's share
// when several calls run side by side):
//   warp 0  TMA producer (K tiles of 128 keys, Q of the current KV head),
//   warp 1  MMA issuer (single thread) and TMEM owner (512 columns),
//   warp 2  publisher of finished pass-1 pieces and merges (one release each),
//   warp 3  idle (its warpgroup gives its registers to the consumers),
//   then NSG consumer super-groups of two warpgroups: super-group s reads
//     the tiles of TMEM buffer s (NSG = 2 at W*g = 256: alternate tiles; 1 at
//     128: every tile), warpgroup w of it the column half w; the buffer goes
//     back to the MMA as soon as the columns are in registers, so the MMA of
//     the tile after next overlaps their exp2 work.  Pass-2 half sums meet
//     in the zeroed score array (two addends: order-independent).
// Work items come from a device-wide queue in the order
//   P1(0) | P1(1) M(0) | P1(2) M(1) P2(0) | ... | M(G-1) P2(G-2) | P2(G-1)
// (small launches: every P1, then every M, then every P2) where a group is
// ~1024 key tiles of whole KV heads, P1 / P2 are pass-1 / pass-2 pieces of
// up to 8 tiles and M are merge items.  Pass 2 of a group re-reads K that
// pass 1 streamed through L2 two groups earlier.  A merge item
// waits for its group's pass-1 pieces and a pass-2 item for its group's
// merges; both always sit later in the queue than what they wait for, so
// the waits cannot form a cycle whatever the number of resident CTAs.
// Every wait is bounded: on expiry the kernel sets the status word to
// "timeout", stops taking work, lets its own copies and MMAs drain, frees its
// TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <algorithm>
#include <cstring>

#include "plan.h"
#include "tmem_ld.cuh"
#include "wait.cuh"

namespace snapkv {
namespace tc {

// NSG consumer super-groups of two warpgroups each (8 warps) beside the role
// warpgroup: 1 for W * g = 128, 2 (ping-ponging over the two TMEM buffers)
// for W * g = 256, where the longer tiles hide the hand-offs
__host__ __device__ constexpr int threads_for(int nsg) { return 128 + 256 * nsg; }
constexpr int kTileKeys = 128;
constexpr int kTilesPerPiece = 8;  // at most 1024 keys per piece (the call chooses)
constexpr int kMaxStages = 8;
constexpr int kRing = 4;
constexpr int kPub = 4;  // pass-1 publication slots between consumers and the helper warp
constexpr int kMaxGroups = 128;
constexpr int kGroupTiles = 1024;
constexpr int kMinGroups = 8;  // groups per launch the sizing aims for
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSmemLimit = 232448;
constexpr float kLog2e = 1.4426950408889634f;

enum : int { kP1 = 0, kMerge = 1, kP2 = 2, kDone = 3 };

struct Group {
  int u0, u1;                       // units (seq * H_kv + head) [u0, u1)
  int p1_items, m_items, p2_items;  // items of each kind
  int p1_start, m_start, p2_start;  // their first queue index
};

struct TcPlan {
  int ngroups, total_items, stages, wp;
  int tpp;        // key tiles per piece (the call's piece size / 128)
  int merge_rows; // window rows per merge item: 4 per consumer warp
  int* counters;  // [0] queue head; [1+g] pass-1 pieces done; [1+G+g] merges done
  Group grp[kMaxGroups];
};

struct Entry {
  int type, g, u, piece, tile0, ntiles, row0, nrows;
};

// ------------------------------------------------------------ PTX layer ---

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_addr(b)),
               "r"(bytes)
               : "memory");
}
// One bounded try: the thread is suspended until the phase completes or a
// 20 us hint runs out, so a waiting warp does not take issue slots from the
// warps that work.
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 20000;\n"
      " selp.b32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_addr(b)), "r"(parity)
      : "memory");
  return done != 0;
}
// Bounded wait for the phase of parity `parity` of barrier b.  Returns false
// when the CTA is aborting (flag already set, or this wait expired).  All of
// it is inline: an out-of-line call on the MMA thread's per-tile path costs
// hundreds of cycles of idle tensor pipe, and calls cannot sit in code whose
// register count setmaxnreg changes.
__device__ __forceinline__ bool wait_bar_slow(uint64_t* b, uint32_t parity, Ctl c) {
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test(b, parity)) return true;
    if ((it & 15) == 0) {  // each try suspends for up to 20 us unless the phase completes
      if (*c.abort) return false;
      if (global_ns() - t0 > kWaitNs) {
        raise_timeout(c);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool wait_bar(uint64_t* b, uint32_t parity, const Ctl& c) {
  return mbar_test(b, parity) || wait_bar_slow(b, parity, c);
}


__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle
// layout (rows of 64 bf16 = 128 B, 8-row atoms 1024 B apart).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);  // start address
  d |= (uint64_t)1u << 16;                  // leading-dimension offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;        // stride between 8-row atoms
  d |= (uint64_t)1u << 46;                  // descriptor version
  d |= (uint64_t)2u << 61;                  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 x bf16 -> fp32, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* b) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(b))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Device-scope release increment: the caller's writes (and those ordered
// before it by a CTA barrier) are visible to whoever acquires the new count.
__device__ __forceinline__ void red_release_add(int* ctr, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(ctr), "r"(v) : "memory");
}

// Lowers this warp's register count (the whole warpgroup executes it).
__device__ __forceinline__ void reg_dealloc() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 40;" ::: "memory");
}

// Pass-2 sum over N query rows of one key: sum_r exp2(v[r] * c2 - lse2[r]).
template <int N>
__device__ __forceinline__ float row_sum(const float* v, const float* lse2, float c2) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int j = 0; j < N; j += 4) {
    const float4 m4 = *reinterpret_cast<const float4*>(lse2 + j);
    a0 += ex2(fmaf(v[j], c2, -m4.x));
    a1 += ex2(fmaf(v[j + 1], c2, -m4.y));
    a2 += ex2(fmaf(v[j + 2], c2, -m4.z));
    a3 += ex2(fmaf(v[j + 3], c2, -m4.w));
  }
  return (a0 + a1) + (a2 + a3);
}

// As row_sum, keeping 8 partial sums by column index mod 8 (the query-head
// member of a row when the group size divides 8).
template <int N>
__device__ __forceinline__ void row_sum_members(const float* v, const float* lse2, float c2,
                                                float (&a)[8]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) a[k] = 0.f;
#pragma unroll
  for (int j = 0; j < N; j += 4) {
    const float4 m4 = *reinterpret_cast<const float4*>(lse2 + j);
    a[j & 7] += ex2(fmaf(v[j], c2, -m4.x));
    a[(j + 1) & 7] += ex2(fmaf(v[j + 1], c2, -m4.y));
    a[(j + 2) & 7] += ex2(fmaf(v[j + 2], c2, -m4.z));
    a[(j + 3) & 7] += ex2(fmaf(v[j + 3], c2, -m4.w));
  }
}

// Packed fp32x2 arithmetic (one instruction for two lanes of values).
__device__ __forceinline__ uint64_t pk(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk(uint64_t x, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(x));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t ex2x2(uint64_t x) {
  float a, b;
  upk(x, a, b);
  return pk(ex2(a), ex2(b));
}
__device__ __forceinline__ float sum4(const uint64_t (&a)[4]) {
  float x0, x1, x2, x3, x4, x5, x6, x7;
  upk(a[0], x0, x1);
  upk(a[1], x2, x3);
  upk(a[2], x4, x5);
  upk(a[3], x6, x7);
  return ((x0 + x1) + (x2 + x3)) + ((x4 + x5) + (x6 + x7));
}

// Pass 2, one 32-column chunk of a key's row of logits: adds
// exp2(v[j] * c2 - lse2[j]) into four pair accumulators (pair p of the chunk
// goes to acc[p % 4], so acc[k] holds the columns 2k, 2k+1 mod 8).  nl holds
// -lse2 of the chunk's 32 query rows (shared memory, 16-byte aligned).
__device__ __forceinline__ void p2_chunk(const uint32_t* v, const float* nl, uint64_t c2c2,
                                         uint64_t (&acc)[4]) {
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    const float4 l4 = *reinterpret_cast<const float4*>(nl + j);
    const uint64_t x0 =
        fma2(pk(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), c2c2, pk(l4.x, l4.y));
    const uint64_t x1 =
        fma2(pk(__uint_as_float(v[j + 2]), __uint_as_float(v[j + 3])), c2c2, pk(l4.z, l4.w));
    acc[(j >> 1) & 3] = add2(acc[(j >> 1) & 3], ex2x2(x0));
    acc[((j >> 1) + 1) & 3] = add2(acc[((j >> 1) + 1) & 3], ex2x2(x1));
  }
}

// Pass 1, one 32-key chunk of a query row, all keys visible: the sum of
// exp2(v[j] * c2 - M) for the row's running reference M.
__device__ __forceinline__ float p1_chunk_sum(const uint32_t* v, uint64_t c2c2, uint64_t nMnM) {
  uint64_t a[4] = {0, 0, 0, 0};
#pragma unroll
  for (int j = 0; j < 32; j += 2)
    a[(j >> 1) & 3] = add2(
        a[(j >> 1) & 3],
        ex2x2(fma2(pk(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), c2c2, nMnM)));
  return sum4(a);
}

// Pass 1, one 32-key chunk with an exact reference: keys past `limit` (the
// last key the row sees, relative to the chunk) are masked; the running
// (M, Z) move to the larger of M and the chunk's largest scaled logit.
__device__ __forceinline__ void p1_chunk_exact(uint32_t* v, int limit, float c2, float& M,
                                               float& Z) {
  float tmax = -INFINITY;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float x = j > limit ? -INFINITY : __uint_as_float(v[j]);
    v[j] = __float_as_uint(x);
    tmax = fmaxf(tmax, x);
  }
  if (tmax == -INFINITY) return;  // the row sees no key of this chunk
  const float Mn = fmaxf(M, tmax * c2);
  const float z = p1_chunk_sum(v, pk(c2, c2), pk(-Mn, -Mn));
  Z = Z * ex2(M - Mn) + z;  // M = -inf: ex2 gives 0 and Z was 0
  M = Mn;
}

// ------------------------------------------------------------ schedule ---

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

__device__ Entry decode(const Plan& p, const TcPlan& tp, int idx) {
  Entry e{};
  e.type = kDone;
  if (idx >= tp.total_items) return e;
  for (int g = 0; g < tp.ngroups; ++g) {
    const Group& G = tp.grp[g];
    int kind = -1, local = 0;
    if (idx >= G.p1_start && idx < G.p1_start + G.p1_items) {
      kind = kP1;
      local = idx - G.p1_start;
    } else if (idx >= G.m_start && idx < G.m_start + G.m_items) {
      kind = kMerge;
      local = idx - G.m_start;
    } else if (idx >= G.p2_start && idx < G.p2_start + G.p2_items) {
      kind = kP2;
      local = idx - G.p2_start;
    }
    if (kind < 0) continue;
    e.type = kind;
    e.g = g;
    if (kind == kMerge) {
      e.row0 = local * tp.merge_rows;
      e.nrows = min(tp.merge_rows, (G.u1 - G.u0) * tp.wp - e.row0);
      return e;
    }
    for (int u = G.u0; u < G.u1; ++u) {
      const SeqInfo& S = p.seq[u / p.H_kv];
      if (!S.scored) continue;
      const int keys = kind == kP1 ? S.L : S.P;
      const int tiles = ceil_div(keys, kTileKeys);
      const int pieces = ceil_div(tiles, tp.tpp);
      if (local < pieces) {
        e.u = u;
        e.piece = local;
        e.tile0 = local * tp.tpp;
        e.ntiles = min(tp.tpp, tiles - e.tile0);
        return e;
      }
      local -= pieces;
    }
    e.type = kDone;  // unreachable with a consistent plan
    return e;
  }
  return e;
}

// ---------------------------------------------------------- the kernel ---

// PER_Q: every query head keeps its own pass-2 sums (per-query-head selection)
template <bool PER_Q, int NSG>
__global__ void __launch_bounds__(threads_for(NSG), 1)
score_tc_kernel(const __grid_constant__ Plan p, const __grid_constant__ TcPlan tp,
                const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q) {
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr int kConsumerThreads = 256 * NSG;
  constexpr int kConsumerWarps = kConsumerThreads / 32;
  // registers at launch: 384 x 168 = 64512 (NSG 1) or 640 x 96 = 61440 (NSG 2);
  // the role warpgroup drops to 40, the consumers rise to kConsumerRegs:
  // 128 x 40 + 256 x 232 = 64512, 128 x 40 + 512 x 104 = 58368
  constexpr int kConsumerRegs = NSG == 2 ? 104 : 232;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = tp.stages, wp = tp.wp, d = p.d;
  const int halves = d / 64;
  const uint32_t q_half_bytes = (uint32_t)wp * 128u;
  const uint32_t q_bytes = q_half_bytes * halves;
  const uint32_t k_half_bytes = kTileKeys * 128u;
  const uint32_t k_bytes = k_half_bytes * halves;

  uint8_t* qbuf = smem;
  uint8_t* kbuf = smem + 2 * q_bytes;
  float* aux = reinterpret_cast<float*>(kbuf + (size_t)NS * k_bytes);  // 512 floats
  uint64_t* bars = reinterpret_cast<uint64_t*>(aux + 512);
  uint64_t* full = bars;
  uint64_t* empty = full + kMaxStages;
  uint64_t* qfull = empty + kMaxStages;
  uint64_t* qempty = qfull + 2;
  uint64_t* tfull = qempty + 2;
  uint64_t* tempty = tfull + 2;
  uint64_t* sfull = tempty + 2;
  uint64_t* sempty = sfull + kRing;
  uint64_t* drain = sempty + kRing;  // MMA drain at teardown
  uint64_t* pub_full = drain + 1;     // pass-1 item finished by the consumer warps
  uint64_t* pub_empty = pub_full + kPub;  // helper done with the slot
  uint64_t* gl_full = pub_empty + kPub;   // per warpgroup: its pass-2 LSE copy written
  uint64_t* gl_empty = gl_full + 4;       // per warpgroup: the copy read to the end
  int* pub_grp = reinterpret_cast<int*>(gl_empty + 4);
  Entry* ring = reinterpret_cast<Entry*>(pub_grp + kPub);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ring + kRing);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(abort_flag) + 1);
  const Ctl ctl{abort_flag, p.status};

  if (threadIdx.x == 0) {
    if ((smem_addr(smem) & 1023u) != 0) atomicExch(p.status, kDevTimeout);
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&qfull[b], 1);
      mbar_init(&qempty[b], 1);
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 8);  // the 8 warps of the super-group that reads buffer b
    }
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], 1 + kConsumerWarps);  // MMA thread + the consumer warps
    }
    mbar_init(drain, 1);
    for (int k = 0; k < kPub; ++k) {
      mbar_init(&pub_full[k], kConsumerWarps);
      mbar_init(&pub_empty[k], 1);
    }
    for (int k = 0; k < 4; ++k) {
      mbar_init(&gl_full[k], 4);   // the warpgroup's four warps
      mbar_init(&gl_empty[k], 4);
    }
    *abort_flag = (smem_addr(smem) & 1023u) != 0 ? 1 : 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
            smem_addr(tmem_slot)),
        "r"(kTmemCols)
        : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const float c2 = p.log2e_scale;  // log2(e) / sqrt(d)
  // each role's branch sets its own register count (see kConsumerRegs)

  if (warp < 4) reg_dealloc();  // one instruction for the whole warpgroup
  if (warp == 0) {
    // ------------------------------------------------------ producer ---
    if (lane == 0) {
      int ring_n = 0, item_n = 0, st = 0;
      uint32_t sph = 0;  // phase parity of stage st's current use
      int fills[kMaxStages] = {0, 0, 0, 0, 0, 0, 0, 0};
      int qfills[2] = {0, 0};
      for (;;) {
        const int idx = *abort_flag ? tp.total_items : atomicAdd(&tp.counters[0], 1);
        const Entry e = decode(p, tp, idx);
        const int slot = ring_n % kRing;
        if (!wait_bar(&sempty[slot], ((ring_n / kRing) & 1) ^ 1, ctl)) break;
        ring[slot] = e;
        mbar_arrive(&sfull[slot]);
        ++ring_n;
        if (e.type == kDone) break;
        if (e.type == kMerge) continue;
        const SeqInfo& S = p.seq[e.u / p.H_kv];
        const int h = e.u % p.H_kv;
        const int qb = item_n & 1;
        if (!wait_bar(&qempty[qb], ((item_n >> 1) & 1) ^ 1, ctl)) break;
        mbar_arrive_tx(&qfull[qb], q_bytes);
        for (int hf = 0; hf < halves; ++hf)
          tma_load_3d(smem_addr(qbuf + qb * q_bytes + hf * q_half_bytes), &tm_q, &qfull[qb],
                      hf * 64, h * p.g, S.b * p.W);
        ++qfills[qb];
        bool ok = true;
        for (int t = 0; t < e.ntiles; ++t) {
          if (!wait_bar(&empty[st], sph ^ 1, ctl)) {
            ok = false;
            break;
          }
          mbar_arrive_tx(&full[st], k_bytes);
          const int row = (int)S.row0 + (e.tile0 + t) * kTileKeys;
          for (int hf = 0; hf < halves; ++hf)
            tma_load_3d(smem_addr(kbuf + st * k_bytes + hf * k_half_bytes), &tm_k, &full[st],
                        hf * 64, h, row);
          ++fills[st];
          if (++st == NS) {
            st = 0;
            sph ^= 1;
          }
        }
        ++item_n;
        if (!ok) break;
      }
      // drain: every copy this thread issued lands before the CTA leaves
      for (int s = 0; s < NS; ++s)
        if (fills[s] > 0) {  // completion of the last fill of stage s
          const uint64_t t0 = global_ns();
          while (!mbar_test(&full[s], (uint32_t)((fills[s] - 1) & 1)) &&
                 global_ns() - t0 < kWaitNs) {
          }
        }
      for (int b = 0; b < 2; ++b)
        if (qfills[b] > 0) {
          const uint64_t t0 = global_ns();
          while (!mbar_test(&qfull[b], (uint32_t)((qfills[b] - 1) & 1)) &&
                 global_ns() - t0 < kWaitNs) {
          }
        }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA ---
    if (lane == 0) {
      int ring_n = 0, item_n = 0, st = 0, tile_n = 0;
      uint32_t sph = 0;
      const uint32_t id_p1 = idesc_bf16(128, 128);
      const uint32_t id_p2 = idesc_bf16(128, wp);
      const int R = wp / 128;
      bool issued = false;
      for (;;) {
        const int slot = ring_n % kRing;
        if (!wait_bar(&sfull[slot], (ring_n / kRing) & 1, ctl)) break;
        const Entry e = ring[slot];
        ++ring_n;
        mbar_arrive(&sempty[slot]);
        if (e.type == kDone) break;
        if (e.type == kMerge) continue;
        const int qb = item_n & 1;
        if (!wait_bar(&qfull[qb], (item_n >> 1) & 1, ctl)) break;
        tc_fence_after();
        const uint32_t qa = smem_addr(qbuf + qb * q_bytes);
        bool ok = true;
        for (int t = 0; t < e.ntiles; ++t) {
          const int ab = tile_n & 1;
          if (!wait_bar(&full[st], sph, ctl) ||
              !wait_bar(&tempty[ab], ((tile_n >> 1) & 1) ^ 1, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ka = smem_addr(kbuf + st * k_bytes);
          const uint32_t dcol = tmem + (uint32_t)ab * 256u;
          if (e.type == kP1) {
            for (int rb = 0; rb < R; ++rb)
              for (int kk = 0; kk < d / 16; ++kk) {
                const uint64_t ad = sw128_desc(qa + (uint32_t)(kk >> 2) * q_half_bytes +
                                               (uint32_t)rb * 128u * 128u + (uint32_t)(kk & 3) * 32u);
                const uint64_t bd = sw128_desc(ka + (uint32_t)(kk >> 2) * k_half_bytes +
                                               (uint32_t)(kk & 3) * 32u);
                mma_bf16(dcol + (uint32_t)rb * 128u, ad, bd, id_p1, kk > 0);
              }
          } else {
            for (int kk = 0; kk < d / 16; ++kk) {
              const uint64_t ad = sw128_desc(ka + (uint32_t)(kk >> 2) * k_half_bytes +
                                             (uint32_t)(kk & 3) * 32u);
              const uint64_t bd = sw128_desc(qa + (uint32_t)(kk >> 2) * q_half_bytes +
                                             (uint32_t)(kk & 3) * 32u);
              mma_bf16(dcol, ad, bd, id_p2, kk > 0);
            }
          }
          mma_commit(&empty[st]);
          mma_commit(&tfull[ab]);
          issued = true;
          if (++st == NS) {
            st = 0;
            sph ^= 1;
          }
          ++tile_n;
        }
        mma_commit(&qempty[qb]);
        ++item_n;
        if (!ok) break;
      }
      if (issued) {
        // all MMAs this thread issued have completed once `drain` flips
        mma_commit(drain);
        const uint64_t t0 = global_ns();
        while (!mbar_test(drain, 0) && global_ns() - t0 < kWaitNs) {
        }
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------- helper ---
    // publishes finished pass-1 items: waits until all consumer warps have
    // written an item's statistics, then one device-scope release increment
    // of its group's counter makes them visible to the merge items
    if (lane == 0) {
      for (int n = 0;; ++n) {
        const int k = n % kPub;
        if (!wait_bar(&pub_full[k], (n / kPub) & 1, ctl)) break;
        const int g = pub_grp[k];
        if (g >= 0) red_release_add(&tp.counters[1 + g], 1);
        mbar_arrive(&pub_empty[k]);
        if (g < 0) break;
      }
    }
  } else if (warp >= 4) {
    // ----------------------------------------------------- consumers ---
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsumerRegs) : "memory");
    // two super-groups of two warpgroups: super-group sg reads the tiles of
    // TMEM buffer sg (every other tile), its warpgroup wg the column half wg
    const int ct = threadIdx.x - 128;         // 0..511
    const int sg = NSG == 2 ? ct >> 8 : 0;    // super-group
    const int wg = (ct >> 7) & 1;             // warpgroup within it: column half it reads
    const int grp = ct >> 7;                  // warpgroup index 0..3
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int lrow = quarter * 32 + lane;     // TMEM lane of this thread
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const int R = wp / 128;
    const int half = wp >> 1;
    int ring_n = 0, tile_n = 0, p2_n = 0;  // p2_n: pass-2 items taken (phase of gl_*)
    const uint64_t c2c2 = pk(c2, c2);
    // two 32-column chunks of a tile's accumulator (pass 1: 32 keys of one
    // query row; pass 2: 32 query rows of one key)
    uint32_t v[64];
    // pass 2: -lse2 of the warpgroup's query rows, item-constant, one shared
    // copy per warpgroup (written by its four warps; gl_full / gl_empty, with
    // bounded waits, order the writes and the reads)
    float* gl = aux + grp * 128;
    // pass 1: this thread's query row of a tile (row block wg when there are
    // two, else row block 0 with the group's half of the keys) and the row's
    // window index; both are the same for every item
    const int prow = (R == 2 ? 128 * wg : 0) + lrow;
    const int pwin = prow / p.g;
    const int kofs = R == 2 ? 0 : 64 * wg;  // first key of the group's share of a tile
    const int cw = warp - 4;                // consumer warp 0..15
    // hands a finished pass-1 item (group g; -1: no more) to the helper warp,
    // which publishes it with one device-scope release once all consumer
    // warps have written their statistics
    int pub_n = 0;
    auto publish = [&](int g) -> bool {
      const int k = pub_n % kPub;
      const bool ok = wait_bar(&pub_empty[k], ((pub_n / kPub) & 1) ^ 1, ctl);
      ++pub_n;
      if (!ok) return false;
      if (lane == 0) pub_grp[k] = g;
      __syncwarp();
      if (lane == 0) mbar_arrive(&pub_full[k]);
      return true;
    };
    for (;;) {
      const int slot = ring_n % kRing;
      if (!wait_bar(&sfull[slot], (ring_n / kRing) & 1, ctl)) break;
      const Entry e = ring[slot];
      ++ring_n;
      if (e.type == kDone) {
        publish(-1);  // the helper warp stops
        break;
      }
      const Group& G = tp.grp[e.g];
      // partial statistics per piece and row: one per super-group with two
      // row blocks (a row block has one warpgroup per super-group), two per
      // super-group with one (the warpgroups split the keys)
      const int nslot = R == 2 ? NSG : 2 * NSG;
      if (e.type == kMerge) {
        // each warp merges 4 of the item's 4 x kConsumerWarps rows, 8 lanes per row with the
        // partial statistics strided over them; every lane issues its loads
        // before it combines any of them
        if (lane == 0) wait_counter(&tp.counters[1 + e.g], G.p1_items, ctl);
        __syncwarp();
        if (*abort_flag) break;
        const int rl = cw * 4 + (lane >> 3), sub = lane & 7;
        const int gr = e.row0 + rl;
        float M = -INFINITY, Z = 0.f;
        int u = -1, r = 0;
        if (rl < e.nrows) {
          u = G.u0 + gr / wp;
          r = gr % wp;
          const SeqInfo& S = p.seq[u / p.H_kv];
          if (S.scored) {
            const int h = u % p.H_kv;
            const int parts = nslot * S.chunks;
            // part c = piece (c / nslot), slot (c % nslot)
            const float2* st = p.stats + (size_t)(S.piece0 + h * S.chunks) * 512 + r;
            for (int c0 = sub; c0 < parts; c0 += 64) {
              float2 x[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const int c = c0 + 8 * k;
                x[k] = c < parts ? __ldcg(st + (size_t)(c / nslot) * 512 + (size_t)(c % nslot) * wp)
                                 : make_float2(-INFINITY, 0.f);
              }
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                if (x[k].x == -INFINITY) continue;
                if (x[k].x > M) {
                  Z = Z * exp2f(M - x[k].x) + x[k].y;
                  M = x[k].x;
                } else {
                  Z += x[k].y * exp2f(x[k].x - M);
                }
              }
            }
          } else {
            u = -1;
          }
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
          const float Mo = __shfl_xor_sync(0xffffffffu, M, o);
          const float Zo = __shfl_xor_sync(0xffffffffu, Z, o);
          const float Mn = fmaxf(M, Mo);
          if (Mn != -INFINITY) Z = Z * exp2f(M - Mn) + Zo * exp2f(Mo - Mn);
          M = Mn;
        }
        if (sub == 0 && u >= 0) p.lse[(size_t)u * wp + r] = M + log2f(Z);
        // the warp's writes are ordered before one release of the counter
        __syncwarp();
        if (lane == 0) {
          red_release_add(&tp.counters[1 + tp.ngroups + e.g], 1);
          mbar_arrive(&sempty[slot]);
        }
        continue;
      }

      const int s_idx = e.u / p.H_kv, h = e.u % p.H_kv;
      const SeqInfo& S = p.seq[s_idx];
      bool ok = true;
      if (e.type == kP2) {
        // the window rows' LSE (merged above, or the caller's): the
        // warpgroup's rows half wg ... half wg + half - 1, the same for every
        // lane, go to its shared copy; warp quarter q writes rows 32q ...
        // 32q + 31 once the previous item's readers are done (gl_empty)
        if (!p.lse_in && lane == 0)
          wait_counter(&tp.counters[1 + tp.ngroups + e.g], G.m_items * kConsumerWarps, ctl);
        __syncwarp();
        if (*abort_flag) break;
        if (!wait_bar(&gl_empty[grp], (p2_n & 1) ^ 1, ctl)) break;
        const int r0 = wg * half;  // first query row of the group's share
        if (quarter * 32 < half) {
          const int rr = r0 + quarter * 32 + lane;
          if (p.lse_in) {
            // the caller's natural-log LSE, row r = i g + member; g divides
            // W * g, a power of two, so it is one too
            const int lg = __ffs(p.g) - 1;
            const float* base = p.lse_in + (size_t)S.b * p.W * p.H_q + (size_t)h * p.g;
            gl[quarter * 32 + lane] = -__ldg(base + (size_t)(rr >> lg) * p.H_q + (rr & (p.g - 1))) * kLog2e;
          } else {
            gl[quarter * 32 + lane] = -__ldcg(p.lse + (size_t)e.u * wp + rr);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&gl_full[grp]);
        if (!wait_bar(&gl_full[grp], p2_n & 1, ctl)) break;
      }
      float Mr = -INFINITY, Zr = 0.f;  // pass 1: running reference and sum of this thread's row
      float* raw_out = p.raw + S.score0 + (size_t)h * S.P;
      const float inv_g = 1.0f / (float)p.g;
      // pass 1: the last key the row sees, relative to the first key of the
      // group's share of tile 0
      const int last = min(S.P + pwin, S.L - 1) - kofs;
      // first TMEM column of this thread's share: pass 1, the row block's
      // keys (128 per row block) or the group's 64 of them; pass 2, query
      // rows half wg ...
      const uint32_t col0 = e.type == kP1 ? (R == 2 ? 128u * wg : 64u * wg) : (uint32_t)(wg * half);
      auto chunk1 = [&](uint32_t* vc, int lim) {
        // all 32 keys visible and a finite reference: sum against it; a sum
        // past 2^100 means a logit far above the reference (or an overflow),
        // and the chunk is redone with an exact reference (rare)
        if (Mr != -INFINITY && lim >= 31) {
          const float Zn = Zr + p1_chunk_sum(vc, c2c2, pk(-Mr, -Mr));
          if (Zn < 0x1p100f) {
            Zr = Zn;
            return;
          }
        }
        p1_chunk_exact(vc, lim, c2, Mr, Zr);
      };
      for (int t = 0; t < e.ntiles; ++t, ++tile_n) {
        const int ab = tile_n & 1;  // TMEM buffer of this tile; its super-group reads it
        if (NSG == 2 && ab != sg) continue;
        if (!wait_bar(&tfull[ab], (tile_n >> 1) & 1, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int key0 = (e.tile0 + t) * kTileKeys;
        const uint32_t tb = tmem + lane_addr + (uint32_t)ab * 256u + col0;
        // rolling pair of 32-column chunks: chunk c + 1 loads while chunk c is
        // processed; the buffer goes back to the MMA once the last chunk has
        // landed in registers
        __syncwarp();  // tcgen05.ld is warp-collective
        tmem_ld32_async(tb, v);
        tmem_wait32(v);
        tmem_ld32_async(tb + 32u, v + 32);
        if (e.type == kP1) {
          const int lim = last - key0;
          chunk1(v, lim);
          tmem_wait32(v + 32);
          if (R == 2) {
            __syncwarp();
            tmem_ld32_async(tb + 64u, v);
            chunk1(v + 32, lim - 32);
            tmem_wait32(v);
            __syncwarp();
            tmem_ld32_async(tb + 96u, v + 32);
            chunk1(v, lim - 64);
            tmem_wait32(v + 32);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[ab]);
            chunk1(v + 32, lim - 96);
          } else {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[ab]);
            chunk1(v + 32, lim - 32);
          }
        } else {
          uint64_t acc[4] = {0, 0, 0, 0};
          p2_chunk(v, gl, c2c2, acc);
          tmem_wait32(v + 32);
          if (half == 128) {
            __syncwarp();
            tmem_ld32_async(tb + 64u, v);
            p2_chunk(v + 32, gl + 32, c2c2, acc);
            tmem_wait32(v);
            __syncwarp();
            tmem_ld32_async(tb + 96u, v + 32);
            p2_chunk(v, gl + 64, c2c2, acc);
            tmem_wait32(v + 32);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[ab]);
            p2_chunk(v + 32, gl + 96, c2c2, acc);
          } else {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[ab]);
            p2_chunk(v + 32, gl + 32, c2c2, acc);
          }
          const int key = key0 + lrow;
          if (PER_Q) {
            // every query head keeps its own sum: member m of the group owns
            // the rows r with r % g == m (g divides 8; acc[k] holds the
            // columns 2k, 2k+1 mod 8); the two warpgroups' halves add up in the
            // zeroed score array (two addends onto zero: order-independent)
            float am[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) upk(acc[k], am[2 * k], am[2 * k + 1]);
            if (key < S.P) {
              float* base = p.raw + S.score0 + (size_t)h * p.g * S.P + key;
              for (int m = 0; m < p.g; ++m) {
                float x = 0.f;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                  if (k % p.g == m) x += am[k];
                atomicAdd(base + (size_t)m * S.P, x);
              }
            }
          } else if (key < S.P) {
            // the two warpgroups' halves meet in the zeroed score array (two
            // addends onto zero: the result does not depend on their order)
            atomicAdd(raw_out + key, sum4(acc) * inv_g);
          }
        }
      }
      if (!ok) break;
      if (e.type == kP1) {
        // clear the piece's prefix keys in the score array, into which pass 2
        // adds its two halves; the release below orders these stores before
        // every pass-2 item of the group
        {
          const int k_lo = e.tile0 * kTileKeys;
          const int k_hi = min(S.P, k_lo + e.ntiles * kTileKeys);
          const int rows = PER_Q ? p.g : 1;  // score vectors per KV head
          float* z = p.raw + S.score0 + (size_t)h * rows * S.P;
          for (int m = 0; m < rows; ++m)
            for (int k = k_lo + ct; k < k_hi; k += kConsumerThreads) z[(size_t)m * S.P + k] = 0.f;
        }
        // publish this row's statistics for the piece (slot sg with two row
        // blocks; 2 sg + wg with one, where the two warpgroups hold halves of
        // the keys); the
        // device-scope release that publishes them takes a while (it waits
        // for this warp's writes to land): the helper warp does it
        const size_t piece = (size_t)S.piece0 + (size_t)h * S.chunks + e.piece;
        const int q = R == 2 ? sg : 2 * sg + wg;
        p.stats[piece * 512 + (size_t)q * wp + prow] = make_float2(Mr, Zr);
        if (!publish(e.g)) break;
      }
      if (e.type == kP2) {  // the warpgroup's LSE copy may be overwritten
        __syncwarp();
        if (lane == 0) mbar_arrive(&gl_empty[grp]);
        ++p2_n;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[slot]);
    }
  }

  // ---------------------------------------------------------- teardown ---
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
}

// --------------------------------------------------------------- host ---

using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiled get_encoder() {
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

// 3-D bf16 tensor map {d, heads, rows}, box {64, box1, box2}, 128 B swizzle.
bool make_map(CUtensorMap* m, const void* base, int d, int heads, long long rows, int box1,
              int box2) {
  EncodeTiled enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * heads};
  cuuint32_t box[3] = {64, (cuuint32_t)box1, (cuuint32_t)box2};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

// Builds the item queues for one launch group and launches the kernel, or
// declines (taken = false) for shapes it does not cover: anything but bf16
// with d in {64, 128} and W * g in {128, 256}.  A shape it covers always runs
// here: a launch group with more KV heads than one launch's queue can describe
// is split into several launches, and any failure is returned as an error.
int launch_score_tc(const Plan& p, void* stream, bool* taken, int* counter_off) {
  using namespace tc;
  *taken = false;
  if (p.dtype != 0 || (p.d != 64 && p.d != 128) || (p.Wp != 128 && p.Wp != 256)) return cudaSuccess;
  *taken = true;
  if (p.chunk_keys % kTileKeys != 0 || p.chunk_keys > kTileKeys * kTilesPerPiece ||
      p.counters == nullptr)
    return cudaErrorInvalidValue;
  const int tpp = p.chunk_keys / kTileKeys;
  const DeviceInfo* di = current_device_info();
  if (!di) return cudaErrorUnknown;
  const int sms = di->sms;

  const uint32_t halves = p.d / 64;
  const uint32_t q_bytes = (uint32_t)p.Wp * 128u * halves;
  const uint32_t k_bytes = (uint32_t)kTileKeys * 128u * halves;
  const uint32_t misc = 512 * 4 + (2 * kMaxStages + 16 + 2 * kRing + 1 + 2 * kPub) * 8 +
                        kPub * 4 + kRing * sizeof(Entry) + 8;
  const long long room = (long long)kSmemLimit - 2 * (long long)q_bytes - misc;
  int stages = (int)(room / k_bytes);
  if (stages > 6) stages = 6;
  if (stages < 2) return cudaErrorInvalidConfiguration;  // cannot happen for W * g <= 256
  const size_t smem = 2 * (size_t)q_bytes + (size_t)stages * k_bytes + misc;

  // the K map covers the rows of the whole call (rows past the end read as zeros)
  CUtensorMap tm_k, tm_q;
  if (!make_map(&tm_k, p.k, p.d, p.H_kv, p.total_rows, 1, kTileKeys) ||
      !make_map(&tm_q, p.q, p.d, p.H_q, (long long)p.batch * p.W, p.g, p.W))
    return cudaErrorInvalidValue;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // two consumer super-groups at W * g = 256, one at 128 (the shorter tiles
  // do not hide the ping-pong's per-item hand-offs)
  const int nsg = p.Wp == 256 ? 2 : 1;
  const int threads = threads_for(nsg);
  auto kern = p.out_heads != p.H_kv
                  ? (nsg == 2 ? score_tc_kernel<true, 2> : score_tc_kernel<true, 1>)
                  : (nsg == 2 ? score_tc_kernel<false, 2> : score_tc_kernel<false, 1>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  if (p.lse_in) {  // no pass 1 to clear the scores: pass 2 adds two halves into zeroed ones
    long long lo = -1, hi = 0;
    for (int s = 0; s < p.nseq; ++s) {
      const SeqInfo& S = p.seq[s];
      if (!S.scored) continue;
      if (lo < 0) lo = S.score0;
      hi = S.score0 + (long long)p.out_heads * S.P;
    }
    if (hi > lo && lo >= 0) {
      e = cudaMemsetAsync(p.raw + lo, 0, sizeof(float) * (size_t)(hi - lo), st);
      if (e != cudaSuccess) return e;
    }
  }

  const int units = p.nseq * p.H_kv;
  // groups of whole KV heads of about group_tiles key tiles: at most
  // kGroupTiles, and small enough that a launch has several groups, so that
  // pass 2 of one group overlaps pass 1 of the next ones
  long long total_tiles = 0;
  for (int u = 0; u < units; ++u) {
    const SeqInfo& S = p.seq[u / p.H_kv];
    if (S.scored) total_tiles += (S.L + kTileKeys - 1) / kTileKeys;
  }
  const int group_tiles =
      (int)std::max(1LL, std::min((long long)kGroupTiles, total_tiles / kMinGroups));
  int u_begin = 0;
  while (u_begin < units) {
    TcPlan tp;
    std::memset(&tp, 0, sizeof tp);
    tp.wp = p.Wp;
    tp.tpp = tpp;
    tp.merge_rows = 32 * nsg;  // 4 rows per consumer warp
    tp.counters = p.counters;
    tp.stages = stages;
    // groups of whole KV heads, ~kGroupTiles key tiles each, at most
    // kMaxGroups per launch
    int g = 0, acc = 0, u0 = u_begin, u = u_begin;
    for (; u < units && g < kMaxGroups; ++u) {
      const SeqInfo& S = p.seq[u / p.H_kv];
      if (S.scored) acc += (S.L + kTileKeys - 1) / kTileKeys;
      const bool last = u == units - 1;
      if (acc >= group_tiles || (last && acc > 0)) {
        tp.grp[g].u0 = u0;
        tp.grp[g].u1 = u + 1;
        ++g;
        u0 = u + 1;
        acc = 0;
      }
    }
    if (g == 0) break;  // the remaining units have nothing to score
    u_begin = tp.grp[g - 1].u1;
    tp.ngroups = g;
    for (int i = 0; i < g; ++i) {
      Group& G = tp.grp[i];
      for (int x = G.u0; x < G.u1; ++x) {
        const SeqInfo& S = p.seq[x / p.H_kv];
        if (!S.scored) continue;
        const int t1 = (S.L + kTileKeys - 1) / kTileKeys, t2 = (S.P + kTileKeys - 1) / kTileKeys;
        G.p1_items += (t1 + tpp - 1) / tpp;
        G.p2_items += (t2 + tpp - 1) / tpp;
      }
      G.m_items = ((G.u1 - G.u0) * p.Wp + tp.merge_rows - 1) / tp.merge_rows;
    }
    // queue order: P1(0) | P1(1) M(0) | P1(2) M(1) P2(0) | ... | M(G-1) P2(G-2) | P2(G-1):
    // merges follow the next group's pass 1, pass 2 trails by two groups, so
    // pass-2 items rarely wait for their merge while K is still in L2.  A
    // launch with at most two pass-1 items per SM of the GPU takes every
    // pass 1, then every merge, then every pass 2 instead: with the lagged
    // order its first wave would park CTAs on pass-2 items of early groups
    // (waiting for their merges) while later groups' pass-1 items wait for
    // a CTA.  Every item waits only on items earlier in the queue either way.
    long long p1_total = 0;
    for (int k = 0; k < g; ++k) p1_total += tp.grp[k].p1_items;
    const bool one_wave = p1_total <= 2LL * sms;
    const int lag_m = one_wave ? g : 1, lag_p2 = one_wave ? 2 * g : 2;  // lag_m < lag_p2
    int idx = 0;
    if (p.lse_in) {  // the caller's LSE: pass 2 only
      for (int k = 0; k < g; ++k) {
        Group& G = tp.grp[k];
        G.p1_items = G.m_items = 0;
        G.p1_start = G.m_start = 1 << 30;
        G.p2_start = idx;
        idx += G.p2_items;
      }
    }
    for (int k = 0; k < g + lag_p2 && !p.lse_in; ++k) {
      if (k < g) {
        tp.grp[k].p1_start = idx;
        idx += tp.grp[k].p1_items;
      }
      if (k >= lag_m && k - lag_m < g) {
        tp.grp[k - lag_m].m_start = idx;
        idx += tp.grp[k - lag_m].m_items;
      }
      if (k >= lag_p2 && k - lag_p2 < g) {
        tp.grp[k - lag_p2].p2_start = idx;
        idx += tp.grp[k - lag_p2].p2_items;
      }
    }
    tp.total_items = idx;
    // the queue head and the per-group counters: a fresh slice of the
    // call's zeroed counter region (zeroed again when it runs out)
    const int need = 1 + 2 * g;
    if (*counter_off + need > kCounterInts) {
      e = cudaMemsetAsync(p.counters, 0, sizeof(int) * kCounterInts, st);
      if (e != cudaSuccess) return e;
      *counter_off = 0;
    }
    tp.counters = p.counters + *counter_off;
    *counter_off += need;
    // one CTA per SM, or per SM of this call's share when several calls run
    // side by side (their waits are only on their own items: no deadlock)
    const int width = p.gpu_share > 1 ? std::max(1, sms / p.gpu_share) : sms;
    const int grid = width < tp.total_items ? width : tp.total_items;
    kern<<<grid, threads, smem, st>>>(p, tp, tm_k, tm_q);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launches(1);
    count_score_launches(kScorePathTensorCores, 1);
  }
  return cudaSuccess;
}

}  // namespace snapkv
