// Internal launch plan shared by the host side and the kernels of libsnapkv.
//
// A call is split into groups of at most kGroupSeqs sequences; each group's
// per-sequence table travels to the kernels by value as a __grid_constant__
// parameter, so a launch needs no host-to-device copy and no allocation.
#pragma once

#include <cstddef>
#include <cstdint>

namespace snapkv {

constexpr int kGroupSeqs = 64;     // sequences per launch group
constexpr int kMaxRows = 256;      // W * g limit (query rows per KV head)
constexpr int kMaxBatch = 4096;
constexpr int kClusterCTAs = 8;    // CTAs per (sequence, KV head) in select/gather
constexpr int kSelectThreads = 512;
constexpr int kCounterInts = 1024;  // work-queue counters in the workspace

// Status word values written by kernels (0 = fine).
constexpr int kDevOk = 0;
constexpr int kDevTimeout = 5;

struct SeqInfo {
  int b;             // index of the sequence in the caller's batch
  int L;             // prompt length
  int P;             // L - W (prefix length; may be <= 0)
  int scored;        // 1 if L > C: scores, pooling and selection run
  long long row0;    // first packed row of this sequence in k / v
  long long score0;  // float offset of (b, h=0) in raw / pooled; (b,h) at score0 + h*P
  int piece0;        // first score piece of this sequence (group-local)
  int chunks;        // score pieces per KV head
};

struct Plan {
  // problem
  int nseq;          // sequences in this group
  int H_q, H_kv, g, d, W, Wp, C, n, kp, pool, dtype;
  float scale;       // 1 / sqrt(d)
  float log2e_scale; // log2(e) / sqrt(d)
  // score pieces (pass 1 and pass 2 share them)
  int chunk_keys;
  int total_pieces;
  // buffers
  const void* q;
  const void* k;
  const void* v;
  void* out_k;
  void* out_v;
  int32_t* out_idx;
  float* raw;        // [sum P] packed (b, h, j)
  float* pooled;     // same packing
  float2* stats;     // [total_pieces * 512] partial (running max, sum of exp) per piece and row
  float* lse;        // [nseq * H_kv * Wp] natural-log LSE per (sequence, head, row)
  const float* lse_in;  // caller's window LSE [B, W, H_q] (natural log), or null
  const void* q_all;     // all-query scoring: every prompt query [T, H_q, d], or null
  const float* lse_all;  // and its rows' natural-log LSE [T, H_q]
  // output heads: H_kv (scores averaged over each KV head's query group), or
  // H_q when every query head selects for itself (head_div = g: output head
  // o gathers KV head o / head_div)
  int out_heads, head_div;
  int v_zero_copy;  // v is page-locked host memory read in place (plain loads only)
  int gpu_share;  // n > 1: n such calls run side by side, the score kernel takes 1/n of the SMs
  int* status;       // device status word
  int* counters;     // work-queue head and per-group completion counters
  long long total_rows;  // rows of k / v in the whole call (T)
  int batch;         // sequences in the whole call (B)
  SeqInfo seq[kGroupSeqs];
};

// Adds n to the library's process-wide kernel-launch counter.
void count_launches(int n);

// Per-path count of scoring launches (one per pass-2 sweep over K): the
// tcgen05 kernel or the CUDA-core kernels.  Values match snapkv.h's
// SNAPKV_SCORE_PATH_* constants.
constexpr int kScorePathTensorCores = 0;
constexpr int kScorePathCudaCores = 1;
void count_score_launches(int path, int n);

// Attributes of the calling thread's current device, looked up once per
// device under a lock: concurrent first calls from several host threads are
// safe, and a process that drives GPUs of different kinds plans each launch
// with its own device's values.  Null if the query fails.
struct DeviceInfo {
  int sms;         // streaming multiprocessors
  int smem_optin;  // largest dynamic shared memory per block (opt-in), bytes
};
const DeviceInfo* current_device_info();

// Launchers (each returns a cudaError_t as int).
int launch_score_simt(const Plan& p, void* stream);
int launch_select_gather(const Plan& p, void* stream);
int launch_score_allq(const Plan& p, void* stream);

}  // namespace snapkv
