// Internal interface between the Scissorhands step (scissorhands.cu) and the
// decode-attention kernels (decode.cu) it reuses.
#pragma once

#include <cstddef>

#include <cuda_runtime.h>

namespace snapkv {

struct ShAttention {
  int B, H_q, H_kv, d, dtype;
  int cap;            // slots per sequence (budget + 1)
  int budget, evict;  // rows after the step: n + 1, less evict when above budget
  const void* q;      // [B, H_q, d]
  const void* k;      // [B, cap, H_kv, d]
  const void* v;
  const int* state;   // [B, 4] device cache state, as it was before the step
  float* out;         // [B, H_q, d]
  float* part_o;      // split-K partials, sh_attention_units() * g * d floats
  float2* part_ml;    // sh_attention_units() * g
  float* logits;      // [B, H_kv, cap, g]
  float2* ml;         // [B, H_q]
};

// Upper bound on the split-K units of one launch group.
size_t sh_attention_units(int B, int cap, int H_kv);

// Enqueues decode_chunk + decode_combine in their Scissorhands instantiation;
// returns a cudaError_t as int.
int launch_sh_attention(const ShAttention& a, void* stream);

}  // namespace snapkv
