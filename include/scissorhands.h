/*
 * scissorhands.h - Scissorhands decode-time KV-cache eviction in libsnapkv.so
 * (GB300, sm_103a).
 *
 * What it computes follows the abeam.tech summary of "Scissorhands:
 * Exploiting the Persistence of Importance Hypothesis for LLM KV Cache
 * Compression at Test Time", section 技術の仕組み:
 *
 *   - every KV head keeps at most `budget` tokens ("固定予算で残すトークンを
 *     選ぶ");
 *   - each decode step appends the new token's key and value; when that takes
 *     the cache past the budget, a batch of `evict` tokens is dropped (the
 *     page's setting: half the budget, "層ごと・ヘッドごとの予算配分") before
 *     the step attends, so attention always runs over at most `budget` rows;
 *   - the tokens dropped are those whose attention weight was below the
 *     average weight 1/n most often over the last `history` (w) decode steps;
 *     equal counts drop the older token first; the `recent` (r) newest tokens
 *     are never dropped (the page's runs: w = 400, r = 10);
 *   - with grouped-query attention a token's weight for a KV head is the mean
 *     of its weights over the g query heads the KV head serves;
 *   - the step's output is ordinary softmax attention over the rows that
 *     remain, one query token per sequence:
 *       out[b, hq] = sum_j softmax_j(q[b, hq] . k[b, j, h] / sqrt(d)) v[b, j, h].
 *
 * Budgets may differ per layer: each layer has its own cache and parameters.
 * The cache starts from any prefix of at most `budget` tokens per head, for
 * example the compressed cache snapkv_compress emits.
 *
 * The whole cache state lives in device memory, so scissorhands_step makes no
 * decision on the host, reads nothing back and may be captured in a CUDA
 * graph and replayed step after step.  Conventions (device pointers, streams,
 * status codes, no allocation) are those of snapkv.h.
 */
#ifndef SCISSORHANDS_H
#define SCISSORHANDS_H

#include "snapkv.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 *   budget   tokens kept per KV head, 1 .. 16383
 *   recent   r, newest tokens never evicted, 1 .. budget
 *   history  w, decode steps a token's count looks back over, 1 .. 1024
 *   evict    m, tokens evicted per head in one batch, 1 .. budget + 1 - recent
 */
typedef struct {
    int32_t budget;
    int32_t recent;
    int32_t history;
    int32_t evict;
} scissorhands_params;

/*
 * One layer's cache: caller-owned device buffers, sized by
 * scissorhands_buffer_bytes, 16-byte aligned.  S = budget + 1 slots per
 * sequence; HW = ceil(history / 32) words of history per slot.
 *   k, v   [B, S, H_kv, d] in shape->dtype.  Slot s of head h holds that
 *          head's s-th oldest cached token; heads hold different tokens but
 *          the same number n[b] of them (slots n[b] .. S-1 are unused).
 *   pos    int32 [B, H_kv, S]: the position of each slot's token.
 *   hist   uint32 [B, H_kv, HW, S]: with u = t mod history, bit u % 32 of
 *          word u / 32 of a slot is 1 when the slot's token was below average
 *          at decode step t.  The words hold the last `history` steps; a new
 *          slot starts at zero.
 *   state  int32 [B, 4]: per sequence { n (tokens cached), t (decode steps
 *          taken), next position, 0 }.
 */
typedef struct {
    void *k;
    void *v;
    int32_t *pos;
    uint32_t *hist;
    int32_t *state;
} scissorhands_cache;

typedef enum {
    SCISSORHANDS_BUF_K = 0,
    SCISSORHANDS_BUF_V = 1,
    SCISSORHANDS_BUF_POS = 2,
    SCISSORHANDS_BUF_HIST = 3,
    SCISSORHANDS_BUF_STATE = 4
} scissorhands_buffer;

/* Bytes of one cache buffer (0 if the arguments are invalid or unsupported). */
size_t scissorhands_buffer_bytes(const snapkv_shape *shape, const scissorhands_params *params,
                                 int32_t which);

/* Workspace bytes for scissorhands_step (0 if invalid or unsupported). */
size_t scissorhands_workspace_size(const snapkv_shape *shape, const scissorhands_params *params);

/*
 * Loads a prefix into the cache and resets its state and history.
 *   shape       B, H_q, H_kv (H_q / H_kv in {1, 2, 4, 8, 16}), d in {64, 128},
 *               bf16 or fp32.
 *   k0, v0      device, [B, C0, H_kv, d] in shape->dtype (snapkv_compress's
 *               out_k / out_v layout); may be NULL when every lens0 is 0.
 *   C0          slots per sequence of k0 / v0 (>= max lens0).
 *   pos0        device int32 [B, H_kv, C0] positions of the prefix rows
 *               (snapkv_compress's out_idx), or NULL for positions 0 .. n-1.
 *   lens0_host  host, B entries, 0 <= lens0[b] <= min(C0, budget): rows used.
 *   next_pos0_host  host, B entries >= 0: the position of each sequence's
 *               first decoded token (its prompt length).
 * Returns SNAPKV_OK once enqueued, SNAPKV_ERR_INVALID_ARG, SNAPKV_ERR_UNSUPPORTED
 * or SNAPKV_ERR_CUDA.  Copies lens0 / next_pos0 from host memory before it
 * returns (not capturable in a CUDA graph).
 */
int scissorhands_init(const snapkv_shape *shape, const scissorhands_params *params,
                      const scissorhands_cache *cache, const void *k0, const void *v0,
                      int32_t C0, const int32_t *pos0, const int32_t *lens0_host,
                      const int32_t *next_pos0_host, void *stream);

/*
 * One decode step of one layer: append k_new / v_new at each sequence's next
 * position, evict `evict` tokens per head where the cache then holds
 * budget + 1, attend, record which tokens were below average, advance the
 * state.
 *   q          device [B, H_q, d] in shape->dtype (the step's queries).
 *   k_new      device [B, H_kv, d] in shape->dtype; v_new likewise.
 *   out        device fp32 [B, H_q, d].
 *   workspace  device, 256-byte aligned, >= scissorhands_workspace_size bytes.
 * Returns SNAPKV_OK once enqueued, SNAPKV_ERR_INVALID_ARG (null or misaligned
 * pointer, bad parameters), SNAPKV_ERR_UNSUPPORTED, SNAPKV_ERR_WORKSPACE or
 * SNAPKV_ERR_CUDA; nothing is enqueued on argument errors.  Four kernels,
 * asynchronous, no host synchronisation, no allocation.
 */
int scissorhands_step(const snapkv_shape *shape, const scissorhands_params *params,
                      const scissorhands_cache *cache, const void *q, const void *k_new,
                      const void *v_new, float *out, void *workspace, size_t workspace_bytes,
                      void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SCISSORHANDS_H */
