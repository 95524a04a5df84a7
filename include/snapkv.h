/*
 * snapkv.h - C ABI of the GB300 (sm_103a) SnapKV prefill-time KV-cache
 * compression library (libsnapkv.so).
 *
 * What the library computes, for each sequence b (prompt length L) and each
 * KV head h, with W the observation window and C the total budget:
 *
 *   - the last W prompt queries (the observation window) attend over the
 *     prompt keys with softmax(q.k / sqrt(d)) under the causal mask
 *     (jisaku.com glossary "SnapKV", section "SnapKVの仕組み": Observation
 *     Window and the algorithm flow, steps 1-2);
 *   - each prefix key j < P = L - W gets the sum of its probabilities over
 *     the window rows, averaged over the g = H_q / H_kv query heads of the KV
 *     group (hotpaper.ai summary of "SnapKV: LLM Knows What You are Looking
 *     for Before Generation": abstract and "핵심 아이디어", per-head selection;
 *     the glossary's FAQ Q1 on MHA and GQA models);
 *   - the scores are pooled (stride 1, kernel_size // 2 zeros of padding,
 *     average divides by kernel_size, or maximum) (glossary, "Pooling for
 *     Robustness"; summary, "기술적 접근법": max or average pooling, kernel
 *     5-13);
 *   - the C - W best prefix positions are kept, ties to the lower position
 *     (glossary, algorithm flow step 3: keep the top-B pairs; summary,
 *     "기술적 접근법": compressed size 1024-4096);
 *   - the compressed cache holds the kept rows in ascending position, then
 *     the W window rows, plus their positions (glossary, step 4: decode uses
 *     the compressed cache).  When L <= C every position is kept.
 *
 * The same library also runs decode steps over a cache (snapkv_decode_attention
 * below) and Scissorhands decode-time eviction over a budgeted cache that can
 * start from the compressed one (scissorhands.h).
 *
 * The parameter names of the glossary's usage example map as follows:
 * window_size -> W, max_capacity_prompt -> C, kernel_size -> kernel_size,
 * pooling ("avgpool" / "maxpool") -> pool_type.
 *
 * Conventions for every entry point:
 *   - Device pointers are plain CUDA device addresses of the current device;
 *     host pointers are ordinary process memory.  The library keeps no
 *     pointer after a call returns and allocates no memory: the caller owns
 *     every buffer, including the workspace.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  snapkv_compress is asynchronous on that stream and never
 *     synchronizes.  Calls that share one workspace must not overlap in time.
 *   - Return values are snapkv_status codes.  An argument error returns
 *     before anything is enqueued.
 */
#ifndef SNAPKV_H
#define SNAPKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SNAPKV_OK = 0,
    SNAPKV_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned buffer */
    SNAPKV_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels cover */
    SNAPKV_ERR_WORKSPACE = 3,   /* workspace smaller than snapkv_workspace_size */
    SNAPKV_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
    SNAPKV_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up */
} snapkv_status;

typedef enum { SNAPKV_POOL_AVG = 0, SNAPKV_POOL_MAX = 1 } snapkv_pool;

typedef enum { SNAPKV_BF16 = 0, SNAPKV_FP32 = 1 } snapkv_dtype;

/*
 * Problem shape shared by all calls.
 *   batch        B >= 1 sequences (at most 4096)
 *   num_q_heads  H_q >= 1
 *   num_kv_heads H_kv >= 1, H_q % H_kv == 0 (g = H_q / H_kv)
 *   head_dim     d, one of 64 or 128
 *   dtype        element type of q_win, k, v, out_k, out_v (snapkv_dtype)
 */
typedef struct {
    int32_t batch;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t dtype;
} snapkv_shape;

/*
 * Bytes of device workspace snapkv_compress needs for this problem.
 * seqlens_host: host array of B prompt lengths.  Returns 0 if the arguments
 * are invalid (the same checks snapkv_compress makes).
 */
size_t snapkv_workspace_size(const snapkv_shape *shape, const int32_t *seqlens_host,
                             int32_t W, int32_t C);

/*
 * Compress one layer's prompt KV cache.
 *
 * Inputs (device, 16-byte aligned, element type shape->dtype):
 *   q_win  [B, W, H_q, d]  queries of positions L_b-W .. L_b-1 of each
 *                          sequence, exactly as the layer's attention uses
 *                          them (position encoding already applied)
 *   k, v   [T, H_kv, d]    packed prompt keys / values, T = sum of seqlens;
 *                          sequence b owns rows off_b .. off_b + L_b - 1 with
 *                          off_b = L_0 + ... + L_{b-1}
 * seqlens_host: host array of B lengths, each >= 1.
 * W >= 1 (window), C >= W (total budget per sequence and KV head),
 * kernel_size odd and >= 1 (1 = no pooling), pool_type a snapkv_pool.
 *
 * Outputs (device, 16-byte aligned):
 *   out_k, out_v [B, C, H_kv, d]  slot s of (b, h) holds the row of position
 *                                 out_idx[b, h, s]; slots with index -1 are
 *                                 zero-filled
 *   out_idx      [B, H_kv, C]     int32 positions within the sequence: the
 *                                 C - W kept prefix positions ascending, then
 *                                 L_b - W .. L_b - 1.  If L_b <= C: 0 .. L_b-1
 *                                 then -1.
 * workspace: device, 256-byte aligned, at least snapkv_workspace_size bytes.
 *
 * Errors: SNAPKV_ERR_INVALID_ARG for a null pointer, B < 1 or > 4096, any
 * L_b < 1, H_q % H_kv != 0, W < 1, C < W, an even or non-positive
 * kernel_size, an unknown pool_type or dtype, or a misaligned buffer;
 * SNAPKV_ERR_UNSUPPORTED for d not in {64, 128} or W * g > 256;
 * SNAPKV_ERR_WORKSPACE if workspace_bytes is too small; SNAPKV_ERR_CUDA if a
 * launch fails.  Nothing is enqueued when an error is returned.
 */
int snapkv_compress(const snapkv_shape *shape, const void *q_win, const void *k,
                    const void *v, const int32_t *seqlens_host, int32_t W,
                    int32_t kernel_size, int32_t pool_type, int32_t C, void *out_k,
                    void *out_v, int32_t *out_idx, void *workspace,
                    size_t workspace_bytes, void *stream);

/*
 * Only the scoring step of snapkv_compress (window attention sums with the
 * GQA mean; no pooling, selection or emission), with the same meaning of
 * every argument.  The raw scores land in the workspace where
 * snapkv_score_offsets says; the pooled-score region is not touched.
 * Useful on its own (score inspection) and to time the score kernel alone.
 * Errors as for snapkv_compress.
 */
int snapkv_score(const snapkv_shape *shape, const void *q_win, const void *k,
                 const int32_t *seqlens_host, int32_t W, int32_t C, void *workspace,
                 size_t workspace_bytes, void *stream);

/*
 * Selection variants (flags of the _ex entry points).
 *
 * SNAPKV_PER_QUERY_HEAD: every query head selects its own positions instead
 * of one selection per KV head from the group-averaged score (the pages
 * select "for each attention head": hotpaper.ai summary of "SnapKV: LLM
 * Knows What You are Looking for Before Generation", abstract; GQA support,
 * glossary "SnapKV" FAQ Q1).  Query head hq's raw score is its own window
 * sum, without the 1/g mean; pooling and selection are per query head, and
 * query head hq gathers the K and V rows of KV head hq / g.  The outputs then
 * have H_q heads: out_k, out_v [B, C, H_q, d], out_idx [B, H_q, C], and the
 * fp32 score vectors hold H_q * P_b values per sequence, packed (b, hq, j).
 * Needs g = H_q / H_kv <= 8 (else SNAPKV_ERR_UNSUPPORTED).  With g = 1 it is
 * exactly snapkv_compress.
 */
#define SNAPKV_PER_QUERY_HEAD 1

size_t snapkv_workspace_size_ex(const snapkv_shape *shape, const int32_t *seqlens_host,
                                int32_t W, int32_t C, int32_t flags);

int snapkv_score_offsets_ex(const snapkv_shape *shape, const int32_t *seqlens_host, int32_t W,
                            int32_t C, int32_t flags, size_t *raw_offset,
                            size_t *pooled_offset, size_t *count);

/* snapkv_compress with flags (0 = snapkv_compress).  Unknown flags are
 * SNAPKV_ERR_INVALID_ARG. */
int snapkv_compress_ex(const snapkv_shape *shape, const void *q_win, const void *k,
                       const void *v, const int32_t *seqlens_host, int32_t W,
                       int32_t kernel_size, int32_t pool_type, int32_t C, void *out_k,
                       void *out_v, int32_t *out_idx, void *workspace, size_t workspace_bytes,
                       void *stream, int32_t flags);

/*
 * All-query ("heavy hitter") scoring, a scoring variant: every prompt query
 * votes instead of the observation window -- the accumulated attention H2O
 * uses, the method the SnapKV summary compares against (hotpaper.ai summary,
 * "주요 결과").  For each prefix key j < P_b of KV head h:
 *
 *   raw[j] = (1/g) sum_{hq in group} sum_{i=j}^{L_b-1} exp(q_i . k_j / sqrt(d) - lse_all[i, hq])
 *
 * then pooling, selection and emission exactly as snapkv_compress.  The
 * cost is quadratic in the prompt (~L^2/2 * H_q * d multiply-adds), which is
 * why SnapKV looks only at a window.
 *   q_all    device, [T, H_q, d] (packed like k), element type shape->dtype,
 *            16-byte aligned: every prompt query.
 *   lse_all  device, fp32 [T, H_q], 4-byte aligned: natural-log LSE of each
 *            query row over the keys it sees (j <= i) with these q and k, as
 *            the prefill attention computes it; trusted, not checked.
 * Every other argument, the workspace and the outputs are those of
 * snapkv_compress (W = the recent window that is always kept).
 */
int snapkv_compress_all_queries(const snapkv_shape *shape, const void *q_all, const void *k,
                                const void *v, const float *lse_all,
                                const int32_t *seqlens_host, int32_t W, int32_t kernel_size,
                                int32_t pool_type, int32_t C, void *out_k, void *out_v,
                                int32_t *out_idx, void *workspace, size_t workspace_bytes,
                                void *stream);

/*
 * snapkv_compress and snapkv_score with the window rows' log-sum-exp given
 * by the caller.  The prefill attention that precedes SnapKV already
 * normalises every window query row over its causally visible keys (the
 * scoring rides along with prefill: jisaku.com glossary "SnapKV", FAQ Q3);
 * a caller that keeps that row normaliser passes it here and the library
 * skips the first of its two sweeps over K (the per-row max and sum of
 * exponentials), computing only the column sums of
 *   exp(q_i . k_j / sqrt(d) - lse_win[b, i, head]).
 *
 *   lse_win   device, fp32, [B, W, H_q] row-major, 4-byte aligned: natural-
 *             log LSE of window query i of sequence b and query head `head`,
 *             log(sum_{j <= L_b - W + i} exp(q . k_j / sqrt(d))) over the
 *             keys that query sees (its own position included), with q and
 *             k exactly the q_win and k passed here.  Rows of sequences with
 *             L_b <= C are not read.
 *
 * Every other argument, the workspace size, the outputs and the status
 * behaviour are those of snapkv_compress / snapkv_score.  The values are
 * trusted, not checked: a wrong LSE gives wrong scores (an LSE far below
 * the true one can overflow them to +inf).  lse_win == NULL is
 * SNAPKV_ERR_INVALID_ARG.
 */
int snapkv_compress_with_lse(const snapkv_shape *shape, const void *q_win, const void *k,
                             const void *v, const float *lse_win,
                             const int32_t *seqlens_host, int32_t W, int32_t kernel_size,
                             int32_t pool_type, int32_t C, void *out_k, void *out_v,
                             int32_t *out_idx, void *workspace, size_t workspace_bytes,
                             void *stream);

int snapkv_score_with_lse(const snapkv_shape *shape, const void *q_win, const void *k,
                          const float *lse_win, const int32_t *seqlens_host, int32_t W,
                          int32_t C, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Where the last snapkv_compress on this workspace left its fp32 score
 * vectors.  For every sequence with L_b > C and every KV head, the P_b =
 * L_b - W raw scores (window sums, group mean) and pooled scores are packed
 * in (b, h, j) order; a sequence with L_b <= C has no scores and takes no
 * room.  *raw_offset / *pooled_offset receive byte offsets into the
 * workspace; *count receives the number of floats in each vector.
 */
int snapkv_score_offsets(const snapkv_shape *shape, const int32_t *seqlens_host, int32_t W,
                         int32_t C, size_t *raw_offset, size_t *pooled_offset,
                         size_t *count);

/*
 * Several device-resident layers in one call, consecutive layers overlapping:
 * layer l is enqueued on layer_streams[l % n_streams] with its own part of
 * the workspace, and each layer's score kernel runs on 1/n_streams of the
 * SMs, so that n_streams layers' latency-bound scoring chains (pass 1 ->
 * merge -> pass 2) and their selections run side by side.  Same outputs,
 * bit for bit, as snapkv_compress on each layer.  The call forks the layer
 * streams off
 * `stream` (events[0]) and joins them back (events[1 .. n_streams]), so work
 * enqueued on `stream` afterwards sees every layer's outputs; it works under
 * stream capture.  Asynchronous; nothing is allocated.  With lse_win each
 * layer's outputs equal snapkv_compress_with_lse's instead.
 *
 *   n_layers       >= 1
 *   q_win, k, v    host arrays of n_layers device pointers, each a layer's
 *                  input as in snapkv_compress (all layers share shape,
 *                  seqlens_host, W, kernel_size, pool_type and C)
 *   lse_win        NULL (the call computes the window rows' LSE, as
 *                  snapkv_compress), or a host array of n_layers device
 *                  pointers, each a layer's lse_win as in
 *                  snapkv_compress_with_lse (pass 2 only)
 *   out_k, out_v, out_idx  host arrays of n_layers device pointers
 *   workspace      device, 256-byte aligned, >= snapkv_workspace_size_layers
 *                  bytes for n_streams (n_streams single-layer workspaces
 *                  back to back)
 *   stream         the caller's cudaStream_t
 *   n_streams      1 .. SNAPKV_MAX_LAYER_STREAMS; each layer's score kernel takes
 *                  1/n_streams of the SMs (4 measured best on GB300)
 *   layer_streams  array of n_streams distinct cudaStream_t of the current
 *                  device, owned by the caller (non-blocking streams
 *                  recommended)
 *   events         array of n_streams + 1 cudaEvent_t created by the caller
 *                  (the library creates none)
 * One status word serves the whole call: snapkv_get_status on `workspace`
 * reports SNAPKV_ERR_TIMEOUT if any layer's bounded device wait gave up.
 * Returns SNAPKV_OK once every layer is enqueued, or the error of the first
 * layer that could not be (the streams are joined either way); argument
 * errors return before anything is enqueued.  snapkv_workspace_size_layers
 * returns 0 for an invalid problem or n_streams.
 */
#define SNAPKV_MAX_LAYER_STREAMS 8

size_t snapkv_workspace_size_layers(const snapkv_shape *shape, const int32_t *seqlens_host,
                                    int32_t W, int32_t C, int32_t n_streams);

int snapkv_compress_layers(const snapkv_shape *shape, int32_t n_layers,
                           const void *const *q_win, const void *const *k, const void *const *v,
                           const float *const *lse_win, const int32_t *seqlens_host, int32_t W,
                           int32_t kernel_size, int32_t pool_type, int32_t C,
                           void *const *out_k, void *const *out_v,
                           int32_t *const *out_idx, void *workspace, size_t workspace_bytes,
                           void *stream, int32_t n_streams, void *const *layer_streams,
                           void *const *events);

/*
 * Synchronize `stream`, then read the device status word that the kernels
 * of the last snapkv_compress on this workspace wrote: SNAPKV_OK, or
 * SNAPKV_ERR_TIMEOUT if a bounded device-side wait gave up.
 */
int snapkv_get_status(const void *workspace, size_t workspace_bytes, void *stream);

/*
 * Host-buffer variant.  Inputs and outputs are host arrays with the layouts
 * of snapkv_compress (page-locked memory makes the copies asynchronous and
 * fast).  The call copies q_win and k to `staging` on the device, runs the
 * compression there, copies out_k, out_v and out_idx back and waits for the
 * stream, so the outputs are complete when it returns.  Only the kept rows
 * of v are ever read: page-locked v is read in place by the gather (those
 * rows cross the host link, the rest never move); pageable v is copied to
 * staging whole.  staging: device, 256-byte aligned, at least
 * snapkv_host_staging_size bytes.
 */
size_t snapkv_host_staging_size(const snapkv_shape *shape, const int32_t *seqlens_host,
                                int32_t W, int32_t C);

int snapkv_compress_host(const snapkv_shape *shape, const void *q_win_host,
                         const void *k_host, const void *v_host,
                         const int32_t *seqlens_host, int32_t W, int32_t kernel_size,
                         int32_t pool_type, int32_t C, void *out_k_host, void *out_v_host,
                         int32_t *out_idx_host, void *staging, size_t staging_bytes,
                         void *stream);

/*
 * Several layers through host buffers, with the host-to-device copies of one
 * layer overlapping the compression of the previous one.  Equivalent to
 * snapkv_compress_host on each layer in turn (same outputs, bit for bit), but
 * the inputs of layer l + 1 upload on `copy_stream` while layer l compresses
 * on `stream`, through two staging slots; the call waits for both streams
 * once, after the last layer.
 *
 *   n_layers     >= 1
 *   q_win_host, k_host, v_host          arrays of n_layers host pointers, each
 *                                        a layer's input as in snapkv_compress_host
 *                                        (page-locked v is read in place)
 *   out_k_host, out_v_host, out_idx_host arrays of n_layers host pointers
 *   staging      device, 256-byte aligned, >= snapkv_host_staging_size_layers
 *   stream, copy_stream  two different cudaStream_t of the current device
 *   events       array of 4 cudaEvent_t created by the caller (the library
 *                creates none); recorded and waited on by the call
 * Returns SNAPKV_OK when every layer's outputs are complete, or the error of
 * the first layer that failed (earlier layers' outputs may then have been
 * written); argument errors return before anything is enqueued.
 */
size_t snapkv_host_staging_size_layers(const snapkv_shape *shape, const int32_t *seqlens_host,
                                       int32_t W, int32_t C);

int snapkv_compress_host_layers(const snapkv_shape *shape, int32_t n_layers,
                                const void *const *q_win_host, const void *const *k_host,
                                const void *const *v_host, const int32_t *seqlens_host,
                                int32_t W, int32_t kernel_size, int32_t pool_type, int32_t C,
                                void *const *out_k_host, void *const *out_v_host,
                                int32_t *const *out_idx_host, void *staging,
                                size_t staging_bytes, void *stream, void *copy_stream,
                                void *const *events);

/*
 * Number of CUDA kernels this library has launched in this process so far
 * (all devices, all streams), for launch accounting.
 */
uint64_t snapkv_kernel_launches(void);

/*
 * Which scoring path ran.  Scoring runs on the 5th-generation tensor cores
 * (one tcgen05 kernel) for bf16 with d in {64, 128} and W * g in {128, 256},
 * and on the CUDA cores (FFMA kernels) for every other supported shape; the
 * choice depends on the shape only, never on a runtime condition.  This
 * returns how many scoring launches (one per sweep over K that produces the
 * scores) the process has made on `path` so far, all devices and streams:
 * SNAPKV_SCORE_PATH_TENSOR_CORES or SNAPKV_SCORE_PATH_CUDA_CORES; 0 for any
 * other value.
 */
#define SNAPKV_SCORE_PATH_TENSOR_CORES 0
#define SNAPKV_SCORE_PATH_CUDA_CORES 1

uint64_t snapkv_score_path_launches(int32_t path);

/*
 * snapkv_compress without a caller-provided workspace.  The SnapKV pages have
 * no counterpart to this entry point; it exists for callers that cannot call
 * cudaMalloc -- for example a plugin inside a serving engine whose device
 * memory is all owned by the engine's own pool, or a latency-critical path
 * that cannot afford cudaMalloc's implicit device-wide synchronisation.
 *
 * Arguments, outputs and results are exactly those of snapkv_compress; the
 * caller still provides q_win, k, v and the three output buffers.  The
 * scratch comes from a 16 MiB array built into the library's device image,
 * which every GPU that loads the library keeps until the process exits.
 * Problems whose snapkv_workspace_size exceeds 16 MiB are rejected with
 * SNAPKV_ERR_WORKSPACE before anything is enqueued (one Llama-3-8B-shaped
 * layer of 131072 tokens needs about 12.6 MB).  The call allocates nothing.
 *
 * Every call looks up the array's device address in the calling thread's
 * current CUDA context (a runtime query that allocates nothing), so a context
 * switch or a cudaDeviceReset between calls is safe.  The first call in a
 * context may load the library's device code: make it before any stream
 * capture.  All calls in a context share the one array and it keeps the last
 * call's contents: calls that may overlap on the GPU (other streams, other
 * host threads) race on it and must be serialised by the caller.
 * snapkv_get_status does not apply to this entry point; use
 * snapkv_noalloc_get_status.
 */
int snapkv_compress_noalloc(const snapkv_shape *shape, const void *q_win, const void *k,
                            const void *v, const int32_t *seqlens_host, int32_t W,
                            int32_t kernel_size, int32_t pool_type, int32_t C, void *out_k,
                            void *out_v, int32_t *out_idx, void *stream);

/*
 * Synchronize `stream`, then read the status word that the kernels of the
 * last snapkv_compress_noalloc in the current context wrote into the
 * built-in scratch: SNAPKV_OK, or SNAPKV_ERR_TIMEOUT if a bounded device-side
 * wait gave up (the outputs of that call are then incomplete).  Like the
 * entry point it serves, the SnapKV pages have no counterpart.  Returns
 * SNAPKV_ERR_CUDA if the synchronize or the read fails.
 */
int snapkv_noalloc_get_status(void *stream);

/*
 * ---- Decode step over a KV cache ----
 *
 * After compression the generation (decode) phase attends over the
 * compressed cache instead of the full one (jisaku.com glossary "SnapKV",
 * "SnapKVの仕組み", algorithm flow step 4), which relieves the memory-bandwidth
 * bound of decoding (glossary FAQ Q2; hotpaper.ai summary of "SnapKV: LLM
 * Knows What You are Looking for Before Generation", "주요 결과").
 * snapkv_decode_attention computes one decode step of attention for one
 * query token per sequence:
 *
 *   out[b, hq, :] = sum_j softmax_j(q[b, hq] . k[b, j, h] / sqrt(d)) v[b, j, h]
 *
 * with h = hq / g, over the lens[b] cached rows j of sequence b (no mask: the
 * caller appends the new token's own key and value to the cache if it is to
 * be attended).
 */
typedef enum {
  SNAPKV_CACHE_PACKED = 0, /* k, v [sum_b lens[b], H_kv, d]: sequences back to back
                              (the layout snapkv_compress takes: the full cache) */
  SNAPKV_CACHE_SLOTS = 1   /* k, v [B, C, H_kv, d]: sequence b's rows are its slots
                              0 .. lens[b]-1 (snapkv_compress's outputs, with
                              lens[b] = min(L_b, C)) */
} snapkv_cache_layout;

/*
 * Workspace bytes for snapkv_decode_attention (0 if the arguments are
 * invalid or unsupported).  lens_host: host, B entries.
 */
size_t snapkv_decode_workspace_size(const snapkv_shape *shape, const int32_t *lens_host,
                                    int32_t layout, int32_t C);

/*
 *   shape      B, H_q, H_kv (H_q / H_kv in {1, 2, 4, 8, 16}), d in {64, 128},
 *              dtype of q, k and v (bf16 or fp32).
 *   q          device, [B, H_q, d], 16-byte aligned.
 *   k_cache    device, layout per `layout`, 16-byte aligned; v_cache likewise.
 *   lens_host  host, B entries, each >= 1 (and <= C for SNAPKV_CACHE_SLOTS).
 *   C          slots per sequence for SNAPKV_CACHE_SLOTS (ignored otherwise).
 *   out        device, fp32 [B, H_q, d], 16-byte aligned.
 *   workspace  device, 16-byte aligned, >= snapkv_decode_workspace_size bytes.
 *   stream     cudaStream_t.
 * Returns SNAPKV_OK, SNAPKV_ERR_INVALID_ARG (null or misaligned pointer, bad
 * lens, layout or shape), SNAPKV_ERR_UNSUPPORTED (d or group size),
 * SNAPKV_ERR_WORKSPACE or SNAPKV_ERR_CUDA; nothing is enqueued on argument
 * errors.  Asynchronous; allocates nothing.
 */
int snapkv_decode_attention(const snapkv_shape *shape, const void *q, const void *k_cache,
                            const void *v_cache, int32_t layout, const int32_t *lens_host,
                            int32_t C, float *out, void *workspace, size_t workspace_bytes,
                            void *stream);

/*
 * Self-test of the bounded device-side waits (the SnapKV pages have no
 * counterpart; it lets the failure path be tested without faulting or
 * hanging a GPU).  Enqueues one kernel whose single thread waits, with the
 * same bounded wait the kernels use for their cross-CTA counters (2 s limit),
 * on a device flag in workspace: set_flag = 0 leaves the flag unset, so the
 * wait runs out and the status word becomes "timeout"; set_flag = 1 sets it
 * first, so the wait succeeds.  Read the outcome with snapkv_get_status on
 * the same workspace (SNAPKV_ERR_TIMEOUT or SNAPKV_OK).
 *   workspace  device, 256-byte aligned, >= 512 bytes (overwritten).
 * Returns SNAPKV_OK once enqueued, SNAPKV_ERR_INVALID_ARG, SNAPKV_ERR_CUDA.
 */
int snapkv_selftest_wait(void *workspace, size_t workspace_bytes, int32_t set_flag, void *stream);

/* Static text for a status code. */
const char *snapkv_status_string(int status);

/* Library version, e.g. 0x000100 for 0.1.0. */
int snapkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SNAPKV_H */
