/*
 * CPU oracle for SnapKV prefill-time KV-cache compression.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the compression computes, in fp64, with no blocking, no
 * fusion and no reordering.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code, header, table or
 * helper with the CUDA library, and the CUDA library never calls it.
 *
 * Method (sources: jisaku.com glossary "SnapKV", section "SnapKVの仕組み":
 * Observation Window, the algorithm flow and "Pooling for Robustness";
 * hotpaper.ai summary of "SnapKV: LLM Knows What You are Looking for Before
 * Generation": abstract, "핵심 아이디어", "기술적 접근법"):
 *
 *   1. The last W prompt tokens are the observation window.  Their queries
 *      attend (softmax(q.k / sqrt(d)), causal) over the prompt keys.
 *   2. For every prefix key j < P = L - W the attention probabilities are
 *      summed over the window queries; under grouped-query attention the
 *      sums of the g query heads of a KV group are averaged.
 *   3. The 1-D score is smoothed by pooling (kernel k, stride 1, k//2 zeros
 *      of padding on both sides; average divides by k; or maximum).
 *   4. The C - W prefix positions with the largest pooled score are kept
 *      (ties: lower position first), in ascending order, followed by the W
 *      window positions; K and V rows of those positions are emitted.
 *
 * Readings where the pages are silent (score form, mask, GQA mean, padding,
 * tie rule, output order, L <= C) are the ones stated at each step below.
 *
 * Parity pins: every function here is checked by the CPU test-suite against
 * closed forms, brute force (full causal softmax in torch), invariants and
 * library pooling/sorting routines.  No function is "parity unpinned".
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define REF_BF16 0
#define REF_FP32 1

#define REF_OK 0
#define REF_ERR_ARG 1
#define REF_ERR_NONFINITE 2
#define REF_ERR_NOMEM 3

#define REF_POOL_AVG 0
#define REF_POOL_MAX 1

/* Element i of a bf16 (uint16 bit pattern) or fp32 array, widened exactly. */
static double ref_elem(const void *base, int dtype, size_t i)
{
    float f;
    if (dtype == REF_BF16) {
        uint32_t bits = ((const uint16_t *)base)[i];
        bits <<= 16;
        memcpy(&f, &bits, sizeof f);
    } else {
        f = ((const float *)base)[i];
    }
    return (double)f;
}

/*
 * Steps 1-2 for one (sequence b, KV head h): raw[j] for j in [0, P).
 *
 * q_win: [B, W, H_q, d]; k: [T, H_kv, d] (packed, sequence b at rows
 * off .. off+L-1).  Window row i sits at position t = P + i and sees keys
 * 0..t (causal).  Its logits are s_j = (q . k_j) / sqrt(d); its softmax
 * denominator runs over all visible keys, window keys included.  Only the
 * prefix columns j < P are summed into raw.  KV head h serves query heads
 * h*g .. h*g+g-1; raw is divided by g (mean over the group).
 *
 * window_mass receives the probability the window rows put on the window
 * keys themselves (also divided by g), so that raw summed over j plus
 * window_mass equals W: a conservation check.
 */
int ref_scores_unit(const void *q_win, const void *k, int dtype, int W, int H_q,
                    int H_kv, int d, int b, int h, int L, long long off,
                    double *raw, double *window_mass)
{
    int P = L - W;
    int g;
    double *s;
    double wm = 0.0;
    if (P < 1 || H_kv < 1 || H_q % H_kv != 0 || d < 1)
        return REF_ERR_ARG;
    g = H_q / H_kv;
    s = (double *)malloc(sizeof(double) * (size_t)L);
    if (!s)
        return REF_ERR_NOMEM;
    for (int j = 0; j < P; j++)
        raw[j] = 0.0;
    for (int r = 0; r < g; r++) {
        int hq = h * g + r;
        for (int i = 0; i < W; i++) {
            int t = P + i; /* position of this window row */
            size_t qbase = (((size_t)b * W + i) * H_q + hq) * (size_t)d;
            double m = -INFINITY, Z = 0.0;
            for (int j = 0; j <= t; j++) {
                size_t kbase = (((size_t)(off + j)) * H_kv + h) * (size_t)d;
                double dot = 0.0;
                for (int c = 0; c < d; c++)
                    dot += ref_elem(q_win, dtype, qbase + c) * ref_elem(k, dtype, kbase + c);
                s[j] = dot / sqrt((double)d);
                if (!isfinite(s[j])) {
                    free(s);
                    return REF_ERR_NONFINITE;
                }
                if (s[j] > m)
                    m = s[j];
            }
            for (int j = 0; j <= t; j++)
                Z += exp(s[j] - m);
            for (int j = 0; j < P; j++)
                raw[j] += exp(s[j] - m) / Z;
            for (int j = P; j <= t; j++)
                wm += exp(s[j] - m) / Z;
        }
    }
    for (int j = 0; j < P; j++)
        raw[j] /= (double)g;
    *window_mass = wm / (double)g;
    free(s);
    return REF_OK;
}

/*
 * ref_scores_unit with its window rows spread over nthreads POSIX threads,
 * giving the same doubles bit for bit: each row's logits, maximum, sum and
 * probabilities are computed by the same expressions in the same order as
 * there, and kept; the per-key sums then add the rows in the same order
 * (query head major, window row minor), starting from zero, and the window
 * mass adds the same terms in the same order.  Only the work is split.
 */
typedef struct {
    const void *q_win, *k;
    int dtype, W, H_q, H_kv, d, b, h, L, P, g;
    long long off;
    double *prob;  /* [W*g][P]   probabilities of the prefix keys per row */
    double *win;   /* [W*g][W]   probabilities of the window keys per row */
    double *raw;
    int nthreads, status;
} ref_rows_job;

typedef struct {
    ref_rows_job *job;
    int tid;
} ref_rows_arg;

static void *ref_rows_worker(void *p)
{
    ref_rows_arg *a = (ref_rows_arg *)p;
    ref_rows_job *J = a->job;
    int W = J->W, d = J->d, P = J->P, g = J->g;
    double *s = (double *)malloc(sizeof(double) * (size_t)J->L);
    if (!s) {
        J->status = REF_ERR_NOMEM;
        return NULL;
    }
    for (int row = a->tid; row < W * g; row += J->nthreads) {
        int r = row / W, i = row % W; /* rows ordered query head major */
        int hq = J->h * g + r;
        int t = P + i;
        size_t qbase = (((size_t)J->b * W + i) * J->H_q + hq) * (size_t)d;
        double m = -INFINITY, Z = 0.0;
        for (int j = 0; j <= t; j++) {
            size_t kbase = (((size_t)(J->off + j)) * J->H_kv + J->h) * (size_t)d;
            double dot = 0.0;
            for (int c = 0; c < d; c++)
                dot += ref_elem(J->q_win, J->dtype, qbase + c) * ref_elem(J->k, J->dtype, kbase + c);
            s[j] = dot / sqrt((double)d);
            if (!isfinite(s[j])) {
                J->status = REF_ERR_NONFINITE;
                free(s);
                return NULL;
            }
            if (s[j] > m)
                m = s[j];
        }
        for (int j = 0; j <= t; j++)
            Z += exp(s[j] - m);
        for (int j = 0; j < P; j++)
            J->prob[(size_t)row * P + j] = exp(s[j] - m) / Z;
        for (int j = P; j <= t; j++)
            J->win[(size_t)row * W + (j - P)] = exp(s[j] - m) / Z;
    }
    free(s);
    return NULL;
}

static void *ref_keys_worker(void *p)
{
    ref_rows_arg *a = (ref_rows_arg *)p;
    ref_rows_job *J = a->job;
    int rows = J->W * J->g, P = J->P;
    int per = (P + J->nthreads - 1) / J->nthreads;
    int j0 = a->tid * per, j1 = j0 + per < P ? j0 + per : P;
    for (int j = j0; j < j1; j++) {
        double acc = 0.0;
        for (int row = 0; row < rows; row++)
            acc += J->prob[(size_t)row * P + j];
        J->raw[j] = acc / (double)J->g;
    }
    return NULL;
}

int ref_scores_unit_mt(const void *q_win, const void *k, int dtype, int W, int H_q, int H_kv,
                       int d, int b, int h, int L, long long off, double *raw,
                       double *window_mass, int nthreads)
{
    ref_rows_job J;
    pthread_t th[256];
    ref_rows_arg args[256];
    int P = L - W;
    if (nthreads <= 1)
        return ref_scores_unit(q_win, k, dtype, W, H_q, H_kv, d, b, h, L, off, raw, window_mass);
    if (P < 1 || H_kv < 1 || H_q % H_kv != 0 || d < 1)
        return REF_ERR_ARG;
    if (nthreads > 256)
        nthreads = 256;
    memset(&J, 0, sizeof J);
    J.q_win = q_win; J.k = k; J.dtype = dtype; J.W = W; J.H_q = H_q; J.H_kv = H_kv;
    J.d = d; J.b = b; J.h = h; J.L = L; J.P = P; J.g = H_q / H_kv; J.off = off;
    J.raw = raw; J.nthreads = nthreads;
    J.prob = (double *)malloc(sizeof(double) * (size_t)W * J.g * (size_t)P);
    J.win = (double *)malloc(sizeof(double) * (size_t)W * J.g * (size_t)W);
    if (!J.prob || !J.win) { /* not enough memory to keep the rows: one thread */
        free(J.prob);
        free(J.win);
        return ref_scores_unit(q_win, k, dtype, W, H_q, H_kv, d, b, h, L, off, raw, window_mass);
    }
    for (int t = 0; t < nthreads; t++) {
        args[t].job = &J;
        args[t].tid = t;
        pthread_create(&th[t], NULL, ref_rows_worker, &args[t]);
    }
    for (int t = 0; t < nthreads; t++)
        pthread_join(th[t], NULL);
    if (!J.status) {
        double wm = 0.0;
        for (int t = 0; t < nthreads; t++)
            pthread_create(&th[t], NULL, ref_keys_worker, &args[t]);
        for (int t = 0; t < nthreads; t++)
            pthread_join(th[t], NULL);
        for (int row = 0; row < W * J.g; row++)
            for (int i = 0; i < (row % W) + 1; i++)
                wm += J.win[(size_t)row * W + i];
        *window_mass = wm / (double)J.g;
    }
    free(J.prob);
    free(J.win);
    return J.status;
}

/*
 * Step 3: 1-D pooling of raw[0..P) with kernel kp (odd), stride 1 and kp/2
 * zeros of padding on each side.  Average: window sum / kp (the zeros count,
 * at the edges too).  Maximum: largest value in the zero-padded window.
 */
int ref_pool(const double *raw, int P, int kp, int pool_type, double *pooled)
{
    int r = kp / 2;
    if (P < 0 || kp < 1 || (kp % 2) == 0)
        return REF_ERR_ARG;
    if (pool_type != REF_POOL_AVG && pool_type != REF_POOL_MAX)
        return REF_ERR_ARG;
    for (int j = 0; j < P; j++) {
        double acc = 0.0, mx = -INFINITY;
        for (int t = j - r; t <= j + r; t++) {
            double x = (t >= 0 && t < P) ? raw[t] : 0.0;
            acc += x;
            if (x > mx)
                mx = x;
        }
        pooled[j] = (pool_type == REF_POOL_AVG) ? acc / (double)kp : mx;
    }
    return REF_OK;
}

typedef struct {
    double score;
    int pos;
} ref_item;

/* Order by score descending, then position ascending (ties: lower first). */
static int ref_item_cmp(const void *a, const void *b)
{
    const ref_item *x = (const ref_item *)a, *y = (const ref_item *)b;
    if (x->score > y->score)
        return -1;
    if (x->score < y->score)
        return 1;
    return (x->pos > y->pos) - (x->pos < y->pos);
}

static int ref_int_cmp(const void *a, const void *b)
{
    int x = *(const int *)a, y = *(const int *)b;
    return (x > y) - (x < y);
}

/*
 * Step 4a: the n best positions of pooled[0..P) by (score desc, position
 * asc), returned in ascending position order.  *tau is the score of the
 * n-th best (NAN when n == 0).
 */
int ref_select(const double *pooled, int P, int n, int *sel, double *tau)
{
    ref_item *items;
    if (n < 0 || n > P)
        return REF_ERR_ARG;
    items = (ref_item *)malloc(sizeof(ref_item) * (size_t)(P > 0 ? P : 1));
    if (!items)
        return REF_ERR_NOMEM;
    for (int j = 0; j < P; j++) {
        items[j].score = pooled[j];
        items[j].pos = j;
    }
    qsort(items, (size_t)P, sizeof(ref_item), ref_item_cmp);
    for (int s = 0; s < n; s++)
        sel[s] = items[s].pos;
    *tau = n > 0 ? items[n - 1].score : NAN;
    qsort(sel, (size_t)n, sizeof(int), ref_int_cmp);
    free(items);
    return REF_OK;
}

/* Problem shared by the worker threads of ref_compress. */
typedef struct {
    const void *q_win, *k, *v;
    int dtype, B, W, H_q, H_kv, d, kp, pool_type, C;
    const int *seqlens;
    const long long *offs;        /* first packed row of each sequence */
    const long long *score_offs;  /* per (b, h): offset into pooled / raw */
    double *raw, *pooled, *tau, *window_mass;
    void *out_k, *out_v;
    int *out_idx;
    int nthreads;
    int inner;  /* threads per unit's scores (units run one at a time when > 1) */
    int status;
    pthread_mutex_t lock;
} ref_job;

/* Steps 1-4 plus emission for one (b, h). */
static int ref_compress_unit(ref_job *J, int b, int h)
{
    int L = J->seqlens[b], W = J->W, C = J->C, d = J->d;
    int P = L - W, n = C - W;
    size_t esz = J->dtype == REF_BF16 ? 2 : 4;
    size_t row = (size_t)d * esz;
    int *idx = J->out_idx + ((size_t)b * J->H_kv + h) * (size_t)C;
    long long so = J->score_offs[(size_t)b * J->H_kv + h];
    int rc;
    if (L <= C) {
        /* keep every position, in order; unused slots: index -1, zero rows */
        for (int s = 0; s < C; s++)
            idx[s] = s < L ? s : -1;
        J->tau[(size_t)b * J->H_kv + h] = NAN;
        if (P >= 1) {
            /* scores are still defined and reported */
            rc = ref_scores_unit_mt(J->q_win, J->k, J->dtype, W, J->H_q, J->H_kv, d, b, h,
                                    L, J->offs[b], J->raw + so,
                                    J->window_mass + (size_t)b * J->H_kv + h, J->inner);
            if (rc)
                return rc;
            rc = ref_pool(J->raw + so, P, J->kp, J->pool_type, J->pooled + so);
            if (rc)
                return rc;
        }
    } else {
        double tau;
        rc = ref_scores_unit_mt(J->q_win, J->k, J->dtype, W, J->H_q, J->H_kv, d, b, h, L,
                                J->offs[b], J->raw + so,
                                J->window_mass + (size_t)b * J->H_kv + h, J->inner);
        if (rc)
            return rc;
        rc = ref_pool(J->raw + so, P, J->kp, J->pool_type, J->pooled + so);
        if (rc)
            return rc;
        rc = ref_select(J->pooled + so, P, n, idx, &tau);
        if (rc)
            return rc;
        J->tau[(size_t)b * J->H_kv + h] = tau;
        for (int s = n; s < C; s++)
            idx[s] = P + (s - n); /* the window rows, in order */
    }
    for (int s = 0; s < C; s++) {
        size_t dst = (((size_t)b * C + s) * J->H_kv + h) * row;
        if (idx[s] < 0) {
            memset((char *)J->out_k + dst, 0, row);
            memset((char *)J->out_v + dst, 0, row);
        } else {
            size_t src = ((size_t)(J->offs[b] + idx[s]) * J->H_kv + h) * row;
            memcpy((char *)J->out_k + dst, (const char *)J->k + src, row);
            memcpy((char *)J->out_v + dst, (const char *)J->v + src, row);
        }
    }
    return REF_OK;
}

typedef struct {
    ref_job *job;
    int tid;
} ref_worker_arg;

static void *ref_worker(void *p)
{
    ref_worker_arg *a = (ref_worker_arg *)p;
    ref_job *J = a->job;
    int units = J->B * J->H_kv;
    for (int u = a->tid; u < units; u += J->nthreads) {
        int rc = ref_compress_unit(J, u / J->H_kv, u % J->H_kv);
        if (rc) {
            pthread_mutex_lock(&J->lock);
            if (!J->status)
                J->status = rc;
            pthread_mutex_unlock(&J->lock);
        }
    }
    return NULL;
}

/*
 * The whole compression of one layer.
 *
 * score_offs[b*H_kv+h] locates unit (b, h)'s P = L_b - W values inside raw
 * and pooled (units with P < 1 have none).  tau and window_mass are
 * [B*H_kv].  out_k / out_v: [B, C, H_kv, d] in the input element type;
 * out_idx: [B, H_kv, C] int32.  Units run on nthreads POSIX threads.
 */
int ref_compress(const void *q_win, const void *k, const void *v, int dtype, int B, int W,
                 int H_q, int H_kv, int d, const int *seqlens, const long long *offs,
                 const long long *score_offs, int kp, int pool_type, int C, double *raw,
                 double *pooled, double *tau, double *window_mass, void *out_k, void *out_v,
                 int *out_idx, int nthreads)
{
    ref_job J;
    pthread_t *th;
    ref_worker_arg *args;
    if (B < 1 || W < 1 || C < W || H_kv < 1 || H_q % H_kv || kp < 1 || kp % 2 == 0)
        return REF_ERR_ARG;
    if (dtype != REF_BF16 && dtype != REF_FP32)
        return REF_ERR_ARG;
    if (nthreads < 1)
        nthreads = 1;
    memset(&J, 0, sizeof J);
    J.q_win = q_win; J.k = k; J.v = v; J.dtype = dtype; J.B = B; J.W = W;
    J.H_q = H_q; J.H_kv = H_kv; J.d = d; J.kp = kp; J.pool_type = pool_type; J.C = C;
    J.seqlens = seqlens; J.offs = offs; J.score_offs = score_offs;
    J.raw = raw; J.pooled = pooled; J.tau = tau; J.window_mass = window_mass;
    J.out_k = out_k; J.out_v = out_v; J.out_idx = out_idx; J.nthreads = nthreads;
    J.inner = 1;
    if (B * H_kv < nthreads) { /* fewer units than threads: one unit at a time, all threads on it */
        J.inner = nthreads;
        J.nthreads = nthreads = 1;
    }
    pthread_mutex_init(&J.lock, NULL);
    th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    args = (ref_worker_arg *)malloc(sizeof(ref_worker_arg) * (size_t)nthreads);
    if (!th || !args) {
        free(th);
        free(args);
        return REF_ERR_NOMEM;
    }
    for (int t = 0; t < nthreads; t++) {
        args[t].job = &J;
        args[t].tid = t;
        pthread_create(&th[t], NULL, ref_worker, &args[t]);
    }
    for (int t = 0; t < nthreads; t++)
        pthread_join(th[t], NULL);
    pthread_mutex_destroy(&J.lock);
    free(th);
    free(args);
    return J.status;
}
