/*
 * attn_oracle.c -- plain fp64 CPU oracle for scaled dot-product attention
 * forward with grouped-query heads, causal / local-window limits, tanh
 * soft-capping, an additive f32 mask and ragged per-batch lengths.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: it is used by tests/, by __graft_entry__.smoke() and by
 * the cpu_baseline / reference leg of bench.py.  It shares no code, header,
 * table or helper with the CUDA library.
 *
 * What it computes (one output row per (b, h, qi)):
 *
 *   kvh        = h / (Hq / Hkv)                       grouped-query head
 *   lsk        = total_lengths ? total_lengths[b] : Sk
 *   causal_max = past_lengths ? past_lengths[b] + qi : lsk - Sq + qi
 *   local_min  = local_window > 0 ? max(0, causal_max + 1 - local_window) : 0
 *   key j in [0, Sk) is visible iff  j < lsk  and  j >= local_min
 *                                  and (causal == 0 or j <= causal_max)
 *   S[j] = -inf                                        if j is not visible
 *        = scale * sum_d Q[d] K[j,d]                   otherwise, then
 *          S[j] = softcap * tanh(S[j] / softcap)       if softcap > 0, then
 *          S[j] = S[j] + mask[plane, qi, j]            if a mask is given
 *   M = max_j S[j];  the row is 0 if M = -inf
 *   O[d] = sum_j exp(S[j] - M) V[j,d] / sum_j exp(S[j] - M)
 *   lse  = log sum_j exp(S[j]) = M + log sum_j exp(S[j] - M)   (-inf if M = -inf)
 *
 * Sources: "onnx-runtime-ep-cuda 0.1.0-dev.5, src/kernels/flash_attention.rs"
 * -- the kernel `flash_attention_body` (per-row limits, the masking rule, the
 * order scale -> soft-cap -> additive mask, the mask-plane choice, the zero
 * output of a row whose denominator is 0) and the test helper
 * `cpu_reference` (fp64 dot products over dtype-rounded inputs, full row,
 * max-subtracted softmax).  "pictor-kernels 0.1.0,
 * src/gpu_backend/cuda_imagen_attn_kernels.rs" -- module doc "The op"
 * (full-row max-subtracted softmax, O = softmax(S) V, and the token-major
 * transposed output out[qi, h*D + d]).
 *
 * The pages leave some points open; the readings taken here:
 *  - lsk is used unclamped in causal_max (as the page's kernel does); only
 *    visibility is bounded by Sk, because the page's key loop stops at Sk.
 *  - The mask is f32 [mask_planes, Sq, Sk] with row stride Sk.  Plane
 *    choice follows the page: b when mask_planes == B, b*Hq + h when
 *    mask_planes == B*Hq, else plane 0.
 *  - Token-major output with a batch dimension is [B, Sq, Hq*D].
 *
 * Inputs are the dtype-rounded values held as float (every bf16 / f16 value is
 * exact in float); all arithmetic is double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const float *q, *k, *v, *mask;
    const int32_t *total_lengths, *past_lengths;
    int64_t B, Hq, Hkv, Sq, Sk, kv_capacity, D;
    int causal;
    int64_t local_window;
    double scale, softcap;
    int64_t mask_planes;
} problem_t;

/* One output row: the definition written out. `s` is scratch of Sk doubles.
 * Also returns the row's log-sum-exp of the scores in *lse. */
static void oracle_row(const problem_t *p, int64_t b, int64_t h, int64_t qi,
                       double *s, double *o, double *lse)
{
    const int64_t group = p->Hq / p->Hkv;
    const int64_t kvh = h / group;
    const int64_t lsk = p->total_lengths ? (int64_t)p->total_lengths[b] : p->Sk;
    const int64_t causal_max =
        p->past_lengths ? (int64_t)p->past_lengths[b] + qi : lsk - p->Sq + qi;
    int64_t local_min = 0;
    if (p->local_window > 0) {
        local_min = causal_max + 1 - p->local_window;
        if (local_min < 0) local_min = 0;
    }

    const float *qrow = p->q + ((b * p->Hq + h) * p->Sq + qi) * p->D;
    const int64_t kv_plane = (b * p->Hkv + kvh) * p->kv_capacity;

    int64_t plane = 0;
    if (p->mask_planes == p->B) plane = b;
    else if (p->mask_planes == p->B * p->Hq) plane = b * p->Hq + h;

    double m = -INFINITY;
    for (int64_t j = 0; j < p->Sk; ++j) {
        int visible = (j < lsk) && (j >= local_min) && !(p->causal && j > causal_max);
        if (!visible) {
            s[j] = -INFINITY;
            continue;
        }
        const float *krow = p->k + (kv_plane + j) * p->D;
        double dot = 0.0;
        for (int64_t d = 0; d < p->D; ++d) dot += (double)qrow[d] * (double)krow[d];
        double score = p->scale * dot;
        if (p->softcap > 0.0) score = p->softcap * tanh(score / p->softcap);
        if (p->mask && p->mask_planes > 0)
            score += (double)p->mask[(plane * p->Sq + qi) * p->Sk + j];
        s[j] = score;
        if (score > m) m = score;
    }

    for (int64_t d = 0; d < p->D; ++d) o[d] = 0.0;
    *lse = -INFINITY;
    if (m == -INFINITY) return; /* no finite visible score: the row is 0 */

    double l = 0.0;
    for (int64_t j = 0; j < p->Sk; ++j) {
        s[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
        l += s[j];
    }
    for (int64_t j = 0; j < p->Sk; ++j) {
        if (s[j] == 0.0) continue;
        const float *vrow = p->v + (kv_plane + j) * p->D;
        for (int64_t d = 0; d < p->D; ++d) o[d] += s[j] * (double)vrow[d];
    }
    for (int64_t d = 0; d < p->D; ++d) o[d] /= l;
    *lse = m + log(l);
}

typedef struct {
    const problem_t *p;
    const int64_t *rows; /* NULL: all rows, enumerated (b, h, qi) */
    int64_t n_rows, begin, end;
    double *out;
    double *lse;    /* NULL, or one value per row: [B,Hq,Sq] (rows == NULL) or [n_rows] */
    int out_layout; /* only used when rows == NULL */
    int failed;
} task_t;

static void *worker(void *arg)
{
    task_t *t = (task_t *)arg;
    const problem_t *p = t->p;
    double *s = (double *)malloc(sizeof(double) * (size_t)(p->Sk > 0 ? p->Sk : 1));
    if (!s) {
        t->failed = 1;
        return NULL;
    }
    for (int64_t r = t->begin; r < t->end; ++r) {
        int64_t b, h, qi;
        double *o, lse;
        if (t->rows) {
            b = t->rows[3 * r + 0];
            h = t->rows[3 * r + 1];
            qi = t->rows[3 * r + 2];
            o = t->out + r * p->D;
        } else {
            qi = r % p->Sq;
            h = (r / p->Sq) % p->Hq;
            b = r / (p->Sq * p->Hq);
            if (t->out_layout == 0)
                o = t->out + ((b * p->Hq + h) * p->Sq + qi) * p->D;
            else
                o = t->out + ((b * p->Sq + qi) * p->Hq + h) * p->D;
        }
        oracle_row(p, b, h, qi, s, o, &lse);
        if (t->lse) t->lse[t->rows ? r : (b * p->Hq + h) * p->Sq + qi] = lse;
    }
    free(s);
    return NULL;
}

static int run_tasks(const problem_t *p, const int64_t *rows, int64_t n_rows,
                     double *out, double *lse, int out_layout, int nthreads)
{
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    if (nthreads > 1024) nthreads = 1024;
    if ((int64_t)nthreads > n_rows) nthreads = n_rows > 0 ? (int)n_rows : 1;

    task_t *tasks = (task_t *)calloc((size_t)nthreads, sizeof(task_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!tasks || !tids) {
        free(tasks);
        free(tids);
        return 2;
    }
    const int64_t chunk = 16;
    int rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        tasks[i].p = p;
        tasks[i].rows = rows;
        tasks[i].n_rows = n_rows;
        tasks[i].out = out;
        tasks[i].lse = lse;
        tasks[i].out_layout = out_layout;
        tasks[i].begin = 0;
        tasks[i].end = 0;
    }
    /* simple static split into contiguous ranges of whole chunks */
    int64_t n_chunks = (n_rows + chunk - 1) / chunk;
    for (int i = 0; i < nthreads; ++i) {
        int64_t c0 = n_chunks * i / nthreads, c1 = n_chunks * (i + 1) / nthreads;
        tasks[i].begin = c0 * chunk;
        tasks[i].end = c1 * chunk < n_rows ? c1 * chunk : n_rows;
    }
    int *joined = (int *)calloc((size_t)nthreads, sizeof(int));
    if (!joined) {
        free(tasks);
        free(tids);
        return 2;
    }
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&tids[i], NULL, worker, &tasks[i]) == 0) {
            joined[i] = 1;
        } else {
            worker(&tasks[i]); /* run inline if a thread cannot start */
        }
    }
    worker(&tasks[0]);
    for (int i = 1; i < nthreads; ++i)
        if (joined[i]) pthread_join(tids[i], NULL);
    for (int i = 0; i < nthreads; ++i)
        if (tasks[i].failed) rc = 2;
    free(joined);
    free(tasks);
    free(tids);
    return rc;
}

static int check(const problem_t *p)
{
    if (p->B < 0 || p->Hq <= 0 || p->Hkv <= 0 || p->Sq < 0 || p->Sk < 0 || p->D <= 0) return 1;
    if (p->Hq % p->Hkv != 0) return 1;
    if (p->kv_capacity < p->Sk) return 1;
    if (!p->q || !p->k || !p->v) return 1;
    if (p->mask_planes > 0 && !p->mask) return 1;
    return 0;
}

/* Full forward.  out is [B,Hq,Sq,D] (out_layout 0) or [B,Sq,Hq*D] (1).
 * Returns 0 on success, 1 on a bad argument, 2 on an allocation failure. */
int oracle_attn_fwd(const float *q, const float *k, const float *v, const float *mask,
                    const int32_t *total_lengths, const int32_t *past_lengths, double *out,
                    int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk,
                    int64_t kv_capacity, int64_t D, int causal, int64_t local_window,
                    double scale, double softcap, int out_layout, int64_t mask_planes,
                    int nthreads)
{
    problem_t p = {q, k, v, mask, total_lengths, past_lengths, B, Hq, Hkv, Sq, Sk,
                   kv_capacity, D, causal, local_window, scale, softcap, mask_planes};
    if (check(&p) || !out || (out_layout != 0 && out_layout != 1)) return 1;
    return run_tasks(&p, NULL, B * Hq * Sq, out, NULL, out_layout, nthreads);
}

/* Full forward plus the per-row log-sum-exp of the scores, lse [B,Hq,Sq]. */
int oracle_attn_fwd_lse(const float *q, const float *k, const float *v, const float *mask,
                        const int32_t *total_lengths, const int32_t *past_lengths, double *out,
                        double *lse, int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk,
                        int64_t kv_capacity, int64_t D, int causal, int64_t local_window,
                        double scale, double softcap, int out_layout, int64_t mask_planes,
                        int nthreads)
{
    problem_t p = {q, k, v, mask, total_lengths, past_lengths, B, Hq, Hkv, Sq, Sk,
                   kv_capacity, D, causal, local_window, scale, softcap, mask_planes};
    if (check(&p) || !out || !lse || (out_layout != 0 && out_layout != 1)) return 1;
    return run_tasks(&p, NULL, B * Hq * Sq, out, lse, out_layout, nthreads);
}

/* Selected rows only: rows is [n_rows][3] of (b, h, qi); out_rows is
 * [n_rows][D].  Used to check full-size problems on a sample of rows. */
int oracle_attn_rows(const float *q, const float *k, const float *v, const float *mask,
                     const int32_t *total_lengths, const int32_t *past_lengths,
                     const int64_t *rows, int64_t n_rows, double *out_rows,
                     int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk,
                     int64_t kv_capacity, int64_t D, int causal, int64_t local_window,
                     double scale, double softcap, int64_t mask_planes, int nthreads)
{
    problem_t p = {q, k, v, mask, total_lengths, past_lengths, B, Hq, Hkv, Sq, Sk,
                   kv_capacity, D, causal, local_window, scale, softcap, mask_planes};
    if (check(&p) || !out_rows || (n_rows > 0 && !rows)) return 1;
    for (int64_t r = 0; r < n_rows; ++r) {
        if (rows[3 * r] < 0 || rows[3 * r] >= B || rows[3 * r + 1] < 0 ||
            rows[3 * r + 1] >= Hq || rows[3 * r + 2] < 0 || rows[3 * r + 2] >= Sq)
            return 1;
    }
    return run_tasks(&p, rows, n_rows, out_rows, NULL, 0, nthreads);
}

/* Number of worker threads a call with nthreads <= 0 uses. */
int oracle_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}
