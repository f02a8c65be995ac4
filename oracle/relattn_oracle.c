/*
 * Plain, slow, obviously-correct fp64 CPU oracle for relation-aware self-attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call this
 * file: only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
 * leg use it. It shares no code, header or table with the CUDA library.
 *
 * What it computes (one query row at a time, fp64, no blocking and no fusion):
 *
 *   Shaw, Uszkoreit & Vaswani, "Self-Attention with Relative Position Representations"
 *   (paper summary page, section "Relation-Aware Self-Attention: The Core Modification",
 *   eq. 4 for the compatibility and eq. 3 for the output; section "Relative Position
 *   Representations: From Arbitrary Edges to Sequences" for clip(j - i, k) and the
 *   table order w_{-k} .. w_{k}):
 *
 *     e_ij   = scale * q_i . (k_j + a^K_ij),     a^K_ij = w^K[clip(j - i, k) + k]
 *     alpha  = softmax over the allowed j of e_ij
 *     z_i    = sum_j alpha_ij (v_j + a^V_ij),    a^V_ij = w^V[clip(j - i, k) + k]
 *
 *   The softmax is evaluated as exp(e_ij - m) / sum_j exp(e_ij - m) with m the row
 *   maximum; this is the same number as exp(e_ij) / sum exp(e_ik) (the factor exp(-m)
 *   cancels) and only keeps exp() finite.
 *
 *   Arbitrary labelled edges (the same page, section "Relation-Aware Self-Attention:
 *   The Core Modification": the input is a graph whose edge (i, j) carries a_ij; section
 *   3.4 then specialises the label to clip(j - i, k) + k): the same two equations with
 *   a^K_ij = w^K[L[b][i][j]], a^V_ij = w^V[L[b][i][j]] for a given label matrix L.
 *
 *   T5 scalar bias ("Relative position embeddings" page, section "T5"):
 *     e_ij = scale * q_i . k_j + b[bucket(j - i), h]
 *   The bucket of each offset is computed exactly by oracle/t5.py and handed in as a
 *   table indexed by (j - i) + (n - 1).
 *
 * Allowed keys for row i of sequence b: j < kv_len[b] (all j when kv_len is NULL) and,
 * when causal, j <= i. A row with no allowed key outputs zeros.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    /* shared inputs */
    const double *q, *k, *v;          /* [B, H, n, d] */
    const double *aK, *aV;            /* Shaw: [*, 2k+1, d] with head stride ths, or NULL */
    long long ths;                    /* table head stride, in elements (0 = shared) */
    int clip_k;
    const unsigned char *labels;      /* labelled edges: [*, n, n] or NULL (clip labels) */
    long long label_bstride;          /* elements between batches' label matrices (0 = shared) */
    const double *bias;               /* T5: [num_buckets, H] */
    const int *bucket_of_offset;      /* T5: [2n - 1], index (j - i) + (n - 1) */
    int causal;
    double scale;
    const int *kv_len;                /* [B] or NULL */
    int B, H, n, d;
    const long long *rows;            /* flat (b*H + h)*n + i row ids, or NULL for all */
    long long nrows;
    double *out;                      /* [nrows, d] (or [B,H,n,d] when rows == NULL) */
    int t5;
    /* per-thread partition */
    long long r0, r1;
} job_t;

static long long clip_ll(long long x, long long k) {
    if (x < -k) return -k;
    if (x > k) return k;
    return x;
}

/* table row of edge (i, j) of sequence b: the given label, else clip(j - i, k) + k */
static long long edge_label(const job_t *J, long long b, long long i, long long j) {
    if (J->labels)
        return (long long)J->labels[b * J->label_bstride + i * (long long)J->n + j];
    return clip_ll(j - i, J->clip_k) + J->clip_k;
}

static void one_row(const job_t *J, long long row, double *out_row, double *e, char *ok) {
    const int n = J->n, d = J->d, H = J->H;
    const long long bh = row / n;
    const long long i = row % n;
    const long long b = bh / H;
    const long long h = bh % H;
    const double *qi = J->q + row * d;
    long long valid = n;
    if (J->kv_len) {
        valid = J->kv_len[b];
        if (valid > n) valid = n;
        if (valid < 0) valid = 0;
    }
    double m = -INFINITY;
    int any = 0;
    for (long long j = 0; j < n; ++j) {
        ok[j] = (char)(j < valid && (!J->causal || j <= i));
        if (!ok[j]) continue;
        const double *kj = J->k + (bh * n + j) * d;
        double s = 0.0;
        if (J->t5) {
            for (int c = 0; c < d; ++c) s += qi[c] * kj[c];
            const int bucket = J->bucket_of_offset[(j - i) + (n - 1)];
            e[j] = J->scale * s + J->bias[(long long)bucket * H + h];
        } else {
            const long long r = edge_label(J, b, i, j);
            const double *ak = J->aK ? J->aK + h * J->ths + r * d : NULL;
            for (int c = 0; c < d; ++c) s += qi[c] * (kj[c] + (ak ? ak[c] : 0.0));
            e[j] = J->scale * s;
        }
        if (e[j] > m) m = e[j];
        any = 1;
    }
    for (int c = 0; c < d; ++c) out_row[c] = 0.0;
    if (!any) return;
    double l = 0.0;
    for (long long j = 0; j < n; ++j)
        if (ok[j]) l += exp(e[j] - m);
    for (long long j = 0; j < n; ++j) {
        if (!ok[j]) continue;
        const double alpha = exp(e[j] - m) / l;
        const double *vj = J->v + (bh * n + j) * d;
        const double *av = NULL;
        if (!J->t5 && J->aV) {
            const long long r = edge_label(J, b, i, j);
            av = J->aV + h * J->ths + r * d;
        }
        for (int c = 0; c < d; ++c) out_row[c] += alpha * (vj[c] + (av ? av[c] : 0.0));
    }
}

static void *worker(void *arg) {
    const job_t *J = (const job_t *)arg;
    double *e = (double *)malloc(sizeof(double) * (size_t)J->n);
    char *ok = (char *)malloc((size_t)J->n);
    for (long long t = J->r0; t < J->r1; ++t) {
        const long long row = J->rows ? J->rows[t] : t;
        one_row(J, row, J->out + t * J->d, e, ok);
    }
    free(e);
    free(ok);
    return NULL;
}

static int run(job_t *base, int nthreads) {
    const long long total = base->rows ? base->nrows : (long long)base->B * base->H * base->n;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (total < nthreads) nthreads = total > 0 ? (int)total : 1;
    pthread_t tid[256];
    job_t jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *base;
        jobs[t].r0 = total * t / nthreads;
        jobs[t].r1 = total * (t + 1) / nthreads;
    }
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&tid[t], NULL, worker, &jobs[t]) != 0) return -1;
    worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) pthread_join(tid[t], NULL);
    return 0;
}

/* Shaw relation-aware attention. aK / aV may be NULL (term absent). */
int oracle_relattn_rows(const double *q, const double *k, const double *v,
                        const double *aK, const double *aV, long long table_head_stride,
                        int clip_k, int causal, double scale, const int *kv_len,
                        int B, int H, int n, int d,
                        const long long *rows, long long nrows, double *out, int nthreads) {
    job_t J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.aK = aK; J.aV = aV; J.ths = table_head_stride;
    J.clip_k = clip_k; J.causal = causal; J.scale = scale; J.kv_len = kv_len;
    J.B = B; J.H = H; J.n = n; J.d = d; J.rows = rows; J.nrows = nrows; J.out = out;
    J.t5 = 0;
    return run(&J, nthreads);
}

/* Labelled edges: table rows from labels[b * label_bstride + i * n + j] (values below the
 * tables' row count; the caller checks). aK / aV may be NULL. */
int oracle_labeled_rows(const double *q, const double *k, const double *v,
                        const double *aK, const double *aV, long long table_head_stride,
                        const unsigned char *labels, long long label_bstride, int causal,
                        double scale, const int *kv_len, int B, int H, int n, int d,
                        const long long *rows, long long nrows, double *out, int nthreads) {
    job_t J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.aK = aK; J.aV = aV; J.ths = table_head_stride;
    J.labels = labels; J.label_bstride = label_bstride;
    J.causal = causal; J.scale = scale; J.kv_len = kv_len;
    J.B = B; J.H = H; J.n = n; J.d = d; J.rows = rows; J.nrows = nrows; J.out = out;
    J.t5 = 0;
    return run(&J, nthreads);
}

/* T5 scalar bucketed bias. bucket_of_offset has 2n-1 entries, index (j - i) + n - 1. */
int oracle_t5bias_rows(const double *q, const double *k, const double *v,
                       const double *bias, const int *bucket_of_offset,
                       int causal, double scale, const int *kv_len,
                       int B, int H, int n, int d,
                       const long long *rows, long long nrows, double *out, int nthreads) {
    job_t J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.bias = bias; J.bucket_of_offset = bucket_of_offset;
    J.causal = causal; J.scale = scale; J.kv_len = kv_len;
    J.B = B; J.H = H; J.n = n; J.d = d; J.rows = rows; J.nrows = nrows; J.out = out;
    J.t5 = 1;
    return run(&J, nthreads);
}
