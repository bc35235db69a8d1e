/*
 * attn_oracle.c -- slow, plain fp64 CPU reference for exact scaled-dot-product
 * attention and its gradient.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or helper
 * with the CUDA library.
 *
 * Sources (web pages, cited by title and section):
 *   [G3F]  "Gemini 3 Flash的注意力内核重写：算子融合如何实现亚毫秒级推理"
 *   [RED]  "提示词再优也救不了的性能黑洞：Transformer注意力计算冗余分析
 *           （含FlashAttention-3内核级优化验证数据）"
 *   [FA3P] "Flash Attention V3：大模型加速的核心网络算子优化实践"
 *
 * What is computed, per head (q, k, v, dO are N x d, row-major, fp64):
 *   forward  -- the standard three-step attention of [G3F] §传统注意力计算的
 *               内存带宽瓶颈 (S = scale*Q K^T, P = softmax(S), O = P V), with
 *               the max-subtracted softmax of [RED] §2.2 (stable_softmax) and
 *               the causal flag of [RED] 第一章 (key j visible to query i iff
 *               j <= i, square top-left alignment).  Per row i it also
 *               returns lse_i = m_i + ln(l_i): the row max and normaliser that
 *               [G3F] §4 重计算 says are the only statistics kept, folded into
 *               one natural-log number.
 *               Optional sliding window: [FA3P] §三.1 suggests a hybrid of
 *               local attention (LocalAttention(window_size=...)) and global
 *               attention without defining the window.  Reading used here:
 *               with window W >= 1, key j is visible to query i only if
 *               i - j < W (W keys ending at the diagonal under the causal
 *               flag) and, without the causal flag, also j - i < W; W = 0
 *               means no window.
 *   backward -- the analytic vector-Jacobian product of that forward for a
 *               loss with output gradient dO (textbook softmax VJP; [RED]
 *               §2.2 and §3.2 state parts of it):
 *                 D_i   = sum_c dO_ic o_ic
 *                 dP_ij = sum_c dO_ic v_jc
 *                 dS_ij = p_ij (dP_ij - D_i)
 *                 dQ_i  = scale sum_j dS_ij k_j
 *                 dK_j  = scale sum_i dS_ij q_i
 *                 dV_j  = sum_i p_ij dO_i
 *   online   -- a separate fp64 forward that walks the keys in column tiles
 *               with a running max and running sum, following the step list
 *               of [G3F] §3 在线softmax算法 (both the running sum and the
 *               partial output are rescaled when the max grows).  Used only
 *               to check that the one-pass form equals the three-step form.
 *
 * Every function evaluates the definition for a caller-chosen list of rows
 * (queries) or columns (keys); rows and columns are independent, so the list
 * is split over POSIX threads with no shared accumulator.  No N x N buffer is
 * ever formed: a row of scores is O(N) scratch.
 *
 * Return value: 0 on success, -1 on bad arguments, -2 on allocation failure.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

static int visible(int causal, int window, int i, int j) {
    if (causal && j > i) return 0;
    if (window > 0 && (i - j >= window || (!causal && j - i >= window))) return 0;
    return 1;
}

static double dot(const double* a, const double* b, int d) {
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += a[c] * b[c];
    return s;
}

/* Scores of row i: s_j = scale * q_i . k_j, -inf where masked.
 * Returns the row max m.  */
static double row_scores(const double* q, const double* k, int N, int d, int causal, int window,
                         double scale, int i, double* s) {
    double m = -INFINITY;
    for (int j = 0; j < N; ++j) {
        if (visible(causal, window, i, j)) {
            s[j] = scale * dot(q + (size_t)i * d, k + (size_t)j * d, d);
            if (s[j] > m) m = s[j];
        } else {
            s[j] = -INFINITY;
        }
    }
    return m;
}

/* Three-step forward for one row: probabilities p (length N), output o_i
 * (length d), and lse.  Returns lse. */
static double row_forward(const double* q, const double* k, const double* v, int N, int d,
                          int causal, int window, double scale, int i, double* p, double* o_row) {
    double m = row_scores(q, k, N, d, causal, window, scale, i, p);
    double l = 0.0;
    for (int j = 0; j < N; ++j) {
        p[j] = visible(causal, window, i, j) ? exp(p[j] - m) : 0.0;
        l += p[j];
    }
    for (int j = 0; j < N; ++j) p[j] /= l;
    for (int c = 0; c < d; ++c) o_row[c] = 0.0;
    for (int j = 0; j < N; ++j) {
        if (p[j] == 0.0) continue;
        const double* vj = v + (size_t)j * d;
        for (int c = 0; c < d; ++c) o_row[c] += p[j] * vj[c];
    }
    return m + log(l);
}

/* ------------------------------------------------------------------ threads */

typedef struct {
    int (*fn)(void* ctx, int item, double* scratch);
    void* ctx;
    int n_items;
    int next_start, stride;
    size_t scratch_len;
    int status;
} worker_t;

static void* worker_main(void* arg) {
    worker_t* w = (worker_t*)arg;
    double* scratch = (double*)malloc(sizeof(double) * (w->scratch_len ? w->scratch_len : 1));
    if (!scratch) { w->status = -2; return NULL; }
    for (int it = w->next_start; it < w->n_items; it += w->stride) {
        int rc = w->fn(w->ctx, it, scratch);
        if (rc) { w->status = rc; break; }
    }
    free(scratch);
    return NULL;
}

/* Run fn(ctx, item) for item in [0, n_items) on up to nthreads threads,
 * items dealt round-robin.  Each item writes only its own outputs.  A worker
 * whose thread cannot be started runs on the calling thread instead. */
static int parallel_for(int n_items, int nthreads, size_t scratch_len,
                        int (*fn)(void*, int, double*), void* ctx) {
    if (n_items <= 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n_items) nthreads = n_items;
    worker_t* ws = (worker_t*)calloc((size_t)nthreads, sizeof(worker_t));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    char* started = (char*)calloc((size_t)nthreads, 1);
    if (!ws || !th || !started) { free(ws); free(th); free(started); return -2; }
    for (int t = 0; t < nthreads; ++t) {
        ws[t].fn = fn; ws[t].ctx = ctx; ws[t].n_items = n_items;
        ws[t].next_start = t; ws[t].stride = nthreads;
        ws[t].scratch_len = scratch_len; ws[t].status = 0;
    }
    for (int t = 1; t < nthreads; ++t)
        started[t] = pthread_create(&th[t], NULL, worker_main, &ws[t]) == 0;
    worker_main(&ws[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (started[t]) pthread_join(th[t], NULL);
        else worker_main(&ws[t]);
    }
    int status = 0;
    for (int t = 0; t < nthreads; ++t) if (ws[t].status) status = ws[t].status;
    free(ws); free(th); free(started);
    return status;
}

int oracle_default_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* ------------------------------------------------------------------ forward */

typedef struct {
    const double *q, *k, *v;
    int N, d, causal, window;
    double scale;
    const int* rows;
    double *o, *lse;
} fwd_ctx_t;

static int fwd_item(void* c, int item, double* p) {
    fwd_ctx_t* x = (fwd_ctx_t*)c;
    int i = x->rows[item];
    x->lse[item] = row_forward(x->q, x->k, x->v, x->N, x->d, x->causal, x->window, x->scale, i, p,
                               x->o + (size_t)item * x->d);
    return 0;
}

/* Forward rows rows[0..nrows) of one head.  o_rows is nrows x d, lse_rows is
 * nrows; entry r belongs to query rows[r]. */
int oracle_head_fwd_rows(const double* q, const double* k, const double* v, int N, int d,
                         int causal, int window, double scale, const int* rows, int nrows,
                         double* o_rows, double* lse_rows, int nthreads) {
    if (!q || !k || !v || N < 1 || d < 1 || window < 0 || nrows < 0 ||
        (nrows && (!rows || !o_rows || !lse_rows)))
        return -1;
    for (int r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return -1;
    fwd_ctx_t x = {q, k, v, N, d, causal, window, scale, rows, o_rows, lse_rows};
    return parallel_for(nrows, nthreads, (size_t)N, fwd_item, &x);
}

/* ------------------------------------------------------------------ online */

/* One-pass forward of all rows of one head, keys visited in tiles of
 * tile_cols columns.  Single-threaded: it exists to be compared with the
 * three-step form on small inputs. */
int oracle_head_fwd_online(const double* q, const double* k, const double* v, int N, int d,
                           int causal, int window, double scale, int tile_cols, double* o, double* lse) {
    if (!q || !k || !v || !o || !lse || N < 1 || d < 1 || tile_cols < 1 || window < 0) return -1;
    double* s = (double*)malloc(sizeof(double) * (size_t)tile_cols);
    double* acc = (double*)malloc(sizeof(double) * (size_t)d);
    if (!s || !acc) { free(s); free(acc); return -2; }
    for (int i = 0; i < N; ++i) {
        double m = -INFINITY; /* running max m_i */
        double l = 0.0;       /* running sum l_i */
        for (int c = 0; c < d; ++c) acc[c] = 0.0;
        for (int j0 = 0; j0 < N; j0 += tile_cols) {
            int nt = (N - j0 < tile_cols) ? N - j0 : tile_cols;
            double m_local = -INFINITY;
            for (int t = 0; t < nt; ++t) {
                int j = j0 + t;
                s[t] = visible(causal, window, i, j)
                           ? scale * dot(q + (size_t)i * d, k + (size_t)j * d, d)
                           : -INFINITY;
                if (s[t] > m_local) m_local = s[t];
            }
            if (m_local == -INFINITY) continue; /* tile wholly masked: nothing to add */
            double m_new = m > m_local ? m : m_local;
            /* rescale the running sum and the partial output to the new max */
            double alpha = exp(m - m_new); /* exp(-inf) = 0 on the first tile */
            l *= alpha;
            for (int c = 0; c < d; ++c) acc[c] *= alpha;
            for (int t = 0; t < nt; ++t) {
                if (s[t] == -INFINITY) continue;
                double e = exp(s[t] - m_new);
                l += e;
                const double* vj = v + (size_t)(j0 + t) * d;
                for (int c = 0; c < d; ++c) acc[c] += e * vj[c];
            }
            m = m_new;
        }
        for (int c = 0; c < d; ++c) o[(size_t)i * d + c] = acc[c] / l;
        lse[i] = m + log(l);
    }
    free(s); free(acc);
    return 0;
}

/* ----------------------------------------------------------------- backward */

typedef struct {
    const double *q, *k, *v, *dO;
    int N, d, causal, window;
    double scale;
    const int* rows;
    double* lse_all; /* N: lse_i for every row (filled by stats pass) */
    double* D_all;   /* N: D_i = dO_i . o_i */
    double* dq;
    double *dk, *dv;
} bwd_ctx_t;

/* Row statistics lse_i and D_i for row i (scratch: N + d). */
static int stats_item(void* c, int i, double* scratch) {
    bwd_ctx_t* x = (bwd_ctx_t*)c;
    double* p = scratch;
    double* o_row = scratch + x->N;
    x->lse_all[i] = row_forward(x->q, x->k, x->v, x->N, x->d, x->causal, x->window, x->scale, i, p, o_row);
    x->D_all[i] = dot(x->dO + (size_t)i * x->d, o_row, x->d);
    return 0;
}

/* p_ij from the row statistic: exp(s_ij - lse_i) = exp(s_ij - m_i) / l_i. */
static double prob(const bwd_ctx_t* x, int i, int j) {
    if (!visible(x->causal, x->window, i, j)) return 0.0;
    double s = x->scale * dot(x->q + (size_t)i * x->d, x->k + (size_t)j * x->d, x->d);
    return exp(s - x->lse_all[i]);
}

/* dQ_i = scale * sum_j p_ij (dP_ij - D_i) k_j */
static int dq_item(void* c, int item, double* unused) {
    (void)unused;
    bwd_ctx_t* x = (bwd_ctx_t*)c;
    int i = x->rows[item], d = x->d;
    double* out = x->dq + (size_t)item * d;
    for (int cc = 0; cc < d; ++cc) out[cc] = 0.0;
    for (int j = 0; j < x->N; ++j) {
        double p = prob(x, i, j);
        if (p == 0.0) continue;
        double dP = dot(x->dO + (size_t)i * d, x->v + (size_t)j * d, d);
        double dS = p * (dP - x->D_all[i]);
        const double* kj = x->k + (size_t)j * d;
        for (int cc = 0; cc < d; ++cc) out[cc] += x->scale * dS * kj[cc];
    }
    return 0;
}

/* dK_j = scale * sum_i dS_ij q_i ;  dV_j = sum_i p_ij dO_i */
static int dkdv_item(void* c, int item, double* unused) {
    (void)unused;
    bwd_ctx_t* x = (bwd_ctx_t*)c;
    int j = x->rows[item], d = x->d;
    double* dk = x->dk + (size_t)item * d;
    double* dv = x->dv + (size_t)item * d;
    for (int cc = 0; cc < d; ++cc) { dk[cc] = 0.0; dv[cc] = 0.0; }
    for (int i = 0; i < x->N; ++i) {
        double p = prob(x, i, j);
        if (p == 0.0) continue;
        const double* dOi = x->dO + (size_t)i * d;
        double dP = dot(dOi, x->v + (size_t)j * d, d);
        double dS = p * (dP - x->D_all[i]);
        const double* qi = x->q + (size_t)i * d;
        for (int cc = 0; cc < d; ++cc) {
            dk[cc] += x->scale * dS * qi[cc];
            dv[cc] += p * dOi[cc];
        }
    }
    return 0;
}

typedef struct { bwd_ctx_t* x; const int* stat_rows; } stats_list_t;
static int stats_list_item(void* c, int item, double* scratch) {
    stats_list_t* s = (stats_list_t*)c;
    return stats_item(s->x, s->stat_rows[item], scratch);
}

/* Gradient of one head for the loss L = sum(dO * O).
 *   qrows[0..nq): rows of dQ to produce (dq_rows is nq x d)
 *   krows[0..nk): rows of dK and dV to produce (dk_rows, dv_rows are nk x d)
 * Row statistics lse_i and D_i are computed for exactly the rows that the
 * requested outputs depend on: the listed query rows when nk == 0, every row
 * otherwise (a key gradient sums over all queries).  lse_out and D_out, if
 * non-null, receive those statistics for all N rows (entries not computed
 * are left NaN). */
int oracle_head_bwd_rows(const double* q, const double* k, const double* v, const double* dO,
                         int N, int d, int causal, int window, double scale,
                         const int* qrows, int nq, const int* krows, int nk,
                         double* dq_rows, double* dk_rows, double* dv_rows,
                         double* lse_out, double* D_out, int nthreads) {
    if (!q || !k || !v || !dO || N < 1 || d < 1 || window < 0 || nq < 0 || nk < 0) return -1;
    if (nq && (!qrows || !dq_rows)) return -1;
    if (nk && (!krows || !dk_rows || !dv_rows)) return -1;
    for (int r = 0; r < nq; ++r) if (qrows[r] < 0 || qrows[r] >= N) return -1;
    for (int r = 0; r < nk; ++r) if (krows[r] < 0 || krows[r] >= N) return -1;

    double* lse_all = (double*)malloc(sizeof(double) * (size_t)N);
    double* D_all = (double*)malloc(sizeof(double) * (size_t)N);
    int* all_rows = NULL;
    if (!lse_all || !D_all) { free(lse_all); free(D_all); return -2; }
    for (int i = 0; i < N; ++i) { lse_all[i] = NAN; D_all[i] = NAN; }

    bwd_ctx_t x = {q, k, v, dO, N, d, causal, window, scale, NULL, lse_all, D_all, dq_rows, dk_rows, dv_rows};
    int rc;
    if (nk > 0) {
        all_rows = (int*)malloc(sizeof(int) * (size_t)N);
        if (!all_rows) { free(lse_all); free(D_all); return -2; }
        for (int i = 0; i < N; ++i) all_rows[i] = i;
        stats_list_t sl = {&x, all_rows};
        rc = parallel_for(N, nthreads, (size_t)N + (size_t)d, stats_list_item, &sl);
    } else {
        stats_list_t sl = {&x, qrows};
        rc = parallel_for(nq, nthreads, (size_t)N + (size_t)d, stats_list_item, &sl);
    }
    if (!rc && nq) { x.rows = qrows; rc = parallel_for(nq, nthreads, 1, dq_item, &x); }
    if (!rc && nk) { x.rows = krows; rc = parallel_for(nk, nthreads, 1, dkdv_item, &x); }
    if (!rc && lse_out) memcpy(lse_out, lse_all, sizeof(double) * (size_t)N);
    if (!rc && D_out) memcpy(D_out, D_all, sizeof(double) * (size_t)N);
    free(lse_all); free(D_all); free(all_rows);
    return rc;
}
