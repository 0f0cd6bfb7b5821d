/*
 * oracle.c -- plain, slow fp64 CPU oracle for diagonal-decay gated linear
 * attention (GLA).  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and
 * the CPU-baseline leg of the benchmark call it; the library never does.
 *
 * What it computes (per batch b and head h, all tensors row-major):
 *
 *   S_{-1} = S0                                   (S in R^{dk x dv})
 *   S_t    = diag(alpha_t) S_{t-1} + k_t^T v_t,   alpha_t = exp(log_alpha_t)
 *   o_t    = q_t S_t                              (token t itself included)
 *   S_final = S_{T-1}
 *
 * This is the token recurrence whose chunked, segmented evaluation the ZeCO
 * pages describe: the state is S in R^{dk x dv} and the decay is diagonal
 * ("diagonal-decay gated linear attention", ZeCO: Zero-Communication Overhead
 * Sequence Parallelism for Linear Attention, Limitations; Pith review of ZeCO,
 * "What carries the argument": the All-Scan update scales S by the cumulative
 * decay broadcast along d_v, so the decay acts on the d_k rows of S).  The
 * oracle knows nothing of segments (P), scan blocks (K) or chunks (C): the
 * chunked evaluation must reach the same numbers by regrouping (Pith review of
 * ZeCO, assumptions: Appendix A.1 decomposition).
 *
 * The backward is the brute-force adjoint of the loop above (not on the
 * pages).  With A the adjoint of S_t:
 *
 *   A = dS_final
 *   for t = T-1 .. 0:
 *       A      += q_t^T do_t
 *       dq_t    = do_t S_t^T
 *       dk_t    = A v_t^T
 *       dv_t    = k_t A
 *       dg_t[i] = alpha_t[i] * sum_j A[i,j] S_{t-1}[i,j]
 *       A       = diag(alpha_t) A
 *   dS0 = A
 *
 * Because the decay is diagonal, every element S[i,j] (and A[i,j]) follows a
 * scalar recurrence of its own.  The loops below use that: o[:,j] and dv[:,j]
 * need column j of S or A only, and dq[:,i], dk[:,i], dg[:,i] need row i only.
 * Column and row work is split across threads; within one row or column the
 * arithmetic is exactly the loop above.  The same split lets a caller ask for
 * a subset of columns or rows, which is how outputs of full-size workloads are
 * sampled.  The backward stores row states every CKPT tokens and recomputes
 * them forward inside each block: no division by alpha anywhere.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define CKPT 1024

typedef struct {
    int64_t B, H, T, dk, dv;
} oshape;

/* ---------------------------------------------------------------- threads */

typedef void (*work_fn)(void *ctx, int64_t item, double *scratch);

typedef struct {
    work_fn fn;
    void *ctx;
    int64_t n_items;
    int64_t next;
    pthread_mutex_t mu;
    size_t scratch_doubles;
    int failed;
} pool_t;

static void *pool_main(void *arg) {
    pool_t *p = (pool_t *)arg;
    double *scratch = NULL;
    if (p->scratch_doubles) {
        scratch = (double *)malloc(p->scratch_doubles * sizeof(double));
        if (!scratch) {
            pthread_mutex_lock(&p->mu);
            p->failed = 1;
            pthread_mutex_unlock(&p->mu);
            return NULL;
        }
    }
    for (;;) {
        pthread_mutex_lock(&p->mu);
        int64_t it = p->next++;
        pthread_mutex_unlock(&p->mu);
        if (it >= p->n_items) break;
        p->fn(p->ctx, it, scratch);
    }
    free(scratch);
    return NULL;
}

static int run_pool(work_fn fn, void *ctx, int64_t n_items, int nthreads, size_t scratch_doubles) {
    pool_t p;
    p.fn = fn;
    p.ctx = ctx;
    p.n_items = n_items;
    p.next = 0;
    p.scratch_doubles = scratch_doubles;
    p.failed = 0;
    pthread_mutex_init(&p.mu, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    if (nthreads > n_items) nthreads = n_items > 0 ? (int)n_items : 1;
    pthread_t th[1024];
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, pool_main, &p) != 0) break;
        ++started;
    }
    if (started == 0) pool_main(&p);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    pthread_mutex_destroy(&p.mu);
    return p.failed ? -1 : 0;
}

/* ---------------------------------------------------------------- forward */

typedef struct {
    oshape s;
    const double *q, *k, *v, *g, *S0;
    double *o_cols;      /* [B][H][T][ncols] */
    double *Sfin_cols;   /* [B][H][dk][ncols], may be NULL */
    int64_t ncols;
    const int64_t *cols; /* NULL: column c is column c */
} fwd_ctx;

/* one work item = one (b,h) and one output column j of S */
static void fwd_item(void *vctx, int64_t item, double *Scol) {
    fwd_ctx *c = (fwd_ctx *)vctx;
    const int64_t T = c->s.T, dk = c->s.dk, dv = c->s.dv, nc = c->ncols;
    const int64_t bh = item / nc, ci = item % nc;
    const int64_t j = c->cols ? c->cols[ci] : ci;
    const double *q = c->q + bh * T * dk, *k = c->k + bh * T * dk, *g = c->g + bh * T * dk;
    const double *v = c->v + bh * T * dv;
    for (int64_t i = 0; i < dk; ++i) Scol[i] = c->S0 ? c->S0[bh * dk * dv + i * dv + j] : 0.0;
    for (int64_t t = 0; t < T; ++t) {
        double acc = 0.0;
        const double vtj = v[t * dv + j];
        for (int64_t i = 0; i < dk; ++i) {
            /* S_t[i,j] = alpha_t[i] S_{t-1}[i,j] + k_t[i] v_t[j] */
            Scol[i] = exp(g[t * dk + i]) * Scol[i] + k[t * dk + i] * vtj;
            /* o_t[j] = sum_i q_t[i] S_t[i,j] */
            acc += q[t * dk + i] * Scol[i];
        }
        c->o_cols[(bh * T + t) * nc + ci] = acc;
    }
    if (c->Sfin_cols)
        for (int64_t i = 0; i < dk; ++i) c->Sfin_cols[(bh * dk + i) * nc + ci] = Scol[i];
}

/*
 * Forward.  q,k,g: [B][H][T][dk]; v: [B][H][T][dv]; S0: [B][H][dk][dv] or NULL
 * (zeros).  Output columns: cols[0..ncols) (cols == NULL means all dv columns
 * in order, ncols must then equal dv).  o_cols: [B][H][T][ncols],
 * Sfin_cols: [B][H][dk][ncols] or NULL.  Returns 0 on success.
 */
int oracle_gla_fwd(int64_t B, int64_t H, int64_t T, int64_t dk, int64_t dv, const double *q,
                   const double *k, const double *v, const double *g, const double *S0,
                   int64_t ncols, const int64_t *cols, double *o_cols, double *Sfin_cols,
                   int nthreads) {
    if (B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1 || ncols < 0) return -1;
    if (!cols && ncols != dv) return -1;
    for (int64_t c = 0; cols && c < ncols; ++c)
        if (cols[c] < 0 || cols[c] >= dv) return -1;
    fwd_ctx c = {{B, H, T, dk, dv}, q, k, v, g, S0, o_cols, Sfin_cols, ncols, cols};
    return run_pool(fwd_item, &c, B * H * ncols, nthreads, (size_t)dk);
}

/* --------------------------------------------------------------- backward */

typedef struct {
    oshape s;
    const double *q, *k, *v, *g, *S0, *dO, *dSf;
    int64_t nrows, ncols;
    const int64_t *rows, *cols;
    double *dq_rows, *dk_rows, *dg_rows; /* [B][H][T][nrows] */
    double *dS0_rows;                    /* [B][H][nrows][dv] or NULL */
    double *dv_cols;                     /* [B][H][T][ncols] */
} bwd_ctx;

/*
 * Row work item: one (b,h) and one row i.  Produces dq[:,i], dk[:,i], dg[:,i]
 * and row i of dS0.  Scratch layout: ckpt [(T/CKPT+1) * dv] | blk [(CKPT+1) * dv]
 * | A [dv].  blk holds S_{t0-1}, S_{t0}, ..., S_{t1-1} of the current block.
 */
static void bwd_row_item(void *vctx, int64_t item, double *scr) {
    bwd_ctx *c = (bwd_ctx *)vctx;
    const int64_t T = c->s.T, dk = c->s.dk, dv = c->s.dv, nr = c->nrows;
    const int64_t bh = item / nr, ri = item % nr;
    const int64_t i = c->rows ? c->rows[ri] : ri;
    const double *q = c->q + bh * T * dk, *k = c->k + bh * T * dk, *g = c->g + bh * T * dk;
    const double *v = c->v + bh * T * dv, *dO = c->dO + bh * T * dv;
    const int64_t nblk = (T + CKPT - 1) / CKPT;
    double *ckpt = scr;
    double *blk = ckpt + (nblk + 1) * dv;
    double *A = blk + (CKPT + 1) * dv;

    /* forward over row i, storing S_{t0-1} at each block start t0 */
    double *S = A; /* reuse as the running row before A is needed */
    for (int64_t j = 0; j < dv; ++j) S[j] = c->S0 ? c->S0[bh * dk * dv + i * dv + j] : 0.0;
    for (int64_t b = 0; b < nblk; ++b) {
        memcpy(ckpt + b * dv, S, dv * sizeof(double));
        const int64_t t0 = b * CKPT, t1 = t0 + CKPT < T ? t0 + CKPT : T;
        for (int64_t t = t0; t < t1; ++t) {
            const double a = exp(g[t * dk + i]);
            for (int64_t j = 0; j < dv; ++j) S[j] = a * S[j] + k[t * dk + i] * v[t * dv + j];
        }
    }
    /* reverse */
    for (int64_t j = 0; j < dv; ++j) A[j] = c->dSf ? c->dSf[bh * dk * dv + i * dv + j] : 0.0;
    for (int64_t b = nblk - 1; b >= 0; --b) {
        const int64_t t0 = b * CKPT, t1 = t0 + CKPT < T ? t0 + CKPT : T;
        /* blk[(t - t0 + 1) * dv + j] = S_t[i,j];  blk[0..dv) = S_{t0-1} */
        memcpy(blk, ckpt + b * dv, dv * sizeof(double));
        for (int64_t t = t0; t < t1; ++t) {
            const double a = exp(g[t * dk + i]);
            const double *Sp = blk + (t - t0) * dv;
            double *Sn = blk + (t - t0 + 1) * dv;
            for (int64_t j = 0; j < dv; ++j) Sn[j] = a * Sp[j] + k[t * dk + i] * v[t * dv + j];
        }
        for (int64_t t = t1 - 1; t >= t0; --t) {
            const double a = exp(g[t * dk + i]);
            const double *Sp = blk + (t - t0) * dv;     /* S_{t-1} */
            const double *St = blk + (t - t0 + 1) * dv; /* S_t */
            double sdq = 0.0, sdk = 0.0, sdg = 0.0;
            for (int64_t j = 0; j < dv; ++j) {
                A[j] += q[t * dk + i] * dO[t * dv + j]; /* A += q_t^T do_t */
                sdq += dO[t * dv + j] * St[j];          /* dq_t = do_t S_t^T */
                sdk += A[j] * v[t * dv + j];            /* dk_t = A v_t^T */
                sdg += A[j] * Sp[j];                    /* dg_t = alpha_t sum_j A S_{t-1} */
            }
            c->dq_rows[(bh * T + t) * nr + ri] = sdq;
            c->dk_rows[(bh * T + t) * nr + ri] = sdk;
            c->dg_rows[(bh * T + t) * nr + ri] = a * sdg;
            for (int64_t j = 0; j < dv; ++j) A[j] *= a; /* A = diag(alpha_t) A */
        }
    }
    if (c->dS0_rows)
        for (int64_t j = 0; j < dv; ++j) c->dS0_rows[(bh * nr + ri) * dv + j] = A[j];
}

/* Column work item: one (b,h) and one column j.  Produces dv[:,j]. */
static void bwd_col_item(void *vctx, int64_t item, double *A) {
    bwd_ctx *c = (bwd_ctx *)vctx;
    const int64_t T = c->s.T, dk = c->s.dk, dv = c->s.dv, nc = c->ncols;
    const int64_t bh = item / nc, ci = item % nc;
    const int64_t j = c->cols ? c->cols[ci] : ci;
    const double *q = c->q + bh * T * dk, *k = c->k + bh * T * dk, *g = c->g + bh * T * dk;
    const double *dO = c->dO + bh * T * dv;
    for (int64_t i = 0; i < dk; ++i) A[i] = c->dSf ? c->dSf[bh * dk * dv + i * dv + j] : 0.0;
    for (int64_t t = T - 1; t >= 0; --t) {
        double sdv = 0.0;
        for (int64_t i = 0; i < dk; ++i) {
            A[i] += q[t * dk + i] * dO[t * dv + j]; /* A += q_t^T do_t */
            sdv += k[t * dk + i] * A[i];            /* dv_t = k_t A */
        }
        c->dv_cols[(bh * T + t) * nc + ci] = sdv;
        for (int64_t i = 0; i < dk; ++i) A[i] *= exp(g[t * dk + i]); /* A = diag(alpha_t) A */
    }
}

/*
 * Backward.  Inputs as for the forward plus dO [B][H][T][dv] and dS_final
 * [B][H][dk][dv] (NULL: zeros).  Row outputs for rows[0..nrows) (rows == NULL:
 * all dk rows, nrows must equal dk): dq_rows, dk_rows, dg_rows [B][H][T][nrows],
 * dS0_rows [B][H][nrows][dv] (may be NULL).  Column outputs for
 * cols[0..ncols) (cols == NULL: all, ncols must equal dv): dv_cols
 * [B][H][T][ncols].  nrows or ncols may be 0 to skip that half.
 */
int oracle_gla_bwd(int64_t B, int64_t H, int64_t T, int64_t dk, int64_t dv, const double *q,
                   const double *k, const double *v, const double *g, const double *S0,
                   const double *dO, const double *dS_final, int64_t nrows, const int64_t *rows,
                   double *dq_rows, double *dk_rows, double *dg_rows, double *dS0_rows,
                   int64_t ncols, const int64_t *cols, double *dv_cols, int nthreads) {
    if (B < 1 || H < 1 || T < 0 || dk < 1 || dv < 1 || nrows < 0 || ncols < 0) return -1;
    if (!rows && nrows != 0 && nrows != dk) return -1;
    if (!cols && ncols != 0 && ncols != dv) return -1;
    for (int64_t r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= dk) return -1;
    for (int64_t c = 0; cols && c < ncols; ++c)
        if (cols[c] < 0 || cols[c] >= dv) return -1;
    bwd_ctx c = {{B, H, T, dk, dv}, q, k, v, g, S0, dO, dS_final, nrows, ncols, rows, cols,
                 dq_rows, dk_rows, dg_rows, dS0_rows, dv_cols};
    const int64_t nblk = (T + CKPT - 1) / CKPT;
    int rc = 0;
    if (nrows > 0)
        rc |= run_pool(bwd_row_item, &c, B * H * nrows, nthreads,
                       (size_t)((nblk + 1) * dv + (CKPT + 1) * dv + dv));
    if (ncols > 0) rc |= run_pool(bwd_col_item, &c, B * H * ncols, nthreads, (size_t)dk);
    return rc;
}
