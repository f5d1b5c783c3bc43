/*
 * attn_oracle.c -- plain fp64 CPU attention: the oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load, call or link this code.  The
 * product path (the CUDA library and its Python binding) never touches it,
 * and this file shares no code, header or constant with that path.
 *
 * What it computes is the plain definition of scaled-dot-product attention
 * for ONE head, written out in double precision, with the score row and the
 * probability row materialised (no tiling, no online softmax):
 *
 *   s_rl = c * q_r . k_l            for allowed (r, l), else -inf
 *   p_rl = exp(s_rl - max_l s_rl) / sum_l exp(s_rl - max_l s_rl)
 *   o_r  = sum_l p_rl v_l
 *   lse_r = max_l s_rl + log sum_l exp(s_rl - max_l s_rl)
 *
 * Sources: "FlashAttention -- IO-Aware Exact Attention" (atlas wiki),
 * section "Standard attention, and why it's wasteful" (S = QK^T, P =
 * softmax(S), O = PV); zerotofrontier "FlashAttention" (Efficient attention
 * 12.3), sections "The forward pass" (S_ij = Q_i K_j^T / sqrt(d_k), lse =
 * m + log l, natural logarithm) and "What the forward pass leaves behind"
 * (one log-sum-exp per query row).
 *
 * The backward pass is the exact analytic gradient of O = softmax(c Q K^T) V
 * (zerotofrontier "FlashAttention", section "The backward pass, derived"):
 *
 *   dV = P^T dO,  dP = dO V^T,  D_r = sum_l P_rl dP_rl,
 *   dS = P o (dP - D),  dQ = c dS K,  dK = c dS^T Q.
 *
 * D_r is taken from its definition (the softmax Jacobian's row term); the
 * page's identity D_r = dO_r . O_r is checked against it by the tests, not
 * used here.  The factor c on dQ and dK comes from S = c Q K^T.
 *
 * Masks (zerotofrontier "FlashAttention", "The causal mask, and the tiles
 * you never visit"; "Dropout, block-sparsity, and other real-kernel
 * details": sliding windows are functions of (r, l), and a block mask skips
 * whole tiles): key l is allowed for query r iff
 *    l >= r + (Tk - Tq) - left    (when left >= 0; -1: no lower bound)
 *    l <= r + (Tk - Tq) + right   (when right >= 0; -1: no upper bound)
 *    block[r / bs][l / bs] != 0   (when a block mask is given)
 * Causal is left = -1, right = 0.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - causal masks are aligned bottom-right: key l is allowed for query r iff
 *    l <= r + (Tk - Tq); this is the pages' "query r sees keys l <= r" when
 *    Tq == Tk.  Windows are measured from the same diagonal key.
 *  - a row with no allowed key has O = 0, lse = -inf and zero gradients.
 *
 * Layout: q, o, dO, dq are [Tq][d]; k, v, dk, dv are [Tk][d]; row-major fp64.
 * Threads: rows (and sampled keys) are dealt round-robin to nthreads
 * pthreads; each thread owns its scratch rows.  The arithmetic of one row
 * does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t left, right;     /* window around the diagonal key r + Tk - Tq; -1 = unbounded */
    const uint8_t *block;    /* NULL, or [ceil(Tq / bs)][ceil(Tk / bs)], nonzero = allowed */
    int64_t bs;              /* block size of the block mask (rows and keys) */
} mask_t;

static int is_allowed(int64_t r, int64_t l, int64_t Tq, int64_t Tk, const mask_t *m)
{
    const int64_t diag = r + (Tk - Tq);
    if (m->right >= 0 && l > diag + m->right)
        return 0;
    if (m->left >= 0 && l < diag - m->left)
        return 0;
    if (m->block && !m->block[(r / m->bs) * ((Tk + m->bs - 1) / m->bs) + l / m->bs])
        return 0;
    return 1;
}

static mask_t causal_mask(int causal)
{
    mask_t m = {-1, causal ? 0 : -1, NULL, 1};
    return m;
}

static double dot(const double *a, const double *b, int64_t d)
{
    double acc = 0.0;
    for (int64_t c = 0; c < d; ++c)
        acc += a[c] * b[c];
    return acc;
}

/* ------------------------------------------------------------------ */
/* Forward: one query row, materialising its score and weight rows.    */
/* ------------------------------------------------------------------ */
typedef struct {
    const double *q, *k, *v;
    int64_t Tq, Tk, d;
    mask_t mask;
    double scale;
    const int64_t *rows;   /* which query rows to evaluate */
    int64_t nrows;
    double *o;             /* [nrows][d] */
    double *lse;           /* [nrows] */
    int nthreads, tid;
    int status;
} fwd_task;

static void forward_row(const fwd_task *T, int64_t r, double *p, double *o_r, double *lse_r)
{
    const int64_t d = T->d;
    const double *q_r = T->q + r * d;
    double m = -INFINITY;
    /* scores s_rl, masked entries are -inf */
    for (int64_t l = 0; l < T->Tk; ++l) {
        if (is_allowed(r, l, T->Tq, T->Tk, &T->mask)) {
            p[l] = T->scale * dot(q_r, T->k + l * d, d);
            if (p[l] > m)
                m = p[l];
        } else {
            p[l] = -INFINITY;
        }
    }
    for (int64_t c = 0; c < d; ++c)
        o_r[c] = 0.0;
    if (m == -INFINITY) {          /* no allowed key: empty softmax */
        *lse_r = -INFINITY;
        return;
    }
    /* weights p_rl = exp(s_rl - m) / l */
    double ell = 0.0;
    for (int64_t l = 0; l < T->Tk; ++l) {
        p[l] = (p[l] == -INFINITY) ? 0.0 : exp(p[l] - m);
        ell += p[l];
    }
    for (int64_t l = 0; l < T->Tk; ++l) {
        const double w = p[l] / ell;
        if (w == 0.0)
            continue;
        const double *v_l = T->v + l * d;
        for (int64_t c = 0; c < d; ++c)
            o_r[c] += w * v_l[c];
    }
    *lse_r = m + log(ell);
}

static void *fwd_worker(void *arg)
{
    fwd_task *T = (fwd_task *)arg;
    double *p = (double *)malloc(sizeof(double) * (size_t)(T->Tk > 0 ? T->Tk : 1));
    if (!p) {
        T->status = 1;
        return NULL;
    }
    for (int64_t i = T->tid; i < T->nrows; i += T->nthreads)
        forward_row(T, T->rows[i], p, T->o + i * T->d, T->lse + i);
    free(p);
    return NULL;
}

/*
 * oracle_fwd: O and lse for the listed query rows of one head.
 * Returns 0 on success, nonzero on a bad argument or allocation failure.
 */
static int fwd_run(const double *q, const double *k, const double *v,
                   int64_t Tq, int64_t Tk, int64_t d, mask_t mask, double scale,
                   const int64_t *rows, int64_t nrows,
                   double *o, double *lse, int nthreads)
{
    if (Tq < 0 || Tk < 0 || d < 1 || nrows < 0 || nthreads < 1)
        return 2;
    for (int64_t i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= Tq)
            return 2;
    fwd_task *tasks = (fwd_task *)calloc((size_t)nthreads, sizeof(fwd_task));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!tasks || !th) {
        free(tasks);
        free(th);
        return 1;
    }
    for (int t = 0; t < nthreads; ++t) {
        fwd_task x = {q, k, v, Tq, Tk, d, mask, scale, rows, nrows, o, lse, nthreads, t, 0};
        tasks[t] = x;
        pthread_create(&th[t], NULL, fwd_worker, &tasks[t]);
    }
    int status = 0;
    for (int t = 0; t < nthreads; ++t) {
        pthread_join(th[t], NULL);
        status |= tasks[t].status;
    }
    free(tasks);
    free(th);
    return status;
}

int oracle_fwd(const double *q, const double *k, const double *v,
               int64_t Tq, int64_t Tk, int64_t d, int causal, double scale,
               const int64_t *rows, int64_t nrows,
               double *o, double *lse, int nthreads)
{
    return fwd_run(q, k, v, Tq, Tk, d, causal_mask(causal), scale, rows, nrows, o, lse, nthreads);
}

/*
 * oracle_fwd_masked: oracle_fwd under the window (left, right) and block
 * mask (block, bs) described above (block may be NULL).
 */
int oracle_fwd_masked(const double *q, const double *k, const double *v,
                      int64_t Tq, int64_t Tk, int64_t d, int64_t left, int64_t right,
                      const uint8_t *block, int64_t bs, double scale,
                      const int64_t *rows, int64_t nrows,
                      double *o, double *lse, int nthreads)
{
    if (left < -1 || right < -1 || (block && bs < 1))
        return 2;
    mask_t m = {left, right, block, block ? bs : 1};
    return fwd_run(q, k, v, Tq, Tk, d, m, scale, rows, nrows, o, lse, nthreads);
}

/* ------------------------------------------------------------------ */
/* Backward.                                                            */
/*  pass 1 (every query row r): s_r, P_r, dP_r = dO_r V^T, D_r,         */
/*          lse_r, optionally O_r, and dQ_r for the sampled rows.       */
/*  pass 2 (sampled keys l):    dV_l = sum_r P_rl dO_r,                 */
/*          dK_l = c sum_r dS_rl q_r, with P_rl rebuilt as               */
/*          exp(s_rl - lse_r) from the row statistics of pass 1.        */
/* With every row and every key sampled this is the full gradient.      */
/* ------------------------------------------------------------------ */
typedef struct {
    const double *q, *k, *v, *dO;
    int64_t Tq, Tk, d;
    mask_t mask;
    double scale;
    const int64_t *row_slot;  /* [Tq]: index into dq, or -1 */
    const int64_t *keys;
    int64_t nkeys;
    double *dq, *dk, *dv;
    double *o_all, *lse_all, *D_all;
    int nthreads, tid;
    int status;
} bwd_task;

static void *bwd_rows_worker(void *arg)
{
    bwd_task *T = (bwd_task *)arg;
    const int64_t d = T->d, Tk = T->Tk;
    double *p = (double *)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
    double *dp = (double *)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
    if (!p || !dp) {
        free(p);
        free(dp);
        T->status = 1;
        return NULL;
    }
    for (int64_t r = T->tid; r < T->Tq; r += T->nthreads) {
        const double *q_r = T->q + r * d;
        const double *do_r = T->dO + r * d;
        double m = -INFINITY;
        for (int64_t l = 0; l < Tk; ++l) {
            if (is_allowed(r, l, T->Tq, Tk, &T->mask)) {
                p[l] = T->scale * dot(q_r, T->k + l * d, d);
                if (p[l] > m)
                    m = p[l];
            } else {
                p[l] = -INFINITY;
            }
        }
        const int64_t slot = T->row_slot[r];
        if (m == -INFINITY) {      /* fully masked row: no gradient flows */
            T->lse_all[r] = -INFINITY;
            T->D_all[r] = 0.0;
            if (T->o_all)
                for (int64_t c = 0; c < d; ++c)
                    T->o_all[r * d + c] = 0.0;
            if (slot >= 0)
                for (int64_t c = 0; c < d; ++c)
                    T->dq[slot * d + c] = 0.0;
            continue;
        }
        double ell = 0.0;
        for (int64_t l = 0; l < Tk; ++l) {
            p[l] = (p[l] == -INFINITY) ? 0.0 : exp(p[l] - m);
            ell += p[l];
        }
        for (int64_t l = 0; l < Tk; ++l)
            p[l] /= ell;                        /* P_rl */
        double D = 0.0;
        for (int64_t l = 0; l < Tk; ++l) {
            dp[l] = (p[l] == 0.0) ? 0.0 : dot(do_r, T->v + l * d, d);   /* dP_rl */
            D += p[l] * dp[l];
        }
        T->lse_all[r] = m + log(ell);
        T->D_all[r] = D;
        if (T->o_all) {
            double *o_r = T->o_all + r * d;
            for (int64_t c = 0; c < d; ++c)
                o_r[c] = 0.0;
            for (int64_t l = 0; l < Tk; ++l) {
                if (p[l] == 0.0)
                    continue;
                for (int64_t c = 0; c < d; ++c)
                    o_r[c] += p[l] * T->v[l * d + c];
            }
        }
        if (slot >= 0) {
            double *dq_r = T->dq + slot * d;
            for (int64_t c = 0; c < d; ++c)
                dq_r[c] = 0.0;
            for (int64_t l = 0; l < Tk; ++l) {
                const double ds = p[l] * (dp[l] - D);      /* dS_rl */
                if (ds == 0.0)
                    continue;
                for (int64_t c = 0; c < d; ++c)
                    dq_r[c] += ds * T->k[l * d + c];
            }
            for (int64_t c = 0; c < d; ++c)
                dq_r[c] *= T->scale;
        }
    }
    free(p);
    free(dp);
    return NULL;
}

static void *bwd_keys_worker(void *arg)
{
    bwd_task *T = (bwd_task *)arg;
    const int64_t d = T->d;
    for (int64_t i = T->tid; i < T->nkeys; i += T->nthreads) {
        const int64_t l = T->keys[i];
        const double *k_l = T->k + l * d;
        const double *v_l = T->v + l * d;
        double *dk_l = T->dk + i * d;
        double *dv_l = T->dv + i * d;
        for (int64_t c = 0; c < d; ++c) {
            dk_l[c] = 0.0;
            dv_l[c] = 0.0;
        }
        for (int64_t r = 0; r < T->Tq; ++r) {
            if (!is_allowed(r, l, T->Tq, T->Tk, &T->mask) || T->lse_all[r] == -INFINITY)
                continue;
            const double *q_r = T->q + r * d;
            const double *do_r = T->dO + r * d;
            const double P = exp(T->scale * dot(q_r, k_l, d) - T->lse_all[r]);
            const double dP = dot(do_r, v_l, d);
            const double dS = P * (dP - T->D_all[r]);
            for (int64_t c = 0; c < d; ++c) {
                dv_l[c] += P * do_r[c];
                dk_l[c] += dS * q_r[c];
            }
        }
        for (int64_t c = 0; c < d; ++c)
            dk_l[c] *= T->scale;
    }
    return NULL;
}

/*
 * oracle_bwd: gradients of one head.
 *   rows/nrows: query rows whose dQ is wanted  -> dq [nrows][d]
 *   keys/nkeys: key rows whose dK, dV are wanted -> dk, dv [nkeys][d]
 *   lse_all, D_all [Tq] are always written; o_all [Tq][d] if non-NULL.
 * Returns 0 on success.
 */
static int bwd_run(const double *q, const double *k, const double *v, const double *dO,
                   int64_t Tq, int64_t Tk, int64_t d, mask_t mask, double scale,
                   const int64_t *rows, int64_t nrows,
                   const int64_t *keys, int64_t nkeys,
                   double *dq, double *dk, double *dv,
                   double *o_all, double *lse_all, double *D_all, int nthreads)
{
    if (Tq < 0 || Tk < 0 || d < 1 || nrows < 0 || nkeys < 0 || nthreads < 1)
        return 2;
    int64_t *row_slot = (int64_t *)malloc(sizeof(int64_t) * (size_t)(Tq > 0 ? Tq : 1));
    bwd_task *tasks = (bwd_task *)calloc((size_t)nthreads, sizeof(bwd_task));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!row_slot || !tasks || !th) {
        free(row_slot);
        free(tasks);
        free(th);
        return 1;
    }
    int status = 0;
    for (int64_t r = 0; r < Tq; ++r)
        row_slot[r] = -1;
    for (int64_t i = 0; i < nrows; ++i) {
        if (rows[i] < 0 || rows[i] >= Tq || row_slot[rows[i]] >= 0)
            status = 2;
        else
            row_slot[rows[i]] = i;
    }
    for (int64_t i = 0; i < nkeys; ++i)
        if (keys[i] < 0 || keys[i] >= Tk)
            status = 2;
    if (status) {
        free(row_slot);
        free(tasks);
        free(th);
        return status;
    }
    for (int t = 0; t < nthreads; ++t) {
        bwd_task x = {q, k, v, dO, Tq, Tk, d, mask, scale, row_slot, keys, nkeys,
                      dq, dk, dv, o_all, lse_all, D_all, nthreads, t, 0};
        tasks[t] = x;
    }
    for (int t = 0; t < nthreads; ++t)
        pthread_create(&th[t], NULL, bwd_rows_worker, &tasks[t]);
    for (int t = 0; t < nthreads; ++t)
        pthread_join(th[t], NULL);
    for (int t = 0; t < nthreads; ++t)
        status |= tasks[t].status;
    if (!status) {
        for (int t = 0; t < nthreads; ++t)
            pthread_create(&th[t], NULL, bwd_keys_worker, &tasks[t]);
        for (int t = 0; t < nthreads; ++t)
            pthread_join(th[t], NULL);
    }
    free(row_slot);
    free(tasks);
    free(th);
    return status;
}

int oracle_bwd(const double *q, const double *k, const double *v, const double *dO,
               int64_t Tq, int64_t Tk, int64_t d, int causal, double scale,
               const int64_t *rows, int64_t nrows,
               const int64_t *keys, int64_t nkeys,
               double *dq, double *dk, double *dv,
               double *o_all, double *lse_all, double *D_all, int nthreads)
{
    return bwd_run(q, k, v, dO, Tq, Tk, d, causal_mask(causal), scale, rows, nrows, keys, nkeys, dq, dk, dv,
                   o_all, lse_all, D_all, nthreads);
}

/* oracle_bwd_masked: oracle_bwd under the window and block mask of oracle_fwd_masked. */
int oracle_bwd_masked(const double *q, const double *k, const double *v, const double *dO,
                      int64_t Tq, int64_t Tk, int64_t d, int64_t left, int64_t right,
                      const uint8_t *block, int64_t bs, double scale,
                      const int64_t *rows, int64_t nrows,
                      const int64_t *keys, int64_t nkeys,
                      double *dq, double *dk, double *dv,
                      double *o_all, double *lse_all, double *D_all, int nthreads)
{
    if (left < -1 || right < -1 || (block && bs < 1))
        return 2;
    mask_t m = {left, right, block, block ? bs : 1};
    return bwd_run(q, k, v, dO, Tq, Tk, d, m, scale, rows, nrows, keys, nkeys, dq, dk, dv,
                   o_all, lse_all, D_all, nthreads);
}
