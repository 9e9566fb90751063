/*
 * swa_oracle.c -- plain fp64 CPU oracle for sliding-window scaled-dot-product
 * attention: the forward (O, LSE) and the backward (dQ, dK, dV, dSink, D).
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the smoke check and the CPU
 * baseline leg of the benchmark call this code. It shares nothing with the
 * CUDA path (no headers, no helpers, no tables) and must never be reached from
 * the product path.
 *
 * Sources (cuDNN-frontend pull requests, as extracted):
 *  - "frost(sdpa): bound the SM80 backward q-loop by the sliding window ...
 *    + window-aware deterministic relay" (#866), "Change" section: the anchor
 *    of a query row (q, or q + causal_diag under bottom-right alignment), the
 *    statement that a key is attended by no query whose anchor lies more than
 *    W rows past it, the window-only (non-causal) geometry, and THD packing
 *    with in-sequence indices.
 *  - "frost(sdpa): GQA/MQA, padding mask, right-band widening, and sink-token
 *    gradients for the SM120 f16 backward" (#557), "Summary" section: H_q a
 *    multiple of H_kv, per-batch actual lengths, keys right of the diagonal
 *    admitted by a right band, and the sink gradient
 *    dsink[h] = -sum_{b,q} exp(sink[h] - LSE[b,h,q]) * delta[b,h,q] taken over
 *    unpadded query rows only.
 *
 * Everything else is the textbook definition of softmax attention and its
 * gradient, written out term by term in fp64:
 *   s_ij = scale * q_i . k_j                    (attended pairs only)
 *   LSE_i = log( [sink] e^{sink_h} + sum_j e^{s_ij} )
 *   P_ij = e^{s_ij - LSE_i},  O_i = sum_j P_ij v_j
 *   D_i = dO_i . O_i
 *   dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - D_i)
 *   dV_j = sum_{h in group, i} P_ij dO_i
 *   dK_j = scale * sum_{h in group, i} dS_ij q_i
 *   dQ_i = scale * sum_j dS_ij k_j
 *   dSink_h = -sum_{b, i < Lq_b} e^{sink_h - LSE_i} D_i
 *
 * Readings taken where the pages leave a step open (each is listed in the
 * design notes of the repository):
 *  - window edge: key j is attended iff anchor(i) - j <= window_left, i.e.
 *    window_left + 1 keys including the diagonal (the pages' bound "no q with
 *    anchor(q) > kv_base + tile_kv - 1 + W" admits anchor = j + W);
 *  - causal_diag = Lkv_b - Lq_b under bottom-right alignment, 0 otherwise;
 *  - right band: j - anchor(i) <= window_right; causal modes treat a negative
 *    window_right as 0, the non-causal mode as unbounded;
 *  - the sink is a logit in the already scaled score space with no value row;
 *  - a row with no attended key and no sink has LSE = -inf, O = 0 and
 *    contributes nothing to the backward;
 *  - padded query rows get dQ = 0, padded keys dK = dV = 0.
 *
 * Layouts (contiguous, row-major):
 *   BSHD: Q, O, dO, dQ  [b, s_q, h_q, d];  K, V, dK, dV [b, s_kv, h_kv, d];
 *         LSE, D [b, h_q, s_q].
 *   THD:  Q, O, dO, dQ  [T_q, h_q, d];     K, V, dK, dV [T_kv, h_kv, d];
 *         LSE, D [h_q, T_q]; sequence bi occupies tokens
 *         [q_offsets[bi], q_offsets[bi] + Lq_bi) (and likewise for kv).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SWA_BSHD 0
#define SWA_THD 1

#define SWA_MASK_NONE 0
#define SWA_MASK_TOP_LEFT 1
#define SWA_MASK_BOTTOM_RIGHT 2

typedef struct {
    int32_t layout;        /* SWA_BSHD | SWA_THD */
    int32_t mask_mode;     /* SWA_MASK_* */
    int64_t b, h_q, h_kv, s_q, s_kv, d;
    int64_t window_left;   /* < 0: unbounded */
    int64_t window_right;  /* < 0: 0 for causal modes, unbounded otherwise */
    double scale;
    const int32_t *seq_q_lens;   /* [b] or NULL (BSHD: full s_q / s_kv) */
    const int32_t *seq_kv_lens;  /* [b] or NULL (THD: offsets differences) */
    const int64_t *q_offsets;    /* [b+1], THD only */
    const int64_t *kv_offsets;   /* [b+1], THD only */
    int32_t has_sink;
    int32_t nthreads;            /* worker threads, >= 1 */
    const uint8_t *unit_mask;    /* [b * h_kv] or NULL: only listed (batch,
                                    kv-head) units are computed */
} swa_problem;

/* ---- sequence geometry ------------------------------------------------- */

int64_t swa_len_q(const swa_problem *p, int64_t bi)
{
    if (p->seq_q_lens) return p->seq_q_lens[bi];
    if (p->layout == SWA_THD) return p->q_offsets[bi + 1] - p->q_offsets[bi];
    return p->s_q;
}

int64_t swa_len_kv(const swa_problem *p, int64_t bi)
{
    if (p->seq_kv_lens) return p->seq_kv_lens[bi];
    if (p->layout == SWA_THD) return p->kv_offsets[bi + 1] - p->kv_offsets[bi];
    return p->s_kv;
}

/* Element offset of (sequence bi, in-sequence row i, head h, feature 0). */
static int64_t q_index(const swa_problem *p, int64_t bi, int64_t i, int64_t h)
{
    if (p->layout == SWA_THD) return ((p->q_offsets[bi] + i) * p->h_q + h) * p->d;
    return ((bi * p->s_q + i) * p->h_q + h) * p->d;
}

static int64_t kv_index(const swa_problem *p, int64_t bi, int64_t j, int64_t g)
{
    if (p->layout == SWA_THD) return ((p->kv_offsets[bi] + j) * p->h_kv + g) * p->d;
    return ((bi * p->s_kv + j) * p->h_kv + g) * p->d;
}

/* Offset of the per-row statistic (LSE or D) of (bi, h, i). */
static int64_t stat_index(const swa_problem *p, int64_t bi, int64_t h, int64_t i)
{
    if (p->layout == SWA_THD) return h * p->q_offsets[p->b] + p->q_offsets[bi] + i;
    return (bi * p->h_q + h) * p->s_q + i;
}

/* ---- the mask predicate ------------------------------------------------ */

/* causal_diag of sequence bi: the shift that aligns the last query row with
 * the last key under bottom-right causal masking; 0 for the other modes. */
int64_t swa_diag(const swa_problem *p, int64_t bi)
{
    if (p->mask_mode == SWA_MASK_BOTTOM_RIGHT) return swa_len_kv(p, bi) - swa_len_q(p, bi);
    return 0;
}

/* Right bound in effect: causal modes clamp an unset bound to the diagonal. */
int64_t swa_right_bound(const swa_problem *p)
{
    if (p->mask_mode == SWA_MASK_NONE) return p->window_right;  /* < 0: none */
    return p->window_right > 0 ? p->window_right : 0;
}

/* 1 iff query row i of sequence bi attends key j (in-sequence indices). */
int swa_attended(const swa_problem *p, int64_t bi, int64_t i, int64_t j)
{
    int64_t lq = swa_len_q(p, bi), lkv = swa_len_kv(p, bi);
    if (i < 0 || i >= lq || j < 0 || j >= lkv) return 0;
    int64_t anchor = i + swa_diag(p, bi);
    if (p->window_left >= 0 && anchor - j > p->window_left) return 0;
    int64_t right = swa_right_bound(p);
    if (right >= 0 && j - anchor > right) return 0;
    return 1;
}

/* Keys a row can reach: [lo, hi). With dense != 0 the range is every key of
 * the sequence (the definition); otherwise it is cut to the window, which the
 * predicate still filters, so both sweeps add the same terms in the same
 * order. */
static void key_range(const swa_problem *p, int64_t bi, int64_t i, int dense,
                      int64_t *lo, int64_t *hi)
{
    int64_t lkv = swa_len_kv(p, bi);
    *lo = 0;
    *hi = lkv;
    if (dense) return;
    int64_t anchor = i + swa_diag(p, bi);
    if (p->window_left >= 0 && anchor - p->window_left > *lo) *lo = anchor - p->window_left;
    int64_t right = swa_right_bound(p);
    if (right >= 0 && anchor + right + 1 < *hi) *hi = anchor + right + 1;
    if (*hi < *lo) *hi = *lo;
}

static double dot(const double *a, const double *b, int64_t n)
{
    double s = 0.0;
    for (int64_t t = 0; t < n; ++t) s += a[t] * b[t];
    return s;
}

/* ---- work distribution -------------------------------------------------- */

typedef struct {
    const swa_problem *p;
    int64_t next;          /* shared unit counter, guarded by lock */
    pthread_mutex_t lock;
    void (*fn)(void *ctx, int64_t unit);
    void *ctx;
} pool_t;

static void *pool_worker(void *arg)
{
    pool_t *pool = (pool_t *)arg;
    int64_t units = pool->p->b * pool->p->h_kv;
    for (;;) {
        pthread_mutex_lock(&pool->lock);
        int64_t u = pool->next++;
        pthread_mutex_unlock(&pool->lock);
        if (u >= units) break;
        if (pool->p->unit_mask && !pool->p->unit_mask[u]) continue;
        pool->fn(pool->ctx, u);
    }
    return NULL;
}

/* Runs fn(ctx, unit) for every (batch, kv-head) unit. A unit is written by one
 * thread only, so results do not depend on the thread count. */
static void run_units(const swa_problem *p, void (*fn)(void *, int64_t), void *ctx)
{
    pool_t pool;
    pool.p = p;
    pool.next = 0;
    pool.fn = fn;
    pool.ctx = ctx;
    pthread_mutex_init(&pool.lock, NULL);
    int nt = p->nthreads > 0 ? p->nthreads : 1;
    if (nt > 256) nt = 256;
    pthread_t tid[256];
    for (int t = 1; t < nt; ++t) pthread_create(&tid[t], NULL, pool_worker, &pool);
    pool_worker(&pool);
    for (int t = 1; t < nt; ++t) pthread_join(tid[t], NULL);
    pthread_mutex_destroy(&pool.lock);
}

/* ---- forward ------------------------------------------------------------ */

typedef struct {
    const swa_problem *p;
    const double *q, *k, *v, *sink;
    double *o, *lse;
    int dense;
} fwd_ctx;

static void fwd_unit(void *arg, int64_t unit)
{
    fwd_ctx *c = (fwd_ctx *)arg;
    const swa_problem *p = c->p;
    int64_t bi = unit / p->h_kv, g = unit % p->h_kv;
    int64_t group = p->h_q / p->h_kv;
    int64_t lq = swa_len_q(p, bi);
    int64_t d = p->d;
    for (int64_t h = g * group; h < (g + 1) * group; ++h) {
        for (int64_t i = 0; i < lq; ++i) {
            const double *qi = c->q + q_index(p, bi, i, h);
            double *oi = c->o + q_index(p, bi, i, h);
            int64_t lo, hi;
            key_range(p, bi, i, c->dense, &lo, &hi);
            /* pass 1: the largest logit, for a safe exponent */
            double m = -INFINITY;
            if (p->has_sink) m = c->sink[h];
            for (int64_t j = lo; j < hi; ++j) {
                if (!swa_attended(p, bi, i, j)) continue;
                double s = p->scale * dot(qi, c->k + kv_index(p, bi, j, g), d);
                if (s > m) m = s;
            }
            for (int64_t t = 0; t < d; ++t) oi[t] = 0.0;
            if (m == -INFINITY) {  /* nothing attended and no sink */
                c->lse[stat_index(p, bi, h, i)] = -INFINITY;
                continue;
            }
            /* pass 2: the normaliser */
            double z = 0.0;
            if (p->has_sink) z += exp(c->sink[h] - m);
            for (int64_t j = lo; j < hi; ++j) {
                if (!swa_attended(p, bi, i, j)) continue;
                double s = p->scale * dot(qi, c->k + kv_index(p, bi, j, g), d);
                z += exp(s - m);
            }
            double lse = m + log(z);
            c->lse[stat_index(p, bi, h, i)] = lse;
            /* pass 3: O = sum_j P_ij v_j */
            for (int64_t j = lo; j < hi; ++j) {
                if (!swa_attended(p, bi, i, j)) continue;
                double s = p->scale * dot(qi, c->k + kv_index(p, bi, j, g), d);
                double pij = exp(s - lse);
                const double *vj = c->v + kv_index(p, bi, j, g);
                for (int64_t t = 0; t < d; ++t) oi[t] += pij * vj[t];
            }
        }
    }
}

/* O and LSE for every unpadded row; rows of unselected units are left as the
 * caller initialised them. Padded rows are not written. */
void swa_forward(const swa_problem *p, const double *q, const double *k, const double *v,
                 const double *sink, double *o, double *lse, int dense)
{
    fwd_ctx c = {p, q, k, v, sink, o, lse, dense};
    run_units(p, fwd_unit, &c);
}

/* ---- backward ----------------------------------------------------------- */

typedef struct {
    const swa_problem *p;
    const double *q, *k, *v, *o, *dout, *lse, *sink;
    double *dq, *dk, *dv, *delta, *dsink_part; /* dsink_part: [b, h_q] */
    int dense;
} bwd_ctx;

static void bwd_unit(void *arg, int64_t unit)
{
    bwd_ctx *c = (bwd_ctx *)arg;
    const swa_problem *p = c->p;
    int64_t bi = unit / p->h_kv, g = unit % p->h_kv;
    int64_t group = p->h_q / p->h_kv;
    int64_t lq = swa_len_q(p, bi), lkv = swa_len_kv(p, bi);
    int64_t d = p->d;

    /* this unit owns dK, dV of (bi, g) and dQ, D of the group's q-heads */
    for (int64_t j = 0; j < lkv; ++j) {
        double *dkj = c->dk + kv_index(p, bi, j, g), *dvj = c->dv + kv_index(p, bi, j, g);
        for (int64_t t = 0; t < d; ++t) dkj[t] = dvj[t] = 0.0;
    }
    for (int64_t h = g * group; h < (g + 1) * group; ++h) {
        double dsink = 0.0;
        for (int64_t i = 0; i < lq; ++i) {
            const double *qi = c->q + q_index(p, bi, i, h);
            const double *oi = c->o + q_index(p, bi, i, h);
            const double *doi = c->dout + q_index(p, bi, i, h);
            double *dqi = c->dq + q_index(p, bi, i, h);
            for (int64_t t = 0; t < d; ++t) dqi[t] = 0.0;
            double lse = c->lse[stat_index(p, bi, h, i)];
            double di = dot(doi, oi, d);
            c->delta[stat_index(p, bi, h, i)] = di;
            if (lse == -INFINITY) continue;  /* row attends nothing */
            if (p->has_sink) dsink -= exp(c->sink[h] - lse) * di;
            int64_t lo, hi;
            key_range(p, bi, i, c->dense, &lo, &hi);
            for (int64_t j = lo; j < hi; ++j) {
                if (!swa_attended(p, bi, i, j)) continue;
                const double *kj = c->k + kv_index(p, bi, j, g);
                const double *vj = c->v + kv_index(p, bi, j, g);
                double s = p->scale * dot(qi, kj, d);
                double pij = exp(s - lse);
                double dpij = dot(doi, vj, d);
                double dsij = pij * (dpij - di);
                double *dkj = c->dk + kv_index(p, bi, j, g);
                double *dvj = c->dv + kv_index(p, bi, j, g);
                for (int64_t t = 0; t < d; ++t) {
                    dvj[t] += pij * doi[t];
                    dkj[t] += p->scale * dsij * qi[t];
                    dqi[t] += p->scale * dsij * kj[t];
                }
            }
        }
        c->dsink_part[bi * p->h_q + h] = dsink;
    }
}

/* dQ, dK, dV and D for every unpadded row of the selected units; dsink[h]
 * (when the problem has a sink) sums the per-batch parts in batch order over
 * the selected units. Padded rows are not written: the caller zero-fills. */
void swa_backward(const swa_problem *p, const double *q, const double *k, const double *v,
                  const double *o, const double *dout, const double *lse, const double *sink,
                  double *dq, double *dk, double *dv, double *delta, double *dsink, int dense)
{
    double *part = (double *)calloc((size_t)(p->b * p->h_q), sizeof(double));
    bwd_ctx c = {p, q, k, v, o, dout, lse, sink, dq, dk, dv, delta, part, dense};
    run_units(p, bwd_unit, &c);
    if (p->has_sink && dsink) {
        for (int64_t h = 0; h < p->h_q; ++h) {
            double s = 0.0;
            for (int64_t bi = 0; bi < p->b; ++bi) s += part[bi * p->h_q + h];
            dsink[h] = s;
        }
    }
    free(part);
}

/* ---- the method's tile geometry (for brute-force identity checks) -------- */

static int64_t floor_div(int64_t a, int64_t b)
{
    int64_t q = a / b;
    if ((a % b != 0) && ((a < 0) != (b < 0))) --q;
    return q;
}

/* q-tile range [q_lo, q_hi) swept by kv-tile t of sequence bi: the lower bound
 * is the first q-tile holding a row that can reach the tile's first key
 * (causal skip, widened by the right band); the upper bound is the pages'
 * clamp ceil((kv_base + tile_kv + W - diag) / tile_q), capped at the number of
 * q-tiles. */
void swa_tile_q_range(const swa_problem *p, int64_t bi, int64_t t, int64_t tile_q,
                      int64_t tile_kv, int64_t *q_lo, int64_t *q_hi)
{
    int64_t lq = swa_len_q(p, bi);
    int64_t n_q = (lq + tile_q - 1) / tile_q;
    int64_t diag = swa_diag(p, bi);
    int64_t kv_base = t * tile_kv;
    int64_t right = swa_right_bound(p);
    int64_t lo = 0, hi = n_q;
    if (right >= 0) {
        int64_t first_row = kv_base - right - diag;
        lo = first_row > 0 ? first_row / tile_q : 0;
    }
    if (p->window_left >= 0) {
        int64_t c = floor_div(kv_base + tile_kv + p->window_left - diag + tile_q - 1, tile_q);
        if (c < hi) hi = c;
    }
    if (hi < lo) hi = lo;
    if (lo > n_q) lo = hi = n_q;
    *q_lo = lo;
    *q_hi = hi;
}

/* First kv-tile of the deterministic relay for q-tile j:
 * max((q_row0 + diag - W) // tile_kv, 0), or 0 without a left window. */
int64_t swa_kv_first(const swa_problem *p, int64_t bi, int64_t j, int64_t tile_q,
                     int64_t tile_kv)
{
    if (p->window_left < 0) return 0;
    int64_t v = floor_div(j * tile_q + swa_diag(p, bi) - p->window_left, tile_kv);
    return v > 0 ? v : 0;
}
