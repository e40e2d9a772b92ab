/*
 * fp64 CPU oracle for weight-absorbed MLA decode over a paged latent cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) includes, links or calls this file; only the test
 * suite, the smoke check and the CPU-baseline leg of the benchmark do.  It
 * shares no code, header, table or helper with the CUDA sources.
 *
 * What it computes, and where that comes from:
 *
 *  - "Huawei Ascend servers: DeepSeek V3/R1 inference best practice",
 *    section 3.2.1 (Multi-head Latent Attention): all heads share one
 *    compressed KV cache, and decode uses weight absorption, so every head h
 *    of a query token attends over the same cached row r_j = c_kv_j || k_rope_j
 *    (512 + 64 values) with a per-head absorbed query q_lat^h || q_rope^h.
 *  - Same report, section 7.2 (cost formula BS x 3072 x (576+512) x 128 x 2
 *    x 2): the score contracts over 576 dims, the output over 512 dims, and
 *    there are 128 heads.
 *  - Same report, section 6.1: the attention kernel follows FlashAttention,
 *    i.e. it computes exact softmax attention; the plain definition below is
 *    therefore the result every tiling of it must reproduce.
 *
 * For one row (request b, query token t, head h) and the key range [j0, j1):
 *
 *     s_j  = scale * ( sum_{d<512} q_lat[d] r_j[d] + sum_{d<64} q_rope[d] r_j[512+d] )
 *     M    = max_j s_j,     Z = sum_j exp(s_j - M)
 *     o[d] = sum_j exp(s_j - M) r_j[d] / Z          (d < 512: V is c_kv itself)
 *     lse  = M + ln Z                                 (natural log)
 *
 * Readings taken where the pages are silent:
 *  - key j of request b lives at kv_cache[block_table[b][j / page]][j % page];
 *  - seq_lens[b] counts the cache including this step's s_q query tokens, and
 *    query token t (0 <= t < s_q) sees the first L_b - s_q + 1 + t keys
 *    (causal inside the multi-token-prediction step);
 *  - an empty key range yields o = 0 and lse = -inf, which is the neutral
 *    element of the split merge below.
 *
 * Split merge (FlashDecoding, the "MLAKernel performance root cause" part of
 * the Atlas 800I A3 TPOT-jitter troubleshooting post): partial results over
 * disjoint key ranges combine as
 *
 *     M = max_i lse_i,  w_i = exp(lse_i - M),
 *     o = sum_i w_i o_i / sum_i w_i,   lse = M + ln sum_i w_i.
 *
 * Every bf16 input is widened exactly to double; nothing is rounded inside.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_ELEM_BF16 0
#define ORACLE_ELEM_F64 1

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_SEQ_LEN 2
#define ORACLE_ERR_PAGE 3
#define ORACLE_ERR_RANGE 4
#define ORACLE_ERR_NOMEM 5

typedef struct {
    int32_t batch;      /* B */
    int32_t s_q;        /* query tokens per request in this step */
    int32_t num_heads;  /* H */
    int32_t d_latent;   /* 512 */
    int32_t d_rope;     /* 64 */
    int32_t page_size;  /* 64 */
    int32_t max_pages;  /* row stride of block_table */
    int32_t elem;       /* ORACLE_ELEM_BF16 (uint16 bit patterns) or ORACLE_ELEM_F64 */
    int64_t num_pages;  /* pages in kv_cache */
    double scale;
    const void *q_latent;       /* [B][s_q][H][d_latent] */
    const void *q_rope;         /* [B][s_q][H][d_rope]   */
    const void *kv_cache;       /* [num_pages][page_size][d_latent + d_rope] */
    const int32_t *block_table; /* [B][max_pages] */
    const int32_t *seq_lens;    /* [B] */
} mla_oracle_problem;

static double load_elem(const void *base, int64_t i, int32_t elem) {
    if (elem == ORACLE_ELEM_F64) return ((const double *)base)[i];
    /* bf16 is the upper half of an IEEE binary32: widening is exact. */
    uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Number of keys query token t of request b may see, or -1 if seq_len < s_q. */
static int64_t visible_keys(const mla_oracle_problem *P, int32_t b, int32_t t) {
    int64_t L = P->seq_lens[b];
    int64_t v = L - P->s_q + 1 + t;
    return v < 1 ? -1 : v;
}

/* Offset of key j's cached row for request b, or -1 for a bad page index. */
static int64_t row_offset(const mla_oracle_problem *P, int32_t b, int64_t j) {
    int64_t slot = j / P->page_size;
    if (slot >= P->max_pages) return -1;
    int64_t page = P->block_table[(int64_t)b * P->max_pages + slot];
    if (page < 0 || page >= P->num_pages) return -1;
    return (page * P->page_size + j % P->page_size) * (int64_t)(P->d_latent + P->d_rope);
}

/* One row (b, t, h) over keys [j0, j1).  s is scratch for j1 - j0 doubles. */
static int one_row(const mla_oracle_problem *P, int32_t b, int32_t t, int32_t h, int64_t j0,
                   int64_t j1, double *o, double *lse, double *s) {
    const int32_t dl = P->d_latent, dr = P->d_rope;
    const int64_t qrow = ((int64_t)b * P->s_q + t) * P->num_heads + h;
    const int64_t q_lat_off = qrow * dl, q_rope_off = qrow * dr;

    for (int32_t d = 0; d < dl; ++d) o[d] = 0.0;
    if (j0 >= j1) {
        *lse = -INFINITY;
        return ORACLE_OK;
    }
    /* scores */
    double M = -INFINITY;
    for (int64_t j = j0; j < j1; ++j) {
        int64_t r = row_offset(P, b, j);
        if (r < 0) return ORACLE_ERR_PAGE;
        double acc = 0.0;
        for (int32_t d = 0; d < dl; ++d)
            acc += load_elem(P->q_latent, q_lat_off + d, P->elem) *
                   load_elem(P->kv_cache, r + d, P->elem);
        for (int32_t d = 0; d < dr; ++d)
            acc += load_elem(P->q_rope, q_rope_off + d, P->elem) *
                   load_elem(P->kv_cache, r + dl + d, P->elem);
        s[j - j0] = P->scale * acc;
        if (s[j - j0] > M) M = s[j - j0];
    }
    /* softmax-weighted sum of the latent part of each row */
    double Z = 0.0;
    for (int64_t j = j0; j < j1; ++j) {
        double w = exp(s[j - j0] - M);
        Z += w;
        int64_t r = row_offset(P, b, j);
        for (int32_t d = 0; d < dl; ++d) o[d] += w * load_elem(P->kv_cache, r + d, P->elem);
    }
    for (int32_t d = 0; d < dl; ++d) o[d] /= Z;
    *lse = M + log(Z);
    return ORACLE_OK;
}

typedef struct {
    const mla_oracle_problem *P;
    int64_t nrows;
    const int32_t *rows;      /* nrows x (b, t, h), or NULL for all rows in (b, t, h) order */
    const int64_t *ranges;    /* nrows x (j0, j1), or NULL for [0, visible keys) */
    double *o;                /* nrows x d_latent */
    double *lse;              /* nrows */
    int64_t next;             /* shared work counter (under the mutex) */
    pthread_mutex_t mu;
    int err;
} job_t;

static void row_index(const job_t *J, int64_t i, int32_t *b, int32_t *t, int32_t *h) {
    if (J->rows) {
        *b = J->rows[3 * i];
        *t = J->rows[3 * i + 1];
        *h = J->rows[3 * i + 2];
    } else {
        const int64_t H = J->P->num_heads, S = J->P->s_q;
        *h = (int32_t)(i % H);
        *t = (int32_t)((i / H) % S);
        *b = (int32_t)(i / (H * S));
    }
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    const mla_oracle_problem *P = J->P;
    double *s = NULL;
    int64_t s_cap = 0;
    const int64_t chunk = 8;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int64_t i0 = J->next;
        J->next += chunk;
        int stop = J->err != ORACLE_OK;
        pthread_mutex_unlock(&J->mu);
        if (stop || i0 >= J->nrows) break;
        int64_t i1 = i0 + chunk < J->nrows ? i0 + chunk : J->nrows;
        for (int64_t i = i0; i < i1; ++i) {
            int32_t b, t, h;
            row_index(J, i, &b, &t, &h);
            int rc = ORACLE_OK;
            int64_t vis = -1, j0 = 0, j1 = 0;
            if (b < 0 || b >= P->batch || t < 0 || t >= P->s_q || h < 0 || h >= P->num_heads)
                rc = ORACLE_ERR_ARG;
            if (rc == ORACLE_OK) {
                vis = visible_keys(P, b, t);
                if (vis < 0) rc = ORACLE_ERR_SEQ_LEN;
            }
            if (rc == ORACLE_OK) {
                j0 = J->ranges ? J->ranges[2 * i] : 0;
                j1 = J->ranges ? J->ranges[2 * i + 1] : vis;
                if (j0 < 0 || j1 > vis || j0 > j1) rc = ORACLE_ERR_RANGE;
            }
            if (rc == ORACLE_OK && j1 - j0 > s_cap) {
                free(s);
                s_cap = j1 - j0;
                s = (double *)malloc((size_t)s_cap * sizeof(double));
                if (!s) {
                    s_cap = 0;
                    rc = ORACLE_ERR_NOMEM;
                }
            }
            if (rc == ORACLE_OK)
                rc = one_row(P, b, t, h, j0, j1, J->o + i * P->d_latent, J->lse + i, s);
            if (rc != ORACLE_OK) {
                pthread_mutex_lock(&J->mu);
                if (J->err == ORACLE_OK) J->err = rc;
                pthread_mutex_unlock(&J->mu);
                break;
            }
        }
    }
    free(s);
    return NULL;
}

/*
 * Attention rows.  rows == NULL computes all B * s_q * H rows in (b, t, h)
 * order; otherwise rows holds nrows triples (b, t, h).  ranges == NULL uses
 * each row's full visible key range; otherwise ranges holds nrows pairs
 * (j0, j1) with 0 <= j0 <= j1 <= visible keys.  Returns an ORACLE_* code.
 */
int mla_oracle_rows(const mla_oracle_problem *P, int64_t nrows, const int32_t *rows,
                    const int64_t *ranges, double *o, double *lse, int32_t nthreads) {
    if (!P || !o || !lse || nrows < 0 || P->batch < 1 || P->s_q < 1 || P->num_heads < 1 ||
        P->d_latent < 1 || P->d_rope < 0 || P->page_size < 1 || P->max_pages < 1 ||
        (P->elem != ORACLE_ELEM_BF16 && P->elem != ORACLE_ELEM_F64))
        return ORACLE_ERR_ARG;
    if (!rows && nrows != (int64_t)P->batch * P->s_q * P->num_heads) return ORACLE_ERR_ARG;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;

    job_t J;
    J.P = P;
    J.nrows = nrows;
    J.rows = rows;
    J.ranges = ranges;
    J.o = o;
    J.lse = lse;
    J.next = 0;
    J.err = ORACLE_OK;
    pthread_mutex_init(&J.mu, NULL);

    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) return ORACLE_ERR_NOMEM;
    int32_t started = 0;
    for (int32_t i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) worker(&J);
    for (int32_t i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.mu);
    return J.err;
}

/*
 * Merge n partial results (o_i: n x d values, lse_i: n values) over disjoint
 * key ranges into one (o: d values, lse).  All-empty input gives o = 0,
 * lse = -inf.
 */
int mla_oracle_merge(int32_t n, int32_t d, const double *o_parts, const double *lse_parts,
                     double *o, double *lse) {
    if (n < 0 || d < 1 || !o || !lse || (n > 0 && (!o_parts || !lse_parts))) return ORACLE_ERR_ARG;
    double M = -INFINITY;
    for (int32_t i = 0; i < n; ++i)
        if (lse_parts[i] > M) M = lse_parts[i];
    for (int32_t k = 0; k < d; ++k) o[k] = 0.0;
    if (M == -INFINITY) {
        *lse = -INFINITY;
        return ORACLE_OK;
    }
    double W = 0.0;
    for (int32_t i = 0; i < n; ++i) {
        double w = exp(lse_parts[i] - M);
        W += w;
        for (int32_t k = 0; k < d; ++k) o[k] += w * o_parts[(int64_t)i * d + k];
    }
    for (int32_t k = 0; k < d; ++k) o[k] /= W;
    *lse = M + log(W);
    return ORACLE_OK;
}
