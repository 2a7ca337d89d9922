/*
 * Ulysses sequence parallelism -- plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may call this code.  It shares nothing with the
 * CUDA library: no header, no helper, no table.  It is deliberately slow and
 * written so that each loop can be checked against the definitions by eye.
 *
 * What it computes (definitions, not an algorithm):
 *
 *   seq->head swap ("Ulysses sequence parallelism" page, the all-to-all
 *   diagram; blog summary "How Ulysses Sequence Parallelism Works", step 3):
 *     rank s holds tokens [s*N/P, (s+1)*N/P) for all H heads; after the
 *     all-to-all, rank r holds all N tokens for heads [r*H/P, (r+1)*H/P).
 *       head[r][b][n][h'][k] = seq[n / (N/P)][b][n % (N/P)][r*H/P + h'][k]
 *   head->seq swap: the inverse map (same diagram, second all-to-all; step 5).
 *
 *   attention over a head shard (blog summary, step 4 "Local Attention"):
 *     s_ij  = scale * <q_i, k_j>                     for allowed (i, j)
 *     lse_i = ln sum_j exp(s_ij)
 *     o_i   = sum_j exp(s_ij - lse_i) v_j
 *   allowed(i, j): j <= i when causal; doc(i) == doc(j) when documents are
 *   packed (FlashAttention-style varlen masking, recommended when packing in
 *   the Transformers page "sp_attn_implementation").  GQA: local query head h
 *   reads local KV head h / (Hq/Hkv).
 *
 *   attention backward (the gradient of the above; the pages only say that
 *   the gradients must be correct, blog summary "Transformers Trainer"):
 *     D_i   = <dO_i, O_i>
 *     P_ij  = exp(s_ij - lse_i)
 *     dP_ij = <dO_i, v_j>
 *     dS_ij = P_ij (dP_ij - D_i)
 *     dq_i  = scale sum_j dS_ij k_j
 *     dk_j  = scale sum_{h in group} sum_i dS_ij q_i
 *     dv_j  = sum_{h in group} sum_i P_ij dO_i
 *
 * Layouts (row-major, element counts):
 *   seq  : [P][B][N/P][H][d]       head : [P][B][N][H/P][d]
 *   q, o, dO, dq : [S][B][N][Hq][d]   k, v, dk, dv : [S][B][N][Hkv][d]
 *   lse  : [S][B][Hq][N]
 * where S is the number of head shards passed in (Hq, Hkv are per shard).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ swap */

void oracle_seq_to_head(const uint8_t *x_seq, uint8_t *x_head, int64_t B, int64_t N,
                        int64_t H, int64_t d, int64_t P, int64_t esize)
{
    const int64_t Np = N / P, Hp = H / P;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t r = 0; r < P; r++)
        for (int64_t n = 0; n < N; n++) {
            const int64_t s = n / Np; /* rank that held token n before the swap */
            const int64_t t = n % Np; /* its position inside that rank's chunk */
            for (int64_t b = 0; b < B; b++)
                for (int64_t hh = 0; hh < Hp; hh++)
                    for (int64_t k = 0; k < d; k++) {
                        const int64_t src = (((s * B + b) * Np + t) * H + (r * Hp + hh)) * d + k;
                        const int64_t dst = (((r * B + b) * N + n) * Hp + hh) * d + k;
                        memcpy(x_head + dst * esize, x_seq + src * esize, (size_t)esize);
                    }
        }
}

void oracle_head_to_seq(const uint8_t *x_head, uint8_t *x_seq, int64_t B, int64_t N,
                        int64_t H, int64_t d, int64_t P, int64_t esize)
{
    const int64_t Np = N / P, Hp = H / P;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t r = 0; r < P; r++)
        for (int64_t n = 0; n < N; n++) {
            const int64_t s = n / Np;
            const int64_t t = n % Np;
            for (int64_t b = 0; b < B; b++)
                for (int64_t hh = 0; hh < Hp; hh++)
                    for (int64_t k = 0; k < d; k++) {
                        const int64_t dst = (((s * B + b) * Np + t) * H + (r * Hp + hh)) * d + k;
                        const int64_t src = (((r * B + b) * N + n) * Hp + hh) * d + k;
                        memcpy(x_seq + dst * esize, x_head + src * esize, (size_t)esize);
                    }
        }
}

/* ------------------------------------------------------------ attention */

typedef struct {
    int64_t S, B, N, Hq, Hkv, d;
    int causal;
    const int32_t *cu; /* cu_seqlens [ndocs+1] or NULL */
    int ndocs;
    double scale;
} shape_t;

/* document index of token i: the k with cu[k] <= i < cu[k+1] (0 without docs) */
static int64_t doc_of(const shape_t *sh, int64_t i)
{
    if (!sh->cu)
        return 0;
    for (int k = 0; k < sh->ndocs; k++)
        if (i < (int64_t)sh->cu[k + 1])
            return k;
    return sh->ndocs - 1;
}

static int allowed(const shape_t *sh, int64_t i, int64_t j)
{
    if (sh->causal && j > i)
        return 0;
    if (sh->cu && doc_of(sh, i) != doc_of(sh, j))
        return 0;
    return 1;
}

static const double *row_q(const double *q, const shape_t *sh, int64_t s, int64_t b, int64_t h, int64_t i)
{
    return q + (((s * sh->B + b) * sh->N + i) * sh->Hq + h) * sh->d;
}

static const double *row_kv(const double *x, const shape_t *sh, int64_t s, int64_t b, int64_t kvh, int64_t j)
{
    return x + (((s * sh->B + b) * sh->N + j) * sh->Hkv + kvh) * sh->d;
}

static double dot(const double *a, const double *b, int64_t d)
{
    double acc = 0.0;
    for (int64_t k = 0; k < d; k++)
        acc += a[k] * b[k];
    return acc;
}

/* One query row: scores into sbuf (NAN where not allowed), returns lse_i and
 * writes o_i.  Three passes: max, sum of exponentials, weighted sum of v. */
static double attn_row(const double *q, const double *k, const double *v, const shape_t *sh,
                       int64_t s, int64_t b, int64_t h, int64_t i, double *o_i, double *sbuf)
{
    const int64_t kvh = h / (sh->Hq / sh->Hkv);
    const double *qi = row_q(q, sh, s, b, h, i);
    double m = -INFINITY;
    for (int64_t j = 0; j < sh->N; j++) {
        if (!allowed(sh, i, j)) {
            sbuf[j] = NAN;
            continue;
        }
        sbuf[j] = sh->scale * dot(qi, row_kv(k, sh, s, b, kvh, j), sh->d);
        if (sbuf[j] > m)
            m = sbuf[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < sh->N; j++)
        if (allowed(sh, i, j))
            l += exp(sbuf[j] - m);
    const double lse = m + log(l);
    for (int64_t c = 0; c < sh->d; c++)
        o_i[c] = 0.0;
    for (int64_t j = 0; j < sh->N; j++) {
        if (!allowed(sh, i, j))
            continue;
        const double p = exp(sbuf[j] - lse);
        const double *vj = row_kv(v, sh, s, b, kvh, j);
        for (int64_t c = 0; c < sh->d; c++)
            o_i[c] += p * vj[c];
    }
    return lse;
}

static shape_t make_shape(int64_t S, int64_t B, int64_t N, int64_t Hq, int64_t Hkv, int64_t d,
                          int causal, const int32_t *cu, int ndocs, double scale)
{
    shape_t sh = {S, B, N, Hq, Hkv, d, causal, (ndocs > 0 ? cu : NULL), ndocs, scale};
    return sh;
}

/* Full forward: o [S][B][N][Hq][d], lse [S][B][Hq][N]. */
void oracle_attn_fwd(const double *q, const double *k, const double *v, double *o, double *lse,
                     int64_t S, int64_t B, int64_t N, int64_t Hq, int64_t Hkv, int64_t d,
                     int causal, const int32_t *cu, int ndocs, double scale)
{
    const shape_t sh = make_shape(S, B, N, Hq, Hkv, d, causal, cu, ndocs, scale);
    const int64_t rows = S * B * Hq * N;
#pragma omp parallel
    {
        double *sbuf = (double *)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 16)
        for (int64_t idx = 0; idx < rows; idx++) {
            const int64_t i = idx % N;
            const int64_t h = (idx / N) % Hq;
            const int64_t b = (idx / (N * Hq)) % B;
            const int64_t s = idx / (N * Hq * B);
            double *oi = o + (((s * B + b) * N + i) * Hq + h) * d;
            lse[((s * B + b) * Hq + h) * N + i] = attn_row(q, k, v, &sh, s, b, h, i, oi, sbuf);
        }
        free(sbuf);
    }
}

/* Sampled forward rows.  rows: nrows x 4 int64 (s, b, h, i).
 * o_rows [nrows][d], lse_rows [nrows]. */
void oracle_attn_fwd_rows(const double *q, const double *k, const double *v,
                          int64_t S, int64_t B, int64_t N, int64_t Hq, int64_t Hkv, int64_t d,
                          int causal, const int32_t *cu, int ndocs, double scale,
                          const int64_t *rows, int64_t nrows, double *o_rows, double *lse_rows)
{
    const shape_t sh = make_shape(S, B, N, Hq, Hkv, d, causal, cu, ndocs, scale);
#pragma omp parallel
    {
        double *sbuf = (double *)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; r++) {
            const int64_t *x = rows + 4 * r;
            lse_rows[r] = attn_row(q, k, v, &sh, x[0], x[1], x[2], x[3], o_rows + r * d, sbuf);
        }
        free(sbuf);
    }
}

/* dq_i for one query row, given that row's lse_i and D_i. */
static void dq_row(const double *q, const double *k, const double *v, const double *dout,
                   const shape_t *sh, int64_t s, int64_t b, int64_t h, int64_t i,
                   double lse_i, double D_i, double *dq_i)
{
    const int64_t kvh = h / (sh->Hq / sh->Hkv);
    const double *qi = row_q(q, sh, s, b, h, i);
    const double *doi = row_q(dout, sh, s, b, h, i);
    for (int64_t c = 0; c < sh->d; c++)
        dq_i[c] = 0.0;
    for (int64_t j = 0; j < sh->N; j++) {
        if (!allowed(sh, i, j))
            continue;
        const double *kj = row_kv(k, sh, s, b, kvh, j);
        const double *vj = row_kv(v, sh, s, b, kvh, j);
        const double P = exp(sh->scale * dot(qi, kj, sh->d) - lse_i);
        const double dP = dot(doi, vj, sh->d);
        const double dS = P * (dP - D_i);
        for (int64_t c = 0; c < sh->d; c++)
            dq_i[c] += sh->scale * dS * kj[c];
    }
}

/* dk_j, dv_j for one key row of KV head kvh; lse/D indexed [S][B][Hq][N]. */
static void dkv_row(const double *q, const double *k, const double *v, const double *dout,
                    const double *lse, const double *D, const shape_t *sh,
                    int64_t s, int64_t b, int64_t kvh, int64_t j, double *dk_j, double *dv_j)
{
    const int64_t G = sh->Hq / sh->Hkv;
    const double *kj = row_kv(k, sh, s, b, kvh, j);
    const double *vj = row_kv(v, sh, s, b, kvh, j);
    for (int64_t c = 0; c < sh->d; c++) {
        dk_j[c] = 0.0;
        dv_j[c] = 0.0;
    }
    for (int64_t h = kvh * G; h < (kvh + 1) * G; h++) {
        const double *lse_h = lse + ((s * sh->B + b) * sh->Hq + h) * sh->N;
        const double *D_h = D + ((s * sh->B + b) * sh->Hq + h) * sh->N;
        for (int64_t i = 0; i < sh->N; i++) {
            if (!allowed(sh, i, j))
                continue;
            const double *qi = row_q(q, sh, s, b, h, i);
            const double *doi = row_q(dout, sh, s, b, h, i);
            const double P = exp(sh->scale * dot(qi, kj, sh->d) - lse_h[i]);
            const double dP = dot(doi, vj, sh->d);
            const double dS = P * (dP - D_h[i]);
            for (int64_t c = 0; c < sh->d; c++) {
                dk_j[c] += sh->scale * dS * qi[c];
                dv_j[c] += P * doi[c];
            }
        }
    }
}

/* Full backward.  Runs its own forward for O and lse, then the gradients.
 * Optional outputs o_out / lse_out (may be NULL) return that forward. */
void oracle_attn_bwd(const double *q, const double *k, const double *v, const double *dout,
                     double *dq, double *dk, double *dv, double *o_out, double *lse_out,
                     int64_t S, int64_t B, int64_t N, int64_t Hq, int64_t Hkv, int64_t d,
                     int causal, const int32_t *cu, int ndocs, double scale)
{
    const shape_t sh = make_shape(S, B, N, Hq, Hkv, d, causal, cu, ndocs, scale);
    const int64_t nq = S * B * N * Hq;
    double *o = (double *)malloc(sizeof(double) * (size_t)(nq * d));
    double *lse = (double *)malloc(sizeof(double) * (size_t)nq);
    double *D = (double *)malloc(sizeof(double) * (size_t)nq);
    oracle_attn_fwd(q, k, v, o, lse, S, B, N, Hq, Hkv, d, causal, cu, ndocs, scale);

    /* D_i = <dO_i, O_i>, stored like lse */
    for (int64_t s = 0; s < S; s++)
        for (int64_t b = 0; b < B; b++)
            for (int64_t h = 0; h < Hq; h++)
                for (int64_t i = 0; i < N; i++) {
                    const int64_t off = (((s * B + b) * N + i) * Hq + h) * d;
                    D[((s * B + b) * Hq + h) * N + i] = dot(dout + off, o + off, d);
                }

    /* query rows -> dq */
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t idx = 0; idx < nq; idx++) {
        const int64_t i = idx % N;
        const int64_t h = (idx / N) % Hq;
        const int64_t b = (idx / (N * Hq)) % B;
        const int64_t s = idx / (N * Hq * B);
        const int64_t li = ((s * B + b) * Hq + h) * N + i;
        dq_row(q, k, v, dout, &sh, s, b, h, i, lse[li], D[li],
               dq + (((s * B + b) * N + i) * Hq + h) * d);
    }

    /* key rows -> dk, dv (summed over the GQA group) */
    const int64_t nk = S * B * Hkv * N;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t idx = 0; idx < nk; idx++) {
        const int64_t j = idx % N;
        const int64_t kvh = (idx / N) % Hkv;
        const int64_t b = (idx / (N * Hkv)) % B;
        const int64_t s = idx / (N * Hkv * B);
        const int64_t off = (((s * B + b) * N + j) * Hkv + kvh) * d;
        dkv_row(q, k, v, dout, lse, D, &sh, s, b, kvh, j, dk + off, dv + off);
    }

    if (o_out)
        memcpy(o_out, o, sizeof(double) * (size_t)(nq * d));
    if (lse_out)
        memcpy(lse_out, lse, sizeof(double) * (size_t)nq);
    free(o);
    free(lse);
    free(D);
}

/* Sampled dq rows.  rows: nrows x 4 (s, b, h, i).  Each row recomputes its
 * own forward (lse_i, o_i) and D_i, then dq_i.  dq_rows [nrows][d]. */
void oracle_attn_bwd_q_rows(const double *q, const double *k, const double *v, const double *dout,
                            int64_t S, int64_t B, int64_t N, int64_t Hq, int64_t Hkv, int64_t d,
                            int causal, const int32_t *cu, int ndocs, double scale,
                            const int64_t *rows, int64_t nrows, double *dq_rows)
{
    const shape_t sh = make_shape(S, B, N, Hq, Hkv, d, causal, cu, ndocs, scale);
#pragma omp parallel
    {
        double *sbuf = (double *)malloc(sizeof(double) * (size_t)N);
        double *oi = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; r++) {
            const int64_t *x = rows + 4 * r;
            const double lse_i = attn_row(q, k, v, &sh, x[0], x[1], x[2], x[3], oi, sbuf);
            const double D_i = dot(row_q(dout, &sh, x[0], x[1], x[2], x[3]), oi, d);
            dq_row(q, k, v, dout, &sh, x[0], x[1], x[2], x[3], lse_i, D_i, dq_rows + r * d);
        }
        free(oi);
        free(sbuf);
    }
}

/* Sampled dk/dv rows.  keys: nkeys x 4 (s, b, kvh, j).  First every query
 * row i of the key's GQA group that may attend to one of the keys gets its
 * own forward (lse_i, o_i by attn_row) and D_i = <dO_i, o_i>, once even when
 * several keys share it; then each key sums over its rows with dkv_row, the
 * same per-key loop the full backward runs.  The result is therefore the
 * full backward's dk_j, dv_j bit for bit, at a cost of (#distinct attending
 * rows) * N * d.  dk_rows, dv_rows [nkeys][d]. */
void oracle_attn_bwd_kv_rows(const double *q, const double *k, const double *v, const double *dout,
                             int64_t S, int64_t B, int64_t N, int64_t Hq, int64_t Hkv, int64_t d,
                             int causal, const int32_t *cu, int ndocs, double scale,
                             const int64_t *keys, int64_t nkeys, double *dk_rows, double *dv_rows)
{
    const shape_t sh = make_shape(S, B, N, Hq, Hkv, d, causal, cu, ndocs, scale);
    const int64_t G = Hq / Hkv;
    const int64_t nq = S * B * Hq * N;
    /* lse and D indexed [S][B][Hq][N] as in oracle_attn_bwd; only the rows
     * some key needs are filled */
    double *lse = (double *)malloc(sizeof(double) * (size_t)nq);
    double *D = (double *)malloc(sizeof(double) * (size_t)nq);
    unsigned char *need = (unsigned char *)calloc((size_t)nq, 1);
    for (int64_t r = 0; r < nkeys; r++) {
        const int64_t s = keys[4 * r], b = keys[4 * r + 1], kvh = keys[4 * r + 2], j = keys[4 * r + 3];
        for (int64_t h = kvh * G; h < (kvh + 1) * G; h++)
            for (int64_t i = 0; i < N; i++)
                if (allowed(&sh, i, j))
                    need[((s * B + b) * Hq + h) * N + i] = 1;
    }
    int64_t nneed = 0;
    for (int64_t idx = 0; idx < nq; idx++)
        nneed += need[idx];
    int64_t *list = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nneed > 0 ? nneed : 1));
    nneed = 0;
    for (int64_t idx = 0; idx < nq; idx++)
        if (need[idx])
            list[nneed++] = idx;
#pragma omp parallel
    {
        double *sbuf = (double *)malloc(sizeof(double) * (size_t)N);
        double *oi = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < nneed; t++) {
            const int64_t idx = list[t];
            const int64_t i = idx % N;
            const int64_t h = (idx / N) % Hq;
            const int64_t b = (idx / (N * Hq)) % B;
            const int64_t s = idx / (N * Hq * B);
            lse[idx] = attn_row(q, k, v, &sh, s, b, h, i, oi, sbuf);
            D[idx] = dot(row_q(dout, &sh, s, b, h, i), oi, d);
        }
        free(oi);
        free(sbuf);
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nkeys; r++)
        dkv_row(q, k, v, dout, lse, D, &sh, keys[4 * r], keys[4 * r + 1], keys[4 * r + 2], keys[4 * r + 3],
                dk_rows + r * d, dv_rows + r * d);
    free(list);
    free(need);
    free(D);
    free(lse);
}
