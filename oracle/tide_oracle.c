/*
 * CPU oracle of the TIDE layout-aware reduce-scatter and all-gather placement.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg load this file's library.  It shares no code, header, table or constant with the CUDA
 * library: it is the plain definition of the result, written out with straight loops, so that
 * a reader can check it against the paper by eye.
 *
 * "TIDE" below is the paper "The Endgame of FSDP Communication: Layout-Aware Collectives on Copy
 * Engines, RDMA, and NVSwitch" (arXiv 2610.38228).  What it fixes:
 *   - abstract: FSDP2 stores each parameter and its gradient as its own tensor; the reduce-scatter
 *     takes those bf16 tensors as they are and sums them into fp32 shards; the all-gather writes
 *     the shards straight into the parameters' storage.
 *   - Fig. 1: each parameter is cut on dim 0 into one piece per rank, and each piece goes to its
 *     destination in a single write.
 *   - Table 2 (notation): for parameter p, the rows each rank holds after padding, the length of a
 *     row, the elements of p in one rank's shard and where they start; the size of one rank's
 *     whole shard and of the unsharded group.
 * Readings taken where the pages are silent (the symbols of Table 2 are lost in the text):
 *   - padded rows  m_p = ceil(rows_p / R)  (FSDP2 / torch.chunk dim-0 sharding);
 *   - per-rank shard  s_p = m_p * L_p  elements, prefix offset  o_p = sum_{q<p} s_q  (tight packing,
 *     no alignment gaps);  S = sum_p s_p,  U = sum_p rows_p * L_p;
 *   - rank d holds rows [d*m_p, d*m_p + m_p) of p; rows past rows_p are padding;
 *   - reduce-scatter sums (no averaging) over ranks r = 0..R-1 in ascending order, starting
 *     from the fp32 value of rank 0's element, with IEEE binary32 round-to-nearest-even adds,
 *     and writes +0.0f into padding;
 *   - the all-gather shard uses the same m_p, o_p in bf16 elements; padding is never read.
 *
 * Build: gcc -O2 -std=c11 -fno-fast-math -ffp-contract=off -fPIC -shared (no FMA contraction,
 * no flush-to-zero).  Pointers to R*P gradient tensors are indexed [r*P + p].
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)

/* bf16 -> fp32 widening is exact: the bf16 pattern is the top half of the fp32 pattern. */
float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Planner (Table 2 quantities).  m, s, o have P entries. */
int oracle_plan(int32_t R, int32_t P, const int64_t *rows, const int64_t *row_len,
                int64_t *m, int64_t *s, int64_t *o, int64_t *S, int64_t *U)
{
    if (R < 1 || P < 1 || !rows || !row_len || !m || !s || !o || !S || !U)
        return ORACLE_EINVAL;
    int64_t offset = 0, unsharded = 0;
    for (int32_t p = 0; p < P; ++p) {
        if (rows[p] < 1 || row_len[p] < 1)
            return ORACLE_EINVAL;
        m[p] = (rows[p] + R - 1) / R;
        s[p] = m[p] * row_len[p];
        o[p] = offset;
        offset += s[p];
        unsharded += rows[p] * row_len[p];
    }
    *S = offset;
    *U = unsharded;
    return ORACLE_OK;
}

/* Valid (non-padding) rows that rank d holds of a parameter with rows_p rows, m_p per rank. */
int64_t oracle_valid_rows(int64_t rows_p, int64_t m_p, int32_t d)
{
    int64_t v = rows_p - (int64_t)d * m_p;
    if (v < 0)
        v = 0;
    if (v > m_p)
        v = m_p;
    return v;
}

typedef struct {
    int64_t *m, *s, *o;
    int64_t S, U;
} oracle_layout;

static int layout_make(oracle_layout *L, int32_t R, int32_t P, const int64_t *rows,
                       const int64_t *row_len)
{
    L->m = NULL;
    L->s = NULL;
    L->o = NULL;
    if (P < 1)
        return ORACLE_EINVAL;
    L->m = (int64_t *)malloc(sizeof(int64_t) * (size_t)P);
    L->s = (int64_t *)malloc(sizeof(int64_t) * (size_t)P);
    L->o = (int64_t *)malloc(sizeof(int64_t) * (size_t)P);
    if (!L->m || !L->s || !L->o)
        return ORACLE_ENOMEM;
    return oracle_plan(R, P, rows, row_len, L->m, L->s, L->o, &L->S, &L->U);
}

static void layout_free(oracle_layout *L)
{
    free(L->m);
    free(L->s);
    free(L->o);
}

/*
 * Reduce-scatter (abstract; Fig. 1; Fig. 2b step 5): for every destination rank d, parameter p,
 * padded row j < m_p and column k < L_p,
 *     shard[d][o_p + j*L_p + k] = g[0][p][i] + g[1][p][i] + ... + g[R-1][p][i]   (fp32, left fold)
 * with i = (d*m_p + j)*L_p + k when d*m_p + j < rows_p, and +0.0f otherwise.
 *
 * oracle_reduce_scatter_part computes that definition for one destination rank d and the
 * parameters p_begin <= p < p_end only (it writes nothing but those elements of shards[d]), so
 * that a caller can run disjoint parts on several host threads; oracle_reduce_scatter is the
 * whole group, every destination rank and every parameter, one part after another.
 */
int oracle_reduce_scatter_part(int32_t R, int32_t P, const int64_t *rows, const int64_t *row_len,
                               const uint16_t *const *grads, float *const *shards, int32_t d,
                               int32_t p_begin, int32_t p_end)
{
    if (!grads || !shards || d < 0 || d >= R || p_begin < 0 || p_end > P || p_begin > p_end)
        return ORACLE_EINVAL;
    oracle_layout L;
    int rc = layout_make(&L, R, P, rows, row_len);
    if (rc != ORACLE_OK) {
        layout_free(&L);
        return rc;
    }
    for (int32_t p = p_begin; p < p_end; ++p) {
        for (int64_t j = 0; j < L.m[p]; ++j) {
            int64_t row = (int64_t)d * L.m[p] + j;
            for (int64_t k = 0; k < row_len[p]; ++k) {
                float acc;
                if (row < rows[p]) {
                    int64_t i = row * row_len[p] + k;
                    acc = oracle_bf16_to_f32(grads[0 * (int64_t)P + p][i]);
                    for (int32_t r = 1; r < R; ++r)
                        acc = acc + oracle_bf16_to_f32(grads[(int64_t)r * P + p][i]);
                } else {
                    acc = 0.0f;
                }
                shards[d][L.o[p] + j * row_len[p] + k] = acc;
            }
        }
    }
    layout_free(&L);
    return ORACLE_OK;
}

int oracle_reduce_scatter(int32_t R, int32_t P, const int64_t *rows, const int64_t *row_len,
                          const uint16_t *const *grads, float *const *shards)
{
    if (!grads || !shards || R < 1)
        return ORACLE_EINVAL;
    for (int32_t d = 0; d < R; ++d) {
        int rc = oracle_reduce_scatter_part(R, P, rows, row_len, grads, shards, d, 0, P);
        if (rc != ORACLE_OK)
            return rc;
    }
    return ORACLE_OK;
}

/* Same layout as oracle_reduce_scatter, but the sum is taken in fp64 (its own rounding error is at
 * most (R-1)*2^-53*sum|g|, far below any fp32 tolerance).  Used only as the reference against which
 * a summation order other than ascending rank is bounded. */
int oracle_exact_sum(int32_t R, int32_t P, const int64_t *rows, const int64_t *row_len,
                     const uint16_t *const *grads, double *const *exact)
{
    if (!grads || !exact)
        return ORACLE_EINVAL;
    oracle_layout L;
    int rc = layout_make(&L, R, P, rows, row_len);
    if (rc != ORACLE_OK) {
        layout_free(&L);
        return rc;
    }
    for (int32_t d = 0; d < R; ++d)
        for (int32_t p = 0; p < P; ++p)
            for (int64_t j = 0; j < L.m[p]; ++j) {
                int64_t row = (int64_t)d * L.m[p] + j;
                for (int64_t k = 0; k < row_len[p]; ++k) {
                    double acc = 0.0;
                    if (row < rows[p])
                        for (int32_t r = 0; r < R; ++r)
                            acc += (double)oracle_bf16_to_f32(
                                grads[(int64_t)r * P + p][row * row_len[p] + k]);
                    exact[d][L.o[p] + j * row_len[p] + k] = acc;
                }
            }
    layout_free(&L);
    return ORACLE_OK;
}

/*
 * All-gather placement (abstract; Fig. 1; Fig. 5b): for every source rank r, parameter p and
 * padded row j < m_p with r*m_p + j < rows_p,
 *     param[p][(r*m_p + j)*L_p + k] = shard[r][o_p + j*L_p + k]     for k < L_p.
 * Padding rows of the shards are never read; nothing outside the rows_p rows is written.
 *
 * oracle_all_gather_part places the rows of one source rank r for the parameters
 * p_begin <= p < p_end only (disjoint parts may run on several host threads);
 * oracle_all_gather is every source rank and every parameter, one part after another.
 */
int oracle_all_gather_part(int32_t R, int32_t P, const int64_t *rows, const int64_t *row_len,
                           const uint16_t *const *shards, uint16_t *const *params, int32_t r,
                           int32_t p_begin, int32_t p_end)
{
    if (!shards || !params || r < 0 || r >= R || p_begin < 0 || p_end > P || p_begin > p_end)
        return ORACLE_EINVAL;
    oracle_layout L;
    int rc = layout_make(&L, R, P, rows, row_len);
    if (rc != ORACLE_OK) {
        layout_free(&L);
        return rc;
    }
    for (int32_t p = p_begin; p < p_end; ++p)
        for (int64_t j = 0; j < L.m[p]; ++j) {
            int64_t row = (int64_t)r * L.m[p] + j;
            if (row >= rows[p])
                continue;
            for (int64_t k = 0; k < row_len[p]; ++k)
                params[p][row * row_len[p] + k] = shards[r][L.o[p] + j * row_len[p] + k];
        }
    layout_free(&L);
    return ORACLE_OK;
}

int oracle_all_gather(int32_t R, int32_t P, const int64_t *rows, const int64_t *row_len,
                      const uint16_t *const *shards, uint16_t *const *params)
{
    if (!shards || !params || R < 1)
        return ORACLE_EINVAL;
    for (int32_t r = 0; r < R; ++r) {
        int rc = oracle_all_gather_part(R, P, rows, row_len, shards, params, r, 0, P);
        if (rc != ORACLE_OK)
            return rc;
    }
    return ORACLE_OK;
}

/* The inverse: pack per-parameter bf16 tensors into R packed shards.  Padding positions are left
 * as the caller filled them. */
int oracle_shard_bf16(int32_t R, int32_t P, const int64_t *rows, const int64_t *row_len,
                      const uint16_t *const *params, uint16_t *const *shards)
{
    if (!shards || !params)
        return ORACLE_EINVAL;
    oracle_layout L;
    int rc = layout_make(&L, R, P, rows, row_len);
    if (rc != ORACLE_OK) {
        layout_free(&L);
        return rc;
    }
    for (int32_t r = 0; r < R; ++r)
        for (int32_t p = 0; p < P; ++p)
            for (int64_t j = 0; j < L.m[p]; ++j) {
                int64_t row = (int64_t)r * L.m[p] + j;
                if (row >= rows[p])
                    continue;
                for (int64_t k = 0; k < row_len[p]; ++k)
                    shards[r][L.o[p] + j * row_len[p] + k] = params[p][row * row_len[p] + k];
            }
    layout_free(&L);
    return ORACLE_OK;
}
