/*
 * qsa_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU oracle for QSA decode attention over a sparse
 * selection of INT8 K/V cells.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load it.  It shares no code,
 * header, table or helper with the CUDA library; the two meet only through
 * the seeded input generator.
 *
 * What is computed (pages: "Strata PR #2220, attn_chunk_q8_v3_kernel",
 * opening description and kernel table; "Strata issue #8, round 9:
 * performance candidate set on v0.2.9", section R9-gpu-11, tests paragraph):
 * every query head scores each selected cell of an INT8 K/V pool reached
 * through a permuted page table; the attention output is the softmax-weighted
 * sum of the selected cells' dequantised V rows.  The page entry -1 masks a
 * cell ("page -1 masking").
 *
 * Readings where the pages are silent:
 *   - dequantised value = per-cell fp32 scale x int8 code (symmetric, no
 *     zero point), one scale per cell row for K and one for V;
 *   - score s = softmax_scale * (q . k_hat);
 *   - a masked cell is left out of the softmax, exactly as if it were not in
 *     the list; no valid cell gives an all-zero output;
 *   - an out-of-range list entry or page slot is an error here (the CUDA
 *     path masks it and raises a status bit instead);
 *   - pages of page_cells cells (1 by default: one entry per cell): logical
 *     position pos lies on page pos / page_cells at offset pos % page_cells,
 *     and a page entry e, a page of the pool, puts it in pool slot
 *     e * page_cells + offset (the pages leave the page size open);
 *   - an optional causal limit per query of the window: query t sees only
 *     the selected cells whose logical position is below limit[t] (a cell
 *     it does not see is left out of its softmax, as if masked).
 *
 * The chunked form (partials m, l, o per chunk and their merge) is here only
 * so the merge identity can be checked; the reference result is the plain
 * unchunked definition below.
 *
 * Everything is evaluated in double: int8 codes, fp32 scales and the caller's
 * query values (widened exactly from fp32 or bf16) convert to double without
 * rounding.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    ORACLE_OK = 0,
    ORACLE_ERR_POSITION = 1, /* selected logical position outside the page table */
    ORACLE_ERR_SLOT = 2,     /* page-table entry outside the pool (and not -1) */
    ORACLE_ERR_ARG = 3,
    ORACLE_ERR_NOMEM = 4
};

/* Step a1 (gather): logical position -> pool slot.  *slot = -1 means masked.
 * The page table has page_table_len entries of page_cells cells each. */
static int resolve_cell(const int32_t *page_table, int page_table_len, int page_cells,
                        int pool_cells, int32_t pos, int32_t *slot)
{
    if (pos < 0 || (int64_t)pos >= (int64_t)page_table_len * page_cells) return ORACLE_ERR_POSITION;
    int32_t s = page_table[pos / page_cells];
    if (s == -1) { *slot = -1; return ORACLE_OK; }
    if (s < 0 || s >= pool_cells / page_cells) return ORACLE_ERR_SLOT;
    *slot = s * page_cells + pos % page_cells;
    return ORACLE_OK;
}

/* Steps a2-a3 for one cell: dequantise the K row, dot it with the query. */
static double cell_score(int D, const double *q, const int8_t *k_row, float k_scale,
                         double softmax_scale)
{
    double dot = 0.0;
    for (int d = 0; d < D; ++d) {
        double k_hat = (double)k_scale * (double)k_row[d];
        dot += q[d] * k_hat;
    }
    return softmax_scale * dot;
}

/*
 * Score list positions [start, start+count) of one (sequence, KV head) for one
 * query row.  slots[i] = pool slot or -1 (masked); s[i] = score (valid cells).
 */
static int score_range(int D, int pool_cells, int page_table_len, int page_cells,
                       int32_t limit, const double *q, const int8_t *k_codes,
                       const float *k_scale, const int32_t *page_table, const int32_t *sel,
                       int start, int count, double softmax_scale, int32_t *slots, double *s)
{
    if (page_cells < 1 || pool_cells % page_cells != 0) return ORACLE_ERR_ARG;
    for (int i = 0; i < count; ++i) {
        int32_t slot;
        int err = resolve_cell(page_table, page_table_len, page_cells, pool_cells,
                               sel[start + i], &slot);
        if (err) return err;
        if (sel[start + i] >= limit) slot = -1; /* beyond this query's causal limit */
        slots[i] = slot;
        if (slot >= 0)
            s[i] = cell_score(D, q, k_codes + (size_t)slot * D, k_scale[slot], softmax_scale);
    }
    return ORACLE_OK;
}

/*
 * The plain definition for one query row over the whole selected list:
 *   m = max_i s_i,  w_i = exp(s_i - m),  out = sum_i w_i v_hat_i / sum_i w_i.
 * Subtracting m does not change the ratio; it only keeps exp finite.
 */
int qsa_oracle_attend_row(int D, int pool_cells, int page_table_len, int page_cells,
                          int32_t limit, const double *q, const int8_t *k_codes,
                          const int8_t *v_codes,
                          const float *k_scale, const float *v_scale,
                          const int32_t *page_table, const int32_t *sel, int n_sel,
                          double softmax_scale, double *out)
{
    if (D <= 0 || n_sel < 0 || !out) return ORACLE_ERR_ARG;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (n_sel == 0) return ORACLE_OK;
    int32_t *slots = (int32_t *)malloc((size_t)n_sel * sizeof(int32_t));
    double *s = (double *)malloc((size_t)n_sel * sizeof(double));
    if (!slots || !s) { free(slots); free(s); return ORACLE_ERR_NOMEM; }
    int err = score_range(D, pool_cells, page_table_len, page_cells, limit, q, k_codes,
                          k_scale, page_table, sel, 0, n_sel, softmax_scale, slots, s);
    if (err) { free(slots); free(s); return err; }

    double m = -INFINITY;
    int n_valid = 0;
    for (int i = 0; i < n_sel; ++i)
        if (slots[i] >= 0) { n_valid++; if (s[i] > m) m = s[i]; }
    if (n_valid > 0) {
        double L = 0.0;
        for (int i = 0; i < n_sel; ++i) {
            if (slots[i] < 0) continue;
            double w = exp(s[i] - m);
            L += w;
            const int8_t *v_row = v_codes + (size_t)slots[i] * D;
            double vs = (double)v_scale[slots[i]];
            for (int d = 0; d < D; ++d) out[d] += w * (vs * (double)v_row[d]);
        }
        for (int d = 0; d < D; ++d) out[d] /= L;
    }
    free(slots);
    free(s);
    return ORACLE_OK;
}

/*
 * Chunk partial over list positions [start, start+count) for one query row
 * (the pages' "partial accumulators, maxima, denominators"):
 *   m = max s_i (-inf if no valid cell), l = sum exp(s_i - m),
 *   o = sum exp(s_i - m) v_hat_i (not normalised).
 */
int qsa_oracle_chunk_partial(int D, int pool_cells, int page_table_len, int page_cells,
                             int32_t limit, const double *q, const int8_t *k_codes,
                             const int8_t *v_codes,
                             const float *k_scale, const float *v_scale,
                             const int32_t *page_table, const int32_t *sel, int start,
                             int count, double softmax_scale, double *m_out, double *l_out,
                             double *o_out)
{
    if (D <= 0 || count < 0 || start < 0 || !m_out || !l_out || !o_out) return ORACLE_ERR_ARG;
    for (int d = 0; d < D; ++d) o_out[d] = 0.0;
    *m_out = -INFINITY;
    *l_out = 0.0;
    if (count == 0) return ORACLE_OK;
    int32_t *slots = (int32_t *)malloc((size_t)count * sizeof(int32_t));
    double *s = (double *)malloc((size_t)count * sizeof(double));
    if (!slots || !s) { free(slots); free(s); return ORACLE_ERR_NOMEM; }
    int err = score_range(D, pool_cells, page_table_len, page_cells, limit, q, k_codes,
                          k_scale, page_table, sel, start, count, softmax_scale, slots, s);
    if (err) { free(slots); free(s); return err; }
    double m = -INFINITY;
    for (int i = 0; i < count; ++i)
        if (slots[i] >= 0 && s[i] > m) m = s[i];
    double l = 0.0;
    if (m > -INFINITY) {
        for (int i = 0; i < count; ++i) {
            if (slots[i] < 0) continue;
            double w = exp(s[i] - m);
            l += w;
            const int8_t *v_row = v_codes + (size_t)slots[i] * D;
            double vs = (double)v_scale[slots[i]];
            for (int d = 0; d < D; ++d) o_out[d] += w * (vs * (double)v_row[d]);
        }
    }
    *m_out = m;
    *l_out = l;
    free(slots);
    free(s);
    return ORACLE_OK;
}

/*
 * Split-K merge of chunk partials (the pages' "chunk kernel + merge"):
 *   M = max over chunks with l > 0 of m_c,  L = sum_c l_c exp(m_c - M),
 *   out = sum_c o_c exp(m_c - M) / L;  out = 0 when every chunk is empty.
 * o is laid out [n_chunks][D].
 */
void qsa_oracle_merge(int D, int n_chunks, const double *m, const double *l, const double *o,
                      double *out)
{
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    double M = -INFINITY;
    for (int c = 0; c < n_chunks; ++c)
        if (l[c] > 0.0 && m[c] > M) M = m[c];
    if (M == -INFINITY) return;
    double L = 0.0;
    for (int c = 0; c < n_chunks; ++c) {
        if (!(l[c] > 0.0)) continue;
        double f = exp(m[c] - M);
        L += l[c] * f;
        for (int d = 0; d < D; ++d) out[d] += o[(size_t)c * D + d] * f;
    }
    for (int d = 0; d < D; ++d) out[d] /= L;
}

/*
 * A whole call: B sequences x G KV heads x T queries x H query heads.
 *   q        [B][T][G*H][D]        (double, widened exactly by the caller)
 *   k/v      [B][G][pool][D]       int8 codes
 *   scales   [B][G][pool]          fp32
 *   pages    [B][page_table_len]   int32, pages of page_cells cells
 *   sel      CSR by sel_offsets[B+1]; the list and the page table belong to
 *            the sequence and are shared by its KV heads.
 *   limits   NULL, or [B][T]: query t of sequence b sees positions < limits[b][t].
 * rows: NULL for every output row, else n_rows flat row ids
 *   ((b*T + t)*G*H + h); out is [rows][D].
 * Rows are independent; OpenMP spreads them over the host cores when built
 * with -fopenmp.
 */
int qsa_oracle_decode_attn(int n_seq, int n_kv_heads, int q_per_kv, int head_dim,
                           int n_queries, int pool_cells, int page_table_len, int page_cells,
                           double softmax_scale, const double *q, const int8_t *k_pool,
                           const int8_t *v_pool, const float *k_scale, const float *v_scale,
                           const int32_t *page_table, const int32_t *sel,
                           const int64_t *sel_offsets, const int32_t *limits,
                           const int64_t *rows, int64_t n_rows, double *out)
{
    const int B = n_seq, G = n_kv_heads, H = q_per_kv, D = head_dim, T = n_queries;
    if (B < 0 || G <= 0 || H <= 0 || D <= 0 || T <= 0) return ORACLE_ERR_ARG;
    const int64_t total = (int64_t)B * T * G * H;
    if (!rows) n_rows = total;
    int err_all = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t flat = rows ? rows[r] : r;
        double *o = out + (size_t)r * D;
        if (flat < 0 || flat >= total) {
#pragma omp critical
            err_all = ORACLE_ERR_ARG;
            continue;
        }
        int h = (int)(flat % (G * H));
        int t = (int)((flat / (G * H)) % T);
        int b = (int)(flat / ((int64_t)G * H * T));
        int g = h / H;
        size_t kv_off = ((size_t)b * G + g) * (size_t)pool_cells;
        int err = qsa_oracle_attend_row(
            D, pool_cells, page_table_len, page_cells,
            limits ? limits[(size_t)b * T + t] : INT32_MAX, q + (size_t)flat * D, k_pool + kv_off * D,
            v_pool + kv_off * D, k_scale + kv_off, v_scale + kv_off,
            page_table + (size_t)b * page_table_len, sel + sel_offsets[b],
            (int)(sel_offsets[b + 1] - sel_offsets[b]), softmax_scale, o);
        if (err) {
#pragma omp critical
            err_all = err;
        }
    }
    return err_all;
}

/* Host threads the oracle uses (1 without OpenMP). */
int qsa_oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void qsa_oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
