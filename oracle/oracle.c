/*
 * Float64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the CUDA library computes.  It is called by the tests, by
 * the smoke check and by the bench's CPU-baseline leg, never by the library.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * Sources (page titles and sections):
 *   [p1] "手搓 Attention：从三行循环到看懂 FlashAttention"
 *        §1 (what attention computes: Q n×d, K m×d, V m×dv, O n×dv, scale),
 *        §2 version 0 (one query at a time, float64 accumulator, the
 *        reference every other version is checked against),
 *        §4 version 2 (subtract the row maximum before exp),
 *        §7 version 4 (the online-softmax recurrence over K/V blocks).
 *   [p2] "S12 FlashAttention"
 *        "解法" (single-query tiled recurrence with alpha = exp(m - m_new)),
 *        "实现" (paged variant: walk the block table, n = min(block_size,
 *        seq_len - logical*block_size), stop when n <= 0; the -inf/NaN note),
 *        "它还解锁了什么" + "练习" 1 (flash-decoding: split the keys, merge the
 *        (m, l, o) triples with the same rescale).
 *   [p3] "FlashAttention推理优化实战100例 01", 实现代码 (outer loop over Q
 *        blocks, inner loop over K/V blocks, state per Q block).
 *
 * Every function takes fp32 inputs (bf16 inputs are first widened exactly to
 * fp32 by the caller) and does all arithmetic in double.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - LSE = M + ln(l), natural log of the summed exp of SCALED scores.
 *   - causal: key j is visible to query i iff j <= i + (m - n) (0-based;
 *     queries are the last n of the m key positions).  For n == m this is the
 *     pages' "the i-th query sees keys up to i"; for n > m the first n - m
 *     queries see no key.
 *   - a row that sees no key at all: O = 0 and LSE = -inf.
 *   - grouped heads: query head h reads kv head h / (H / Hkv).
 *   - in the recurrence, a tile that is fully masked for a row while the
 *     running max is still -inf uses 0 as its subtraction reference, so its
 *     weights are exp(-inf) = 0 and alpha is taken as 1 (the state is empty).
 *
 * Parity pins (tests under tests/, CPU only): closed forms for Q = 0, one
 * dominant score, weights summing to one, invariance under a joint K/V row
 * permutation and under a constant shift of every K row, brute force against
 * a library softmax-attention routine on tiny inputs, the worked seed-42 case
 * of [p3], tile-size-1 recurrence equal to the full softmax [p2, 动手观察], and
 * split-combine equal to the unsplit result.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------- */
/* One query row, the plain definition ([p1] §2 version 0 with the §4 max  */
/* subtraction).  q: d floats; K rows at k + j*k_stride; V rows likewise.  */
/* visible(j) is "j < m_vis".  Writes dv outputs and the LSE; optionally   */
/* the m_vis softmax weights (instrumented mode used by the tests).        */
/* ---------------------------------------------------------------------- */
static void attend_one_row(const float *q, const float *k, long k_stride,
                           const float *v, long v_stride, int m_vis, int d,
                           int dv, double scale, double *o_out, double *lse_out,
                           double *w_out, double *scores /* m_vis scratch */)
{
    if (m_vis <= 0) {
        for (int c = 0; c < dv; ++c) o_out[c] = 0.0;
        *lse_out = -INFINITY;
        return;
    }
    /* step 1: s_j = scale * sum_k q[k] * K[j][k] */
    for (int j = 0; j < m_vis; ++j) {
        const float *kj = k + (long)j * k_stride;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += (double)q[c] * (double)kj[c];
        scores[j] = scale * dot;
    }
    /* step 2: M = max_j s_j */
    double M = scores[0];
    for (int j = 1; j < m_vis; ++j)
        if (scores[j] > M) M = scores[j];
    /* steps 3-4: w_j = exp(s_j - M), l = sum_j w_j */
    double l = 0.0;
    for (int j = 0; j < m_vis; ++j) {
        scores[j] = exp(scores[j] - M);
        l += scores[j];
    }
    /* step 5: O = sum_j w_j V[j] / l */
    for (int c = 0; c < dv; ++c) o_out[c] = 0.0;
    for (int j = 0; j < m_vis; ++j) {
        const float *vj = v + (long)j * v_stride;
        double w = scores[j] / l;
        if (w_out) w_out[j] = w;
        for (int c = 0; c < dv; ++c) o_out[c] += w * (double)vj[c];
    }
    /* step 6: LSE = M + ln l */
    *lse_out = M + log(l);
}

/* keys visible to query i of n, out of m: all of them, or the causal prefix
 * j <= i + (m - n) */
static int visible_keys(int i, int n, int m, int causal)
{
    if (!causal) return m;
    long v = (long)i + 1 + ((long)m - (long)n);
    if (v < 0) v = 0;
    if (v > m) v = m;
    return (int)v;
}

static int check_heads(int H, int Hkv)
{
    return H > 0 && Hkv > 0 && H % Hkv == 0;
}

/*
 * Dense attention, selected rows.
 * q [B][n][H][d], k [B][m][Hkv][d], v [B][m][Hkv][dv] (fp32, row-major).
 * rows: R triples (b, h, i).  Outputs o_rows [R][dv], lse_rows [R],
 * and, if w_rows != NULL, the weights [R][m] (zero where not visible).
 * Returns 0, or -1 on invalid arguments.
 */
int oracle_attention_rows_f64(const float *q, const float *k, const float *v,
                              int B, int H, int Hkv, int n, int m, int d, int dv,
                              double scale, int causal, const int *rows, int R,
                              double *o_rows, double *lse_rows, double *w_rows)
{
    if (!check_heads(H, Hkv) || B < 0 || n < 0 || m < 0 || d <= 0 || dv <= 0)
        return -1;
    for (int r = 0; r < R; ++r) {
        int b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= H || i < 0 || i >= n) return -1;
    }
    const int group = H / Hkv;
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)(m > 0 ? m : 1));
#pragma omp for schedule(dynamic, 16)
        for (int r = 0; r < R; ++r) {
            int b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
            int hk = h / group;
            int m_vis = visible_keys(i, n, m, causal);
            const float *qi = q + (((long)b * n + i) * H + h) * d;
            const float *kb = k + ((long)b * m * Hkv + hk) * d;
            const float *vb = v + ((long)b * m * Hkv + hk) * dv;
            double *w = w_rows ? w_rows + (long)r * m : NULL;
            if (w)
                for (int j = 0; j < m; ++j) w[j] = 0.0;
            attend_one_row(qi, kb, (long)Hkv * d, vb, (long)Hkv * dv, m_vis, d, dv,
                           scale, o_rows + (long)r * dv, lse_rows + r, w, scores);
        }
        free(scores);
    }
    return 0;
}

/*
 * Dense attention, every row.  o [B][n][H][dv], lse [B][H][n].
 */
int oracle_attention_f64(const float *q, const float *k, const float *v,
                         int B, int H, int Hkv, int n, int m, int d, int dv,
                         double scale, int causal, double *o, double *lse)
{
    if (!check_heads(H, Hkv) || B < 0 || n < 0 || m < 0 || d <= 0 || dv <= 0)
        return -1;
    const int group = H / Hkv;
    const long total = (long)B * H * n;
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)(m > 0 ? m : 1));
#pragma omp for schedule(dynamic, 16)
        for (long t = 0; t < total; ++t) {
            int i = (int)(t % n);
            int h = (int)((t / n) % H);
            int b = (int)(t / ((long)n * H));
            int hk = h / group;
            int m_vis = visible_keys(i, n, m, causal);
            const float *qi = q + (((long)b * n + i) * H + h) * d;
            const float *kb = k + ((long)b * m * Hkv + hk) * d;
            const float *vb = v + ((long)b * m * Hkv + hk) * dv;
            attend_one_row(qi, kb, (long)Hkv * d, vb, (long)Hkv * dv, m_vis, d, dv, scale,
                           o + (((long)b * n + i) * H + h) * dv,
                           lse + ((long)b * H + h) * n + i, NULL, scores);
        }
        free(scores);
    }
    return 0;
}

/*
 * Variable-length (packed) attention.  Sequence s owns query tokens
 * [cu_q[s], cu_q[s+1]) and key tokens [cu_k[s], cu_k[s+1]).
 * q [Tq][H][d], k [Tk][Hkv][d], v [Tk][Hkv][dv]; o [Tq][H][dv]; lse [H][Tq].
 * Causal: local key j visible to local query i iff j <= i + (m_s - n_s).
 */
int oracle_varlen_f64(const float *q, const float *k, const float *v,
                      const int *cu_q, const int *cu_k, int num_seqs, int H,
                      int Hkv, int d, int dv, double scale, int causal,
                      double *o, double *lse)
{
    if (!check_heads(H, Hkv) || num_seqs < 0 || d <= 0 || dv <= 0) return -1;
    for (int s = 0; s < num_seqs; ++s)
        if (cu_q[s + 1] < cu_q[s] || cu_k[s + 1] < cu_k[s]) return -1;
    const int group = H / Hkv;
    const int Tq = num_seqs > 0 ? cu_q[num_seqs] : 0;
    int max_m = 1;
    for (int s = 0; s < num_seqs; ++s)
        if (cu_k[s + 1] - cu_k[s] > max_m) max_m = cu_k[s + 1] - cu_k[s];
    const long total = (long)Tq * H;
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)max_m);
#pragma omp for schedule(dynamic, 16)
        for (long t = 0; t < total; ++t) {
            int tok = (int)(t / H), h = (int)(t % H);
            int s = 0;
            while (cu_q[s + 1] <= tok) ++s; /* sequence owning this token */
            int i = tok - cu_q[s];
            int m = cu_k[s + 1] - cu_k[s];
            int m_vis = visible_keys(i, cu_q[s + 1] - cu_q[s], m, causal);
            int hk = h / group;
            const float *qi = q + ((long)tok * H + h) * d;
            const float *kb = k + ((long)cu_k[s] * Hkv + hk) * d;
            const float *vb = v + ((long)cu_k[s] * Hkv + hk) * dv;
            attend_one_row(qi, kb, (long)Hkv * d, vb, (long)Hkv * dv, m_vis, d, dv, scale,
                           o + ((long)tok * H + h) * dv, lse + (long)h * Tq + tok, NULL,
                           scores);
        }
        free(scores);
    }
    return 0;
}

/*
 * Paged decode ([p2] 实现): one query token per sequence.  For sequence s the
 * keys are gathered page by page through block_table[s][*]: logical page p
 * holds min(page_size, seq_len - p*page_size) valid tokens, and the walk stops
 * at the first page with none.  Cache layout [num_pages][Hkv][page_size][d]
 * (and dv for V).  q [S][H][d]; o [S][H][dv]; lse [S][H].
 * Returns 0, -1 on invalid arguments, -2 on a block-table id out of range.
 */
int oracle_paged_decode_f64(const float *q, const float *k_cache, const float *v_cache,
                            const int *block_table, const int *seq_lens, int num_seqs,
                            int H, int Hkv, int d, int dv, int page_size, int num_pages,
                            int max_blocks, double scale, double *o, double *lse)
{
    if (!check_heads(H, Hkv) || num_seqs < 0 || d <= 0 || dv <= 0 || page_size <= 0)
        return -1;
    for (int s = 0; s < num_seqs; ++s) {
        if (seq_lens[s] < 0 || seq_lens[s] > max_blocks * page_size) return -1;
        int pages = (seq_lens[s] + page_size - 1) / page_size;
        for (int p = 0; p < pages; ++p) {
            int phys = block_table[(long)s * max_blocks + p];
            if (phys < 0 || phys >= num_pages) return -2;
        }
    }
    const int group = H / Hkv;
    const long total = (long)num_seqs * H;
    int ok = 0;
#pragma omp parallel reduction(| : ok)
    {
        int cap = max_blocks * page_size > 0 ? max_blocks * page_size : 1;
        float *kg = (float *)malloc(sizeof(float) * (size_t)cap * d);
        float *vg = (float *)malloc(sizeof(float) * (size_t)cap * dv);
        double *scores = (double *)malloc(sizeof(double) * (size_t)cap);
        if (!kg || !vg || !scores) ok |= 1;
#pragma omp for schedule(dynamic, 4)
        for (long t = 0; t < total; ++t) {
            if (!kg || !vg || !scores) continue;
            int s = (int)(t / H), h = (int)(t % H);
            int hk = h / group;
            /* gather this sequence's keys and values for kv head hk */
            int count = 0;
            for (int logical = 0; logical < max_blocks; ++logical) {
                int nvalid = seq_lens[s] - logical * page_size;
                if (nvalid > page_size) nvalid = page_size;
                if (nvalid <= 0) break;
                int phys = block_table[(long)s * max_blocks + logical];
                const float *kp = k_cache + (((long)phys * Hkv + hk) * page_size) * d;
                const float *vp = v_cache + (((long)phys * Hkv + hk) * page_size) * dv;
                for (int r = 0; r < nvalid; ++r) {
                    memcpy(kg + (long)count * d, kp + (long)r * d, sizeof(float) * d);
                    memcpy(vg + (long)count * dv, vp + (long)r * dv, sizeof(float) * dv);
                    ++count;
                }
            }
            attend_one_row(q + ((long)s * H + h) * d, kg, d, vg, dv, count, d, dv, scale,
                           o + ((long)s * H + h) * dv, lse + (long)s * H + h, NULL, scores);
        }
        free(kg);
        free(vg);
        free(scores);
    }
    return ok ? -1 : 0;
}

/*
 * Paged prefill: several new query tokens per sequence against the sequence's
 * paged keys ([p2] 它还解锁了什么: the tiles the recurrence walks need not be
 * contiguous, each may come through the block table).  Sequence s owns query
 * tokens [cu_q[s], cu_q[s+1]) (n_s of them) and seq_lens[s] keys gathered page
 * by page as in oracle_paged_decode_f64.  Causal: the queries are the last n_s
 * of the seq_lens[s] positions, so query i sees keys j <= i + (seq_lens[s] - n_s).
 * q [Tq][H][d]; o [Tq][H][dv]; lse [H][Tq].
 * Returns 0, -1 on invalid arguments, -2 on a block-table id out of range.
 */
int oracle_paged_prefill_f64(const float *q, const int *cu_q, const float *k_cache,
                             const float *v_cache, const int *block_table, const int *seq_lens,
                             int num_seqs, int H, int Hkv, int d, int dv, int page_size,
                             int num_pages, int max_blocks, double scale, int causal,
                             double *o, double *lse)
{
    if (!check_heads(H, Hkv) || num_seqs < 0 || d <= 0 || dv <= 0 || page_size <= 0)
        return -1;
    for (int s = 0; s < num_seqs; ++s) {
        if (cu_q[s + 1] < cu_q[s]) return -1;
        if (seq_lens[s] < 0 || seq_lens[s] > max_blocks * page_size) return -1;
        int pages = (seq_lens[s] + page_size - 1) / page_size;
        for (int p = 0; p < pages; ++p) {
            int phys = block_table[(long)s * max_blocks + p];
            if (phys < 0 || phys >= num_pages) return -2;
        }
    }
    const int group = H / Hkv;
    const int Tq = num_seqs > 0 ? cu_q[num_seqs] : 0;
    const long total = (long)num_seqs * Hkv;
    int ok = 0;
#pragma omp parallel reduction(| : ok)
    {
        int cap = max_blocks * page_size > 0 ? max_blocks * page_size : 1;
        float *kg = (float *)malloc(sizeof(float) * (size_t)cap * d);
        float *vg = (float *)malloc(sizeof(float) * (size_t)cap * dv);
        double *scores = (double *)malloc(sizeof(double) * (size_t)cap);
        if (!kg || !vg || !scores) ok |= 1;
#pragma omp for schedule(dynamic, 1)
        for (long t = 0; t < total; ++t) {
            if (!kg || !vg || !scores) continue;
            int s = (int)(t / Hkv), hk = (int)(t % Hkv);
            /* gather this sequence's keys and values for kv head hk */
            int count = 0;
            for (int logical = 0; logical < max_blocks; ++logical) {
                int nvalid = seq_lens[s] - logical * page_size;
                if (nvalid > page_size) nvalid = page_size;
                if (nvalid <= 0) break;
                int phys = block_table[(long)s * max_blocks + logical];
                const float *kp = k_cache + (((long)phys * Hkv + hk) * page_size) * d;
                const float *vp = v_cache + (((long)phys * Hkv + hk) * page_size) * dv;
                for (int r = 0; r < nvalid; ++r) {
                    memcpy(kg + (long)count * d, kp + (long)r * d, sizeof(float) * d);
                    memcpy(vg + (long)count * dv, vp + (long)r * dv, sizeof(float) * dv);
                    ++count;
                }
            }
            const int n = cu_q[s + 1] - cu_q[s];
            for (int h = hk * group; h < (hk + 1) * group; ++h)
                for (int i = 0; i < n; ++i) {
                    int tok = cu_q[s] + i;
                    attend_one_row(q + ((long)tok * H + h) * d, kg, d, vg, dv,
                                   visible_keys(i, n, count, causal), d, dv, scale,
                                   o + ((long)tok * H + h) * dv, lse + (long)h * Tq + tok, NULL,
                                   scores);
                }
        }
        free(kg);
        free(vg);
        free(scores);
    }
    return ok ? -1 : 0;
}

/*
 * Flash-decoding partials ([p2] 它还解锁了什么, 练习 1): the keys of each
 * sequence are cut into num_splits page-aligned ranges; split x covers logical
 * pages [ceil(x*P/X), ceil((x+1)*P/X)) of the sequence's P pages.  For each
 * split the unnormalised triple is
 *   m = max_j s_j,  l = sum_j exp(s_j - m),  o = sum_j exp(s_j - m) V[j],
 * and an empty split is (-inf, 0, 0).
 * part_m, part_l [S][H][X]; part_o [S][H][X][dv].
 */
int oracle_decode_partials_f64(const float *q, const float *k_cache, const float *v_cache,
                               const int *block_table, const int *seq_lens, int num_seqs,
                               int H, int Hkv, int d, int dv, int page_size, int num_pages,
                               int max_blocks, int num_splits, double scale,
                               double *part_m, double *part_l, double *part_o)
{
    if (!check_heads(H, Hkv) || num_seqs < 0 || d <= 0 || dv <= 0 || page_size <= 0 ||
        num_splits <= 0)
        return -1;
    for (int s = 0; s < num_seqs; ++s) {
        if (seq_lens[s] < 0 || seq_lens[s] > max_blocks * page_size) return -1;
        int pages = (seq_lens[s] + page_size - 1) / page_size;
        for (int p = 0; p < pages; ++p) {
            int phys = block_table[(long)s * max_blocks + p];
            if (phys < 0 || phys >= num_pages) return -2;
        }
    }
    const int group = H / Hkv;
    const long total = (long)num_seqs * H * num_splits;
#pragma omp parallel for schedule(dynamic, 8)
    for (long t = 0; t < total; ++t) {
        int x = (int)(t % num_splits);
        int h = (int)((t / num_splits) % H);
        int s = (int)(t / ((long)num_splits * H));
        int hk = h / group;
        int P = (seq_lens[s] + page_size - 1) / page_size;
        int p_begin = (int)(((long)x * P + num_splits - 1) / num_splits);
        int p_end = (int)(((long)(x + 1) * P + num_splits - 1) / num_splits);
        const float *qv = q + ((long)s * H + h) * d;
        double *om = part_m + t, *ol = part_l + t, *oo = part_o + t * dv;
        /* max over the split's visible keys */
        double M = -INFINITY;
        for (int p = p_begin; p < p_end; ++p) {
            int phys = block_table[(long)s * max_blocks + p];
            int nvalid = seq_lens[s] - p * page_size;
            if (nvalid > page_size) nvalid = page_size;
            for (int r = 0; r < nvalid; ++r) {
                const float *kr = k_cache + ((((long)phys * Hkv + hk) * page_size) + r) * d;
                double dot = 0.0;
                for (int c = 0; c < d; ++c) dot += (double)qv[c] * (double)kr[c];
                if (scale * dot > M) M = scale * dot;
            }
        }
        for (int c = 0; c < dv; ++c) oo[c] = 0.0;
        double l = 0.0;
        if (M != -INFINITY) {
            for (int p = p_begin; p < p_end; ++p) {
                int phys = block_table[(long)s * max_blocks + p];
                int nvalid = seq_lens[s] - p * page_size;
                if (nvalid > page_size) nvalid = page_size;
                for (int r = 0; r < nvalid; ++r) {
                    const float *kr = k_cache + ((((long)phys * Hkv + hk) * page_size) + r) * d;
                    const float *vr = v_cache + ((((long)phys * Hkv + hk) * page_size) + r) * dv;
                    double dot = 0.0;
                    for (int c = 0; c < d; ++c) dot += (double)qv[c] * (double)kr[c];
                    double w = exp(scale * dot - M);
                    l += w;
                    for (int c = 0; c < dv; ++c) oo[c] += w * (double)vr[c];
                }
            }
        }
        *om = M;
        *ol = l;
    }
    return 0;
}

/*
 * Merge of (m, l, o) triples ([p2] 练习 1: the merge rule is the same rescale
 * as the recurrence).  For each (s, h):
 *   M = max_x m_x;  w_x = exp(m_x - M) (0 when m_x = -inf);
 *   l = sum_x w_x l_x;  O = sum_x w_x o_x / l;  LSE = M + ln l.
 * A pair with no key at all (every m_x = -inf) gets O = 0, LSE = -inf.
 * part_m, part_l [S][H][X]; part_o [S][H][X][dv]; o [S][H][dv]; lse [S][H].
 */
int oracle_split_combine_f64(const double *part_m, const double *part_l,
                             const double *part_o, int num_seqs, int H, int num_splits,
                             int dv, double *o, double *lse)
{
    if (num_seqs < 0 || H <= 0 || num_splits <= 0 || dv <= 0) return -1;
    const long pairs = (long)num_seqs * H;
#pragma omp parallel for schedule(static)
    for (long t = 0; t < pairs; ++t) {
        const double *pm = part_m + t * num_splits;
        const double *pl = part_l + t * num_splits;
        const double *po = part_o + t * num_splits * dv;
        double M = -INFINITY;
        for (int x = 0; x < num_splits; ++x)
            if (pm[x] > M) M = pm[x];
        double *ot = o + t * dv;
        for (int c = 0; c < dv; ++c) ot[c] = 0.0;
        if (M == -INFINITY) {
            lse[t] = -INFINITY;
            continue;
        }
        double l = 0.0;
        for (int x = 0; x < num_splits; ++x) {
            double w = pm[x] == -INFINITY ? 0.0 : exp(pm[x] - M);
            l += w * pl[x];
            for (int c = 0; c < dv; ++c) ot[c] += w * po[(long)x * dv + c];
        }
        if (l > 0.0) {
            for (int c = 0; c < dv; ++c) ot[c] /= l;
            lse[t] = M + log(l);
        } else {
            for (int c = 0; c < dv; ++c) ot[c] = 0.0;
            lse[t] = -INFINITY;
        }
    }
    return 0;
}

/*
 * The online-softmax recurrence itself ([p1] §7 version 4, [p2] 解法, [p3]
 * 实现代码), single head, in double: Q rows are processed in blocks of
 * q_block rows ([p3] outer loop); for each Q block the K/V rows are visited
 * in blocks of kv_block rows, in the order given by kv_order (a permutation of
 * the kv block indices; NULL means 0, 1, 2, ...).  Per row and per kv block:
 *   m_new = max(m, max_j s_j)       (over the block's visible keys)
 *   ref   = m_new, or 0 when m_new = -inf (fully masked so far: the guard)
 *   alpha = exp(m - ref), taken as 1 while m = -inf (empty state)
 *   p_j   = exp(s_j - ref)          (0 for masked keys)
 *   l     = alpha*l + sum_j p_j
 *   acc   = alpha*acc + sum_j p_j V[j]
 *   m     = m_new
 * and finally O = acc / l (O = 0, LSE = -inf when l = 0), LSE = m + ln l.
 * q [n][d], k [m][d], v [m][dv]; o [n][dv]; lse [n].
 */
int oracle_online_recurrence_f64(const float *q, const float *k, const float *v, int n,
                                 int m, int d, int dv, double scale, int causal,
                                 int q_block, int kv_block, const int *kv_order,
                                 double *o, double *lse)
{
    if (n < 0 || m < 0 || d <= 0 || dv <= 0 || q_block <= 0 || kv_block <= 0) return -1;
    const int nkv = (m + kv_block - 1) / kv_block;
    if (kv_order) {
        /* must be a permutation of 0..nkv-1 */
        char *seen = (char *)calloc((size_t)(nkv > 0 ? nkv : 1), 1);
        for (int t = 0; t < nkv; ++t) {
            int b = kv_order[t];
            if (b < 0 || b >= nkv || seen[b]) {
                free(seen);
                return -1;
            }
            seen[b] = 1;
        }
        free(seen);
    }
    double *m_run = (double *)malloc(sizeof(double) * (size_t)(q_block > 0 ? q_block : 1));
    double *l_run = (double *)malloc(sizeof(double) * (size_t)q_block);
    double *acc = (double *)malloc(sizeof(double) * (size_t)q_block * dv);
    double *s = (double *)malloc(sizeof(double) * (size_t)kv_block);
    for (int i0 = 0; i0 < n; i0 += q_block) {
        int rows = n - i0 < q_block ? n - i0 : q_block;
        for (int r = 0; r < rows; ++r) {
            m_run[r] = -INFINITY;
            l_run[r] = 0.0;
            for (int c = 0; c < dv; ++c) acc[(long)r * dv + c] = 0.0;
        }
        for (int t = 0; t < nkv; ++t) {
            int blk = kv_order ? kv_order[t] : t;
            int j0 = blk * kv_block;
            int cols = m - j0 < kv_block ? m - j0 : kv_block;
            for (int r = 0; r < rows; ++r) {
                int i = i0 + r;
                double m_blk = -INFINITY;
                for (int c = 0; c < cols; ++c) {
                    int j = j0 + c;
                    if (causal && (long)j > (long)i + ((long)m - (long)n)) {
                        s[c] = -INFINITY;
                        continue;
                    }
                    double dot = 0.0;
                    for (int e = 0; e < d; ++e)
                        dot += (double)q[(long)i * d + e] * (double)k[(long)j * d + e];
                    s[c] = scale * dot;
                    if (s[c] > m_blk) m_blk = s[c];
                }
                double m_new = m_run[r] > m_blk ? m_run[r] : m_blk;
                double ref = m_new == -INFINITY ? 0.0 : m_new;
                double alpha = m_run[r] == -INFINITY ? 1.0 : exp(m_run[r] - ref);
                double psum = 0.0;
                double *a = acc + (long)r * dv;
                for (int c = 0; c < dv; ++c) a[c] *= alpha;
                for (int c = 0; c < cols; ++c) {
                    double p = s[c] == -INFINITY ? 0.0 : exp(s[c] - ref);
                    psum += p;
                    if (p != 0.0)
                        for (int e = 0; e < dv; ++e)
                            a[e] += p * (double)v[(long)(j0 + c) * dv + e];
                }
                l_run[r] = alpha * l_run[r] + psum;
                m_run[r] = m_new;
            }
        }
        for (int r = 0; r < rows; ++r) {
            int i = i0 + r;
            if (l_run[r] > 0.0) {
                for (int c = 0; c < dv; ++c) o[(long)i * dv + c] = acc[(long)r * dv + c] / l_run[r];
                lse[i] = m_run[r] + log(l_run[r]);
            } else {
                for (int c = 0; c < dv; ++c) o[(long)i * dv + c] = 0.0;
                lse[i] = -INFINITY;
            }
        }
    }
    free(m_run);
    free(l_run);
    free(acc);
    free(s);
    return 0;
}

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads the following calls use (for timing the oracle on one core and on
 * all of them); returns the previous count.  The results do not depend on it:
 * every row is computed by one thread in the same order. */
int oracle_set_num_threads(int n)
{
    const int prev = oracle_num_threads();
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#endif
    return prev;
}
