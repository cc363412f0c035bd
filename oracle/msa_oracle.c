/*
 * Plain fp64 CPU oracle for window + landmark sparse attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness authority that the
 * CUDA library is checked against.  It shares no code, header, table or
 * helper with the CUDA path, and nothing in the product path may load it:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg do.
 *
 * What it computes (the method of "Scaling GPU Cluster for Million Token
 * Context", section "Why Sparse Attention Changes the Game" and "What is
 * Flash-MSA Sparse Attention in GPU Clusters?": a local window of w tokens
 * plus a set of landmark tokens that summarise distant context, one fused
 * pass; and the online-softmax partial/merge step of "Training at 1M+ Token
 * Context: Ring Attention, YaRN, NTK-Aware Scaling", Ring Attention
 * paragraph).  The pages leave the exact definition open; the reading taken
 * is:
 *   - row i (global position) attends keys j with i-w < j <= i (causal
 *     window of w keys including itself);
 *   - landmark l is the mean of K (and of V) over the contiguous block of
 *     B = n/G tokens [lB, (l+1)B), and row i attends landmark l only when
 *     that block lies wholly before its window: (l+1)B <= i-w+1;
 *   - one softmax over the union of both sets, scores scale*<q,k>, no extra
 *     bias for landmarks; query head h reads KV head h / (Hq/Hkv);
 *   - outputs: O[i,h,:] and lse[h,i] = natural log of the softmax
 *     denominator (max-shifted), i.e. m + ln(sum exp(s-m)).
 *   - a "partial" restricts the window keys to one contiguous KV chunk and
 *     uses no landmarks; a row with no key gets lse = -inf and O = 0;
 *   - the merge of partials is lse = ln sum_p exp(lse_p) and
 *     O = sum_p exp(lse_p - lse) O_p over the parts with finite lse_p.
 *
 * Every score, exponential and sum is computed in double precision, two
 * passes per row (maximum first, then the sums).  Inputs are read in the
 * precision they are stored in (fp32, or bf16 bit patterns), which every
 * double represents exactly.
 *
 * Pins (see the tests): dense brute force on tiny inputs, reduction to exact
 * causal attention when w >= n and G = 0, merge-of-chunks equals single pass,
 * convexity of every output row, and closed forms (K = 0 gives uniform
 * weights and lse = ln |attended set|; V = c gives O = c; K = position gives
 * exact block means).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* Element idx of a buffer stored as fp32 or as bf16 bit patterns. */
static double oracle_load(const void *base, int64_t idx, int dtype) {
    if (dtype == ORACLE_F32) return (double)((const float *)base)[idx];
    uint16_t h = ((const uint16_t *)base)[idx];
    uint32_t w = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Landmark pooling: out[l][h][c] = (1/B) * sum_{j=lB}^{(l+1)B-1} x[j][h][c],
 * B = n / G.  x is [n][H][d] (fp32 or bf16), out is [G][H][d] fp64.
 * Returns 0, or -1 when G does not divide n.
 */
int oracle_landmark_pool(const void *x, int dtype, int64_t n, int H, int d,
                         int G, double *out) {
    if (G <= 0 || n <= 0 || n % G != 0) return -1;
    int64_t B = n / G;
    int64_t row = (int64_t)H * d;
#pragma omp parallel for schedule(static)
    for (int64_t l = 0; l < G; ++l) {
        for (int64_t e = 0; e < row; ++e) {
            double s = 0.0;
            for (int64_t j = l * B; j < (l + 1) * B; ++j)
                s += oracle_load(x, j * row + e, dtype);
            out[l * row + e] = s / (double)B;
        }
    }
    return 0;
}

/* Number of landmarks whose whole block lies before row pos's window. */
static int64_t oracle_visible_landmarks(int64_t pos, int64_t window,
                                        int64_t B, int G) {
    int64_t count = 0;
    for (int64_t l = 0; l < G; ++l) {
        if ((l + 1) * B <= pos - window + 1) count = l + 1;
        else break;
    }
    return count;
}

/*
 * Attention rows.
 *   q      [n_rows][Hq][d]   the query rows to evaluate (gathered)
 *   pos    [n_rows]          global position of each of those rows
 *   k, v   [n_kv][Hkv][d]    keys/values of global positions kv_start..
 *   k_lm, v_lm [G][Hkv][d]   fp64 landmarks (NULL when G == 0); landmark
 *                            block size B
 *   out    [n_rows][Hq][d]   fp64
 *   lse    [Hq][n_rows]      fp64, natural log; -inf for an empty set
 * Returns 0, or -1 on inconsistent arguments.
 */
int oracle_attn_rows(const void *q, const int64_t *pos, int64_t n_rows,
                     const void *k, const void *v, int64_t n_kv,
                     int64_t kv_start, int dtype, int Hq, int Hkv, int d,
                     int64_t window, const double *k_lm, const double *v_lm,
                     int G, int64_t B, double scale, double *out,
                     double *lse) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || window < 1)
        return -1;
    if (G < 0 || (G > 0 && (k_lm == NULL || v_lm == NULL || B < 1)))
        return -1;
    const int group = Hq / Hkv;
#pragma omp parallel
    {
        double *s_win = NULL, *s_lm = NULL;
        int64_t cap_win = 0;
        s_lm = (double *)malloc(sizeof(double) * (size_t)(G > 0 ? G : 1));
#pragma omp for collapse(2) schedule(dynamic, 4)
        for (int64_t r = 0; r < n_rows; ++r) {
            for (int h = 0; h < Hq; ++h) {
                const int64_t i = pos[r];
                const int c = h / group;
                /* Window keys: i-w < j <= i, intersected with the chunk. */
                int64_t j_lo = i - window + 1;
                if (j_lo < kv_start) j_lo = kv_start;
                int64_t j_hi = i;
                if (j_hi > kv_start + n_kv - 1) j_hi = kv_start + n_kv - 1;
                int64_t n_win = j_hi >= j_lo ? j_hi - j_lo + 1 : 0;
                int64_t n_lm = G > 0 ? oracle_visible_landmarks(i, window, B, G) : 0;
                if (n_win > cap_win) {
                    free(s_win);
                    cap_win = n_win;
                    s_win = (double *)malloc(sizeof(double) * (size_t)cap_win);
                }
                double *o = out + (r * Hq + h) * (int64_t)d;
                if (n_win + n_lm == 0) {
                    for (int e = 0; e < d; ++e) o[e] = 0.0;
                    lse[(int64_t)h * n_rows + r] = -INFINITY;
                    continue;
                }
                const int64_t qoff = (r * Hq + h) * (int64_t)d;
                /* Pass 1: scores and their maximum. */
                double m = -INFINITY;
                for (int64_t t = 0; t < n_win; ++t) {
                    int64_t koff = ((j_lo + t - kv_start) * Hkv + c) * (int64_t)d;
                    double dot = 0.0;
                    for (int e = 0; e < d; ++e)
                        dot += oracle_load(q, qoff + e, dtype) *
                               oracle_load(k, koff + e, dtype);
                    s_win[t] = scale * dot;
                    if (s_win[t] > m) m = s_win[t];
                }
                for (int64_t l = 0; l < n_lm; ++l) {
                    const double *kl = k_lm + (l * Hkv + c) * (int64_t)d;
                    double dot = 0.0;
                    for (int e = 0; e < d; ++e)
                        dot += oracle_load(q, qoff + e, dtype) * kl[e];
                    s_lm[l] = scale * dot;
                    if (s_lm[l] > m) m = s_lm[l];
                }
                /* Pass 2: denominator and weighted sum of values. */
                double denom = 0.0;
                for (int e = 0; e < d; ++e) o[e] = 0.0;
                for (int64_t t = 0; t < n_win; ++t) {
                    double p = exp(s_win[t] - m);
                    denom += p;
                    int64_t voff = ((j_lo + t - kv_start) * Hkv + c) * (int64_t)d;
                    for (int e = 0; e < d; ++e)
                        o[e] += p * oracle_load(v, voff + e, dtype);
                }
                for (int64_t l = 0; l < n_lm; ++l) {
                    double p = exp(s_lm[l] - m);
                    denom += p;
                    const double *vl = v_lm + (l * Hkv + c) * (int64_t)d;
                    for (int e = 0; e < d; ++e) o[e] += p * vl[e];
                }
                for (int e = 0; e < d; ++e) o[e] /= denom;
                lse[(int64_t)h * n_rows + r] = m + log(denom);
            }
        }
        free(s_win);
        free(s_lm);
    }
    return 0;
}

/*
 * Merge of P partial results over disjoint key sets.
 *   o_parts   [P][n_rows][Hq][d] fp64, lse_parts [P][Hq][n_rows] fp64
 *   out       [n_rows][Hq][d],          lse       [Hq][n_rows]
 * A part with lse_p = -inf holds no key for that row and is skipped; when
 * every part is -inf the row's lse is -inf and its O is 0.
 */
int oracle_lse_merge(const double *o_parts, const double *lse_parts, int P,
                     int64_t n_rows, int Hq, int d, double *out,
                     double *lse) {
    if (P < 1 || n_rows < 0 || Hq < 1 || d < 1) return -1;
    const int64_t part_o = n_rows * Hq * (int64_t)d;
    const int64_t part_l = (int64_t)Hq * n_rows;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
        for (int h = 0; h < Hq; ++h) {
            const int64_t li = (int64_t)h * n_rows + r;
            const int64_t oi = (r * Hq + h) * (int64_t)d;
            double mx = -INFINITY;
            for (int p = 0; p < P; ++p) {
                double l = lse_parts[p * part_l + li];
                if (l > mx) mx = l;
            }
            double *o = out + oi;
            for (int e = 0; e < d; ++e) o[e] = 0.0;
            if (mx == -INFINITY) {
                lse[li] = -INFINITY;
                continue;
            }
            double sum = 0.0;
            for (int p = 0; p < P; ++p) {
                double l = lse_parts[p * part_l + li];
                if (l == -INFINITY) continue;
                sum += exp(l - mx);
            }
            const double total = mx + log(sum);
            for (int p = 0; p < P; ++p) {
                double l = lse_parts[p * part_l + li];
                if (l == -INFINITY) continue;
                const double wgt = exp(l - total);
                const double *op = o_parts + p * part_o + oi;
                for (int e = 0; e < d; ++e) o[e] += wgt * op[e];
            }
            lse[li] = total;
        }
    }
    return 0;
}

/*
 * Block-band attention (the 2-D block-sparse mask of "Million Token Context
 * Window Optimization: What Actually Works", section "The indexing game:
 * smarter context management": each 128-token block attends to 16 other
 * blocks, left and right).  Reading taken: with
 * block size bb and half-width hw, row i attends every key j of the blocks
 * within hw of its own, |floor(j/bb) - floor(i/bb)| <= hw, 0 <= j < n_kv (not
 * causal); one softmax, scores scale*<q,k>.
 *   q [n_rows][Hq][d] at positions pos[]; k, v [n_kv][Hkv][d]
 *   out [n_rows][Hq][d], lse [Hq][n_rows] (fp64)
 */
int oracle_attn_band_rows(const void *q, const int64_t *pos, int64_t n_rows,
                          const void *k, const void *v, int64_t n_kv,
                          int dtype, int Hq, int Hkv, int d, int64_t bb,
                          int64_t hw, double scale, double *out,
                          double *lse) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || bb < 1 || hw < 0)
        return -1;
    const int group = Hq / Hkv;
#pragma omp parallel
    {
        double *sc = NULL;
        int64_t cap = 0;
#pragma omp for collapse(2) schedule(dynamic, 4)
        for (int64_t r = 0; r < n_rows; ++r) {
            for (int h = 0; h < Hq; ++h) {
                const int64_t i = pos[r];
                const int c = h / group;
                const int64_t bi = i / bb;
                int64_t j_lo = (bi - hw) * bb;
                if (j_lo < 0) j_lo = 0;
                int64_t j_hi = (bi + hw + 1) * bb - 1;
                if (j_hi > n_kv - 1) j_hi = n_kv - 1;
                const int64_t nk = j_hi >= j_lo ? j_hi - j_lo + 1 : 0;
                double *o = out + (r * Hq + h) * (int64_t)d;
                if (nk == 0) {
                    for (int e = 0; e < d; ++e) o[e] = 0.0;
                    lse[(int64_t)h * n_rows + r] = -INFINITY;
                    continue;
                }
                if (nk > cap) {
                    free(sc);
                    cap = nk;
                    sc = (double *)malloc(sizeof(double) * (size_t)cap);
                }
                const int64_t qoff = (r * Hq + h) * (int64_t)d;
                double m = -INFINITY;
                for (int64_t t = 0; t < nk; ++t) {
                    const int64_t koff = ((j_lo + t) * Hkv + c) * (int64_t)d;
                    double dot = 0.0;
                    for (int e = 0; e < d; ++e)
                        dot += oracle_load(q, qoff + e, dtype) *
                               oracle_load(k, koff + e, dtype);
                    sc[t] = scale * dot;
                    if (sc[t] > m) m = sc[t];
                }
                double denom = 0.0;
                for (int e = 0; e < d; ++e) o[e] = 0.0;
                for (int64_t t = 0; t < nk; ++t) {
                    const double p = exp(sc[t] - m);
                    denom += p;
                    const int64_t voff = ((j_lo + t) * Hkv + c) * (int64_t)d;
                    for (int e = 0; e < d; ++e)
                        o[e] += p * oracle_load(v, voff + e, dtype);
                }
                for (int e = 0; e < d; ++e) o[e] /= denom;
                lse[(int64_t)h * n_rows + r] = m + log(denom);
            }
        }
        free(sc);
    }
    return 0;
}

/*
 * Landmark-scored block selection, standing in for the hierarchical context
 * index of "Million Token Context Window Optimization: What Actually Works",
 * section "The indexing game: smarter context management" (chunks of the
 * input are scored against the query and only the top-k chunks plus a
 * history window are attended; the pages score chunks with a BERT embedding,
 * which needs trained weights, so the chunk's landmark -- its mean key --
 * scores it here).  Reading taken: query blocks of q_block rows; for query
 * block t and KV group c the score of key block l (bs tokens) is
 *   sum over rows i of block t and heads h of group c of <q[i,h], Kbar[l,c]>,
 * defined only for blocks wholly before the window of the block's first row,
 * (l+1)*bs <= t*q_block - w + 1; other blocks score -inf.
 *   q [n][Hq][d]; k_lm [G][Hkv][d] fp64; scores [n_qb][Hkv][G] fp64,
 *   n_qb = ceil(n / q_block).
 */
int oracle_block_scores(const void *q, int dtype, int64_t n, int Hq, int Hkv,
                        int d, const double *k_lm, int G, int64_t bs,
                        int64_t window, int64_t q_block, double *scores) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || G < 1 || bs < 1 ||
        q_block < 1 || window < 1)
        return -1;
    const int group = Hq / Hkv;
    const int64_t n_qb = (n + q_block - 1) / q_block;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t t = 0; t < n_qb; ++t) {
        for (int c = 0; c < Hkv; ++c) {
            double *qsum = (double *)calloc((size_t)d, sizeof(double));
            const int64_t r_end = (t + 1) * q_block < n ? (t + 1) * q_block : n;
            for (int64_t i = t * q_block; i < r_end; ++i)
                for (int hh = 0; hh < group; ++hh) {
                    const int64_t off = (i * Hq + c * group + hh) * (int64_t)d;
                    for (int e = 0; e < d; ++e) qsum[e] += oracle_load(q, off + e, dtype);
                }
            double *row = scores + (t * Hkv + c) * (int64_t)G;
            for (int l = 0; l < G; ++l) {
                if ((l + 1) * bs <= t * q_block - window + 1) {
                    const double *kl = k_lm + ((int64_t)l * Hkv + c) * d;
                    double sc = 0.0;
                    for (int e = 0; e < d; ++e) sc += qsum[e] * kl[e];
                    row[l] = sc;
                } else {
                    row[l] = -INFINITY;
                }
            }
            free(qsum);
        }
    }
    return 0;
}

/*
 * Attention over the causal window plus the tokens of the selected blocks:
 * row i (query block t = i / q_block, KV group c) attends keys
 * i-w < j <= i and every token of the blocks sel[t][c][0..cnt[t][c]).
 * One softmax, scores scale*<q,k>.
 *   q [n_rows][Hq][d] at positions pos[]; k, v [n][Hkv][d];
 *   sel [n_qb][Hkv][topk] int32, cnt [n_qb][Hkv] int32;
 *   out [n_rows][Hq][d], lse [Hq][n_rows] fp64.
 */
int oracle_attn_select_rows(const void *q, const int64_t *pos, int64_t n_rows,
                            const void *k, const void *v, int64_t n, int dtype,
                            int Hq, int Hkv, int d, int64_t window,
                            int64_t bs, int64_t q_block, const int32_t *sel,
                            const int32_t *cnt, int topk, double scale,
                            double *out, double *lse) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || window < 1 ||
        bs < 1 || q_block < 1 || topk < 0)
        return -1;
    const int group = Hq / Hkv;
#pragma omp parallel
    {
        int64_t *keys = NULL;
        double *sc = NULL;
        int64_t cap = 0;
#pragma omp for collapse(2) schedule(dynamic, 4)
        for (int64_t r = 0; r < n_rows; ++r) {
            for (int h = 0; h < Hq; ++h) {
                const int64_t i = pos[r];
                const int c = h / group;
                const int64_t t = i / q_block;
                const int32_t ns = cnt[t * Hkv + c];
                const int32_t *bl = sel + (t * Hkv + c) * (int64_t)topk;
                int64_t j_lo = i - window + 1;
                if (j_lo < 0) j_lo = 0;
                const int64_t need = (i - j_lo + 1) + (int64_t)ns * bs;
                if (need > cap) {
                    free(keys);
                    free(sc);
                    cap = need;
                    keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)cap);
                    sc = (double *)malloc(sizeof(double) * (size_t)cap);
                }
                int64_t nk = 0;
                for (int32_t b = 0; b < ns; ++b)
                    for (int64_t j = (int64_t)bl[b] * bs; j < ((int64_t)bl[b] + 1) * bs; ++j)
                        keys[nk++] = j;
                for (int64_t j = j_lo; j <= i; ++j) keys[nk++] = j;
                const int64_t qoff = (r * Hq + h) * (int64_t)d;
                double m = -INFINITY;
                for (int64_t x = 0; x < nk; ++x) {
                    const int64_t koff = (keys[x] * Hkv + c) * (int64_t)d;
                    double dot = 0.0;
                    for (int e = 0; e < d; ++e)
                        dot += oracle_load(q, qoff + e, dtype) *
                               oracle_load(k, koff + e, dtype);
                    sc[x] = scale * dot;
                    if (sc[x] > m) m = sc[x];
                }
                double *o = out + (r * Hq + h) * (int64_t)d;
                double denom = 0.0;
                for (int e = 0; e < d; ++e) o[e] = 0.0;
                for (int64_t x = 0; x < nk; ++x) {
                    const double p = exp(sc[x] - m);
                    denom += p;
                    const int64_t voff = (keys[x] * Hkv + c) * (int64_t)d;
                    for (int e = 0; e < d; ++e)
                        o[e] += p * oracle_load(v, voff + e, dtype);
                }
                for (int e = 0; e < d; ++e) o[e] /= denom;
                lse[(int64_t)h * n_rows + r] = m + log(denom);
            }
        }
        free(keys);
        free(sc);
    }
    return 0;
}

/*
 * One (row i, head h) of the backward's first pass: the softmax over A(i),
 * O_i, lse_i, D_i = <dO_i, O_i> and dQ_i = scale sum_a P_ia (<dO_i, v_a> -
 * D_i) k_a.  sc and o are scratch of window + G and d doubles.
 */
static void oracle_bwd_row(const void *q, const void *k, const void *v,
                           const void *dout, int dtype, int64_t n, int64_t i,
                           int h, int Hq, int Hkv, int d, int64_t window, int G,
                           int64_t B, const double *k_lm, const double *v_lm,
                           double scale, double *sc, double *o, double *lse_out,
                           double *D_out, double *g) {
    (void)n;
    const int c = h / (Hq / Hkv);
    const int64_t j_lo = i - window + 1 > 0 ? i - window + 1 : 0;
    const int64_t n_win = i - j_lo + 1;
    const int64_t n_lm = G > 0 ? oracle_visible_landmarks(i, window, B, G) : 0;
    const int64_t qoff = (i * Hq + h) * (int64_t)d;
    double m = -INFINITY;
    for (int64_t a = 0; a < n_win + n_lm; ++a) {
        double dot = 0.0;
        for (int e = 0; e < d; ++e) {
            const double ke = a < n_win
                ? oracle_load(k, ((j_lo + a) * Hkv + c) * (int64_t)d + e, dtype)
                : k_lm[((a - n_win) * Hkv + c) * (int64_t)d + e];
            dot += oracle_load(q, qoff + e, dtype) * ke;
        }
        sc[a] = scale * dot;
        if (sc[a] > m) m = sc[a];
    }
    double denom = 0.0;
    for (int e = 0; e < d; ++e) o[e] = 0.0;
    for (int64_t a = 0; a < n_win + n_lm; ++a) {
        const double p = exp(sc[a] - m);
        denom += p;
        for (int e = 0; e < d; ++e)
            o[e] += p * (a < n_win
                ? oracle_load(v, ((j_lo + a) * Hkv + c) * (int64_t)d + e, dtype)
                : v_lm[((a - n_win) * Hkv + c) * (int64_t)d + e]);
    }
    const double L = m + log(denom);
    double Di = 0.0;
    for (int e = 0; e < d; ++e)
        Di += oracle_load(dout, qoff + e, dtype) * (o[e] / denom);
    *lse_out = L;
    *D_out = Di;
    for (int e = 0; e < d; ++e) g[e] = 0.0;
    for (int64_t a = 0; a < n_win + n_lm; ++a) {
        const double p = exp(sc[a] - L);
        double dp = 0.0;
        for (int e = 0; e < d; ++e)
            dp += oracle_load(dout, qoff + e, dtype) * (a < n_win
                ? oracle_load(v, ((j_lo + a) * Hkv + c) * (int64_t)d + e, dtype)
                : v_lm[((a - n_win) * Hkv + c) * (int64_t)d + e]);
        const double ds = p * (dp - Di);
        for (int e = 0; e < d; ++e)
            g[e] += scale * ds * (a < n_win
                ? oracle_load(k, ((j_lo + a) * Hkv + c) * (int64_t)d + e, dtype)
                : k_lm[((a - n_win) * Hkv + c) * (int64_t)d + e]);
    }
}

/*
 * Backward pass: the gradients of L = sum_{i,h} <dO[i,h], O[i,h]> with
 * respect to Q, K and V, for training with the sparse pattern (the
 * Block-Sparse Flash Attention paragraph of "Training at 1M+ Token
 * Context" trains with it).  With A(i) the attended set of row i (window
 * keys and visible landmarks), P the softmax over A(i) and a running over
 * A(i):
 *   D_i   = <dO_i, O_i> = sum_a P_ia <dO_i, v_a>
 *   dS_ia = P_ia (<dO_i, v_a> - D_i)
 *   dQ_i  = scale sum_a dS_ia k_a,  dk_a += scale dS_ia q_i,
 *   dv_a += P_ia dO_i;
 * a landmark is the mean of its B tokens, so its gradient reaches each of
 * them divided by B: dK[j] += dK_lm[l] / B for j in block l (same for V).
 *   q, dout [n][Hq][d]; k, v [n][Hkv][d] (fp32 or bf16 bits, one dtype)
 *   dq [n][Hq][d], dk, dv [n][Hkv][d]  fp64, written
 * Three passes, each free of write conflicts: rows (lse_i, D_i, dQ_i),
 * window keys (the rows i in [j, j+w-1] of each key j), landmarks (the
 * rows that see each landmark), then the scatter of landmark gradients.
 */
int oracle_attn_bwd(const void *q, const void *k, const void *v,
                    const void *dout, int dtype, int64_t n, int Hq, int Hkv,
                    int d, int64_t window, int G, double scale, double *dq,
                    double *dk, double *dv) {
    if (n < 1 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 ||
        window < 1 || G < 0 || (G > 0 && n % G != 0))
        return -1;
    const int group = Hq / Hkv;
    const int64_t B = G > 0 ? n / G : 1;
    const int64_t row_kv = (int64_t)Hkv * d;
    double *k_lm = NULL, *v_lm = NULL, *dk_lm = NULL, *dv_lm = NULL;
    if (G > 0) {
        k_lm = (double *)malloc(sizeof(double) * (size_t)(G * row_kv));
        v_lm = (double *)malloc(sizeof(double) * (size_t)(G * row_kv));
        dk_lm = (double *)calloc((size_t)(G * row_kv), sizeof(double));
        dv_lm = (double *)calloc((size_t)(G * row_kv), sizeof(double));
        oracle_landmark_pool(k, dtype, n, Hkv, d, G, k_lm);
        oracle_landmark_pool(v, dtype, n, Hkv, d, G, v_lm);
    }
    double *lse = (double *)malloc(sizeof(double) * (size_t)(n * Hq));
    double *Dv = (double *)malloc(sizeof(double) * (size_t)(n * Hq));

    /* Pass 1: per (row, head) the softmax, O, D and dQ. */
#pragma omp parallel
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)(window + G));
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for collapse(2) schedule(dynamic, 4)
        for (int64_t i = 0; i < n; ++i)
            for (int h = 0; h < Hq; ++h)
                oracle_bwd_row(q, k, v, dout, dtype, n, i, h, Hq, Hkv, d, window, G, B, k_lm,
                               v_lm, scale, sc, o, &lse[(int64_t)h * n + i],
                               &Dv[(int64_t)h * n + i], dq + (i * Hq + h) * (int64_t)d);
        free(sc);
        free(o);
    }

    /* Pass 2: window keys.  Key j is seen by rows i in [j, j+w-1]. */
#pragma omp parallel for collapse(2) schedule(dynamic, 16)
    for (int64_t j = 0; j < n; ++j) {
        for (int c = 0; c < Hkv; ++c) {
            double *gk = dk + (j * Hkv + c) * (int64_t)d;
            double *gv = dv + (j * Hkv + c) * (int64_t)d;
            for (int e = 0; e < d; ++e) gk[e] = gv[e] = 0.0;
            const int64_t koff = (j * Hkv + c) * (int64_t)d;
            const int64_t i_hi = j + window - 1 < n - 1 ? j + window - 1 : n - 1;
            for (int64_t i = j; i <= i_hi; ++i) {
                for (int h = c * group; h < (c + 1) * group; ++h) {
                    const int64_t qoff = (i * Hq + h) * (int64_t)d;
                    double s = 0.0, dp = 0.0;
                    for (int e = 0; e < d; ++e) {
                        s += oracle_load(q, qoff + e, dtype) * oracle_load(k, koff + e, dtype);
                        dp += oracle_load(dout, qoff + e, dtype) *
                              oracle_load(v, koff + e, dtype);
                    }
                    const double p = exp(scale * s - lse[(int64_t)h * n + i]);
                    const double ds = p * (dp - Dv[(int64_t)h * n + i]);
                    for (int e = 0; e < d; ++e) {
                        gk[e] += scale * ds * oracle_load(q, qoff + e, dtype);
                        gv[e] += p * oracle_load(dout, qoff + e, dtype);
                    }
                }
            }
        }
    }

    /* Pass 3: landmarks.  Landmark l is seen by rows with (l+1)B <= i-w+1. */
    if (G > 0) {
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
        for (int64_t l = 0; l < G; ++l) {
            for (int c = 0; c < Hkv; ++c) {
                const double *kl = k_lm + (l * Hkv + c) * (int64_t)d;
                const double *vl = v_lm + (l * Hkv + c) * (int64_t)d;
                double *gk = dk_lm + (l * Hkv + c) * (int64_t)d;
                double *gv = dv_lm + (l * Hkv + c) * (int64_t)d;
                for (int64_t i = (l + 1) * B + window - 1; i < n; ++i) {
                    for (int h = c * group; h < (c + 1) * group; ++h) {
                        const int64_t qoff = (i * Hq + h) * (int64_t)d;
                        double s = 0.0, dp = 0.0;
                        for (int e = 0; e < d; ++e) {
                            s += oracle_load(q, qoff + e, dtype) * kl[e];
                            dp += oracle_load(dout, qoff + e, dtype) * vl[e];
                        }
                        const double p = exp(scale * s - lse[(int64_t)h * n + i]);
                        const double ds = p * (dp - Dv[(int64_t)h * n + i]);
                        for (int e = 0; e < d; ++e) {
                            gk[e] += scale * ds * oracle_load(q, qoff + e, dtype);
                            gv[e] += p * oracle_load(dout, qoff + e, dtype);
                        }
                    }
                }
            }
        }
        /* Scatter: each token of block l receives 1/B of its landmark's
           gradient. */
#pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < n; ++j) {
            const int64_t l = j / B;
            for (int64_t e = 0; e < row_kv; ++e) {
                dk[j * row_kv + e] += dk_lm[l * row_kv + e] / (double)B;
                dv[j * row_kv + e] += dv_lm[l * row_kv + e] / (double)B;
            }
        }
    }
    free(lse);
    free(Dv);
    free(k_lm);
    free(v_lm);
    free(dk_lm);
    free(dv_lm);
    return 0;
}

/*
 * dQ of selected rows only (the first pass of oracle_attn_bwd on them):
 *   rows [n_rows] positions, dq [n_rows][Hq][d] fp64, written.
 */
int oracle_attn_bwd_dq_rows(const void *q, const void *k, const void *v,
                            const void *dout, int dtype, int64_t n, int Hq,
                            int Hkv, int d, int64_t window, int G, double scale,
                            const int64_t *rows, int64_t n_rows, double *dq) {
    if (n < 1 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 ||
        window < 1 || G < 0 || (G > 0 && n % G != 0))
        return -1;
    const int64_t B = G > 0 ? n / G : 1;
    const int64_t row_kv = (int64_t)Hkv * d;
    double *k_lm = NULL, *v_lm = NULL;
    if (G > 0) {
        k_lm = (double *)malloc(sizeof(double) * (size_t)(G * row_kv));
        v_lm = (double *)malloc(sizeof(double) * (size_t)(G * row_kv));
        oracle_landmark_pool(k, dtype, n, Hkv, d, G, k_lm);
        oracle_landmark_pool(v, dtype, n, Hkv, d, G, v_lm);
    }
#pragma omp parallel
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)(window + G));
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
        double L, Dd;
#pragma omp for collapse(2) schedule(dynamic, 4)
        for (int64_t r = 0; r < n_rows; ++r)
            for (int h = 0; h < Hq; ++h)
                oracle_bwd_row(q, k, v, dout, dtype, n, rows[r], h, Hq, Hkv, d, window, G, B,
                               k_lm, v_lm, scale, sc, o, &L, &Dd,
                               dq + (r * Hq + h) * (int64_t)d);
        free(sc);
        free(o);
    }
    free(k_lm);
    free(v_lm);
    return 0;
}

/*
 * lse_i and D_i = <dO_i, O_i> of one (row i, head h): the first pass of
 * oracle_attn_bwd without dQ.  sc is scratch of window + G doubles, o of d.
 */
static void oracle_row_stats(const void *q, const void *k, const void *v,
                             const void *dout, int dtype, int64_t i, int h,
                             int Hq, int Hkv, int d, int64_t window, int G,
                             int64_t B, const double *k_lm, const double *v_lm,
                             double scale, double *sc, double *o,
                             double *lse_out, double *D_out) {
    const int c = h / (Hq / Hkv);
    const int64_t j_lo = i - window + 1 > 0 ? i - window + 1 : 0;
    const int64_t n_win = i - j_lo + 1;
    const int64_t n_lm = G > 0 ? oracle_visible_landmarks(i, window, B, G) : 0;
    const int64_t qoff = (i * Hq + h) * (int64_t)d;
    double m = -INFINITY;
    for (int64_t a = 0; a < n_win + n_lm; ++a) {
        double dot = 0.0;
        for (int e = 0; e < d; ++e) {
            const double ke = a < n_win
                ? oracle_load(k, ((j_lo + a) * Hkv + c) * (int64_t)d + e, dtype)
                : k_lm[((a - n_win) * Hkv + c) * (int64_t)d + e];
            dot += oracle_load(q, qoff + e, dtype) * ke;
        }
        sc[a] = scale * dot;
        if (sc[a] > m) m = sc[a];
    }
    double denom = 0.0;
    for (int e = 0; e < d; ++e) o[e] = 0.0;
    for (int64_t a = 0; a < n_win + n_lm; ++a) {
        const double p = exp(sc[a] - m);
        denom += p;
        for (int e = 0; e < d; ++e)
            o[e] += p * (a < n_win
                ? oracle_load(v, ((j_lo + a) * Hkv + c) * (int64_t)d + e, dtype)
                : v_lm[((a - n_win) * Hkv + c) * (int64_t)d + e]);
    }
    double Di = 0.0;
    for (int e = 0; e < d; ++e)
        Di += oracle_load(dout, qoff + e, dtype) * (o[e] / denom);
    *lse_out = m + log(denom);
    *D_out = Di;
}

/*
 * dK and dV of listed (key position, KV head) pairs only: the second and
 * third passes of oracle_attn_bwd restricted to those keys, for checking
 * layers whose full backward is out of reach on the host.  For key j of KV
 * head c:
 *   window part:   sum over rows i in [j, j+w-1] and the group's heads h of
 *                  dk += scale dS_ij q_ih,  dv += P_ij dO_ih;
 *   landmark part: the gradient of landmark l = j / B (rows with
 *                  (l+1)B <= i-w+1), divided by B (a landmark is the mean of
 *                  its B tokens).
 * P and dS come from each row's lse and D, computed (first pass) only for
 * the rows and heads that see a listed key or its block's landmark.
 *   keys [n_keys] positions in [0, n), kv_heads [n_keys] in [0, Hkv)
 *   dk, dv [n_keys][d] fp64, written
 * Returns 0, or -1 on inconsistent arguments.
 */
int oracle_attn_bwd_dkdv_keys(const void *q, const void *k, const void *v,
                              const void *dout, int dtype, int64_t n, int Hq,
                              int Hkv, int d, int64_t window, int G,
                              double scale, const int64_t *keys,
                              const int32_t *kv_heads, int64_t n_keys,
                              double *dk, double *dv) {
    if (n < 1 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 ||
        window < 1 || G < 0 || (G > 0 && n % G != 0) || n_keys < 0)
        return -1;
    for (int64_t r = 0; r < n_keys; ++r)
        if (keys[r] < 0 || keys[r] >= n || kv_heads[r] < 0 || kv_heads[r] >= Hkv)
            return -1;
    const int group = Hq / Hkv;
    const int64_t B = G > 0 ? n / G : 1;
    const int64_t row_kv = (int64_t)Hkv * d;
    double *k_lm = NULL, *v_lm = NULL;
    if (G > 0) {
        k_lm = (double *)malloc(sizeof(double) * (size_t)(G * row_kv));
        v_lm = (double *)malloc(sizeof(double) * (size_t)(G * row_kv));
        oracle_landmark_pool(k, dtype, n, Hkv, d, G, k_lm);
        oracle_landmark_pool(v, dtype, n, Hkv, d, G, v_lm);
    }
    /* Which (row, KV group) pairs need their statistics. */
    char *need = (char *)calloc((size_t)(n * Hkv), 1);
    for (int64_t r = 0; r < n_keys; ++r) {
        const int64_t j = keys[r];
        const int c = kv_heads[r];
        const int64_t i_hi = j + window - 1 < n - 1 ? j + window - 1 : n - 1;
        for (int64_t i = j; i <= i_hi; ++i) need[i * Hkv + c] = 1;
        if (G > 0)
            for (int64_t i = (j / B + 1) * B + window - 1; i < n; ++i) need[i * Hkv + c] = 1;
    }
    double *lse = (double *)malloc(sizeof(double) * (size_t)(n * Hq));
    double *Dv = (double *)malloc(sizeof(double) * (size_t)(n * Hq));
#pragma omp parallel
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)(window + G));
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for collapse(2) schedule(dynamic, 16)
        for (int64_t i = 0; i < n; ++i)
            for (int c = 0; c < Hkv; ++c) {
                if (!need[i * Hkv + c]) continue;
                for (int h = c * group; h < (c + 1) * group; ++h)
                    oracle_row_stats(q, k, v, dout, dtype, i, h, Hq, Hkv, d, window, G, B,
                                     k_lm, v_lm, scale, sc, o, &lse[(int64_t)h * n + i],
                                     &Dv[(int64_t)h * n + i]);
            }
        free(sc);
        free(o);
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_keys; ++r) {
        const int64_t j = keys[r];
        const int c = kv_heads[r];
        double *gk = dk + r * (int64_t)d;
        double *gv = dv + r * (int64_t)d;
        for (int e = 0; e < d; ++e) gk[e] = gv[e] = 0.0;
        /* Window part: rows i in [j, j+w-1]. */
        const int64_t koff = (j * Hkv + c) * (int64_t)d;
        const int64_t i_hi = j + window - 1 < n - 1 ? j + window - 1 : n - 1;
        for (int64_t i = j; i <= i_hi; ++i) {
            for (int h = c * group; h < (c + 1) * group; ++h) {
                const int64_t qoff = (i * Hq + h) * (int64_t)d;
                double s = 0.0, dp = 0.0;
                for (int e = 0; e < d; ++e) {
                    s += oracle_load(q, qoff + e, dtype) * oracle_load(k, koff + e, dtype);
                    dp += oracle_load(dout, qoff + e, dtype) * oracle_load(v, koff + e, dtype);
                }
                const double p = exp(scale * s - lse[(int64_t)h * n + i]);
                const double ds = p * (dp - Dv[(int64_t)h * n + i]);
                for (int e = 0; e < d; ++e) {
                    gk[e] += scale * ds * oracle_load(q, qoff + e, dtype);
                    gv[e] += p * oracle_load(dout, qoff + e, dtype);
                }
            }
        }
        /* Landmark part: landmark l = j / B, seen by rows (l+1)B <= i-w+1. */
        if (G > 0) {
            const int64_t l = j / B;
            const double *kl = k_lm + (l * Hkv + c) * (int64_t)d;
            const double *vl = v_lm + (l * Hkv + c) * (int64_t)d;
            double *tk = (double *)calloc((size_t)d, sizeof(double));
            double *tv = (double *)calloc((size_t)d, sizeof(double));
            for (int64_t i = (l + 1) * B + window - 1; i < n; ++i) {
                for (int h = c * group; h < (c + 1) * group; ++h) {
                    const int64_t qoff = (i * Hq + h) * (int64_t)d;
                    double s = 0.0, dp = 0.0;
                    for (int e = 0; e < d; ++e) {
                        s += oracle_load(q, qoff + e, dtype) * kl[e];
                        dp += oracle_load(dout, qoff + e, dtype) * vl[e];
                    }
                    const double p = exp(scale * s - lse[(int64_t)h * n + i]);
                    const double ds = p * (dp - Dv[(int64_t)h * n + i]);
                    for (int e = 0; e < d; ++e) {
                        tk[e] += scale * ds * oracle_load(q, qoff + e, dtype);
                        tv[e] += p * oracle_load(dout, qoff + e, dtype);
                    }
                }
            }
            for (int e = 0; e < d; ++e) {
                gk[e] += tk[e] / (double)B;
                gv[e] += tv[e] / (double)B;
            }
            free(tk);
            free(tv);
        }
    }
    free(need);
    free(lse);
    free(Dv);
    free(k_lm);
    free(v_lm);
    return 0;
}
