/*
 * Float64 CPU oracle for FlashPrefill-style block-sparse causal prefill
 * attention.  TEST INFRASTRUCTURE ONLY: it is called by the tests, by the
 * smoke check and by the benchmark's CPU-baseline leg, never by the product
 * path.  It shares no code, header or table with the CUDA library.
 *
 * Sources (web pages on the method):
 *   [V1]  "FlashPrefill: long-context acceleration 28x" summary (mhpn.cn),
 *         section 3.1 "instantaneous pattern discovery", 3.2 "max-based
 *         dynamic threshold", 3.3 "index-driven physical jump".
 *   [V2]  "FlashPrefill V2 paper reading" (inkeast.github.io MessageDaily),
 *         section 4 (indexing phase: B=128, 256 sink, 512 local, alpha=0.1),
 *         section 4.1 (block-mean correction equations).
 *   [V2p] "FlashPrefill V2" popular article (animattoys.com), section on
 *         mean correction (weight = the number of tokens of the block).
 *
 * Everything is written straight from those definitions: no tiling, no
 * online softmax, no fusion.  Arrays are row-major, doubles.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

static long ceil_div(long a, long b) { return (a + b - 1) / b; }

static double dot(const double *a, const double *b, int d)
{
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += a[c] * b[c];
    return s;
}

/*
 * Block means [V1 3.1 key pooling; V2 4.1 block means of K and V].
 * x: [lk][h][d] (one request, contiguous positions).  xbar: [nkb][h][d] with
 * nkb = ceil(lk/B); block J holds n_J = min(B, lk - J*B) tokens.
 */
void oracle_pool(const double *x, long lk, int h, int d, int B, double *xbar)
{
    long nkb = ceil_div(lk, B);
#pragma omp parallel for schedule(static)
    for (long J = 0; J < nkb; ++J) {
        long t0 = J * B, t1 = t0 + B < lk ? t0 + B : lk;
        double n = (double)(t1 - t0);
        for (int hh = 0; hh < h; ++hh)
            for (int c = 0; c < d; ++c) {
                double s = 0.0;
                for (long t = t0; t < t1; ++t) s += x[(t * h + hh) * d + c];
                xbar[(J * h + hh) * d + c] = s / n;
            }
    }
}

/*
 * Block-score rows [V1 3.1].  For query block I (absolute index, positions
 * I*B .. I*B+B-1) and kv head h, the packed rows are the g query heads of the
 * group times the block's queries.  For each packed row:
 *     s_J = scale * q . kbar_J          for J <= I
 *     m   = max_J s_J                    (per-query normalisation)
 * S'[J] = sum over packed rows of exp(s_J - m), and the row is re-normalised
 * by its largest entry: Score[I,J] = S'[J] / max_J' S'[J'] ("global
 * re-weighting" with the top key block of the row as the reference).
 *
 * q: [lq][hq][d], query i sits at absolute position start + i (start is a
 * multiple of B).  kbar: [nkb][hkv][d].  rows[k] = i_local*hkv + h selects
 * which rows to compute; row k is written at out + row_off[k] (I+1 values).
 */
void oracle_score_rows(const double *q, long lq, long start, int hq, int hkv, int d,
                       int B, double scale, const double *kbar, long nkb,
                       const long *rows, long nrows, const long *row_off, double *out)
{
    int g = hq / hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (long k = 0; k < nrows; ++k) {
        long il = rows[k] / hkv;
        int h = (int)(rows[k] % hkv);
        long I = start / B + il;
        long ncol = I + 1 < nkb ? I + 1 : nkb;
        double *acc = calloc((size_t)ncol, sizeof(double));
        double *s = malloc((size_t)ncol * sizeof(double));
        long i0 = il * B, i1 = i0 + B < lq ? i0 + B : lq;
        for (int hh = h * g; hh < (h + 1) * g; ++hh)
            for (long i = i0; i < i1; ++i) {
                const double *qi = q + (i * hq + hh) * d;
                double m = -INFINITY;
                for (long J = 0; J < ncol; ++J) {
                    s[J] = scale * dot(qi, kbar + (J * hkv + h) * d, d);
                    if (s[J] > m) m = s[J];
                }
                for (long J = 0; J < ncol; ++J) acc[J] += exp(s[J] - m);
            }
        double mx = 0.0;
        for (long J = 0; J < ncol; ++J)
            if (acc[J] > mx) mx = acc[J];
        for (long J = 0; J < ncol; ++J) out[row_off[k] + J] = acc[J] / mx;
        free(acc);
        free(s);
    }
}

/*
 * Selection for one score row [V1 3.2; V2 section 4 "256 sink, 512 local"]:
 *     keep[J] = Score[J] >= alpha * max_{J<=I} Score[J]
 *               or block J holds one of the first `sink` tokens
 *               or block J is one of the ceil(local/B) blocks ending at I.
 * flag[J] marks scores within 1e-4 (relative) of the threshold, where a
 * different rounding order may legitimately flip the decision.
 */
void oracle_select_row(const double *score, long I, double alpha, int B, int sink,
                       int local, unsigned char *keep, unsigned char *flag)
{
    double mx = -INFINITY;
    for (long J = 0; J <= I; ++J)
        if (score[J] > mx) mx = score[J];
    double thr = alpha * mx;
    long sink_blocks = ceil_div(sink, B);
    long local_blocks = ceil_div(local, B);
    for (long J = 0; J <= I; ++J) {
        int k = score[J] >= thr;
        if (J < sink_blocks) k = 1;
        if (J >= I - local_blocks + 1) k = 1;
        keep[J] = (unsigned char)k;
        flag[J] = (unsigned char)(fabs(score[J] - thr) <= 1e-4 * fabs(thr));
    }
}

/*
 * Alternative selection rules [V1 4.4 compares the max threshold with top-k
 * and top-p selection]; kept as ablations.  For the row scores s[0..I]:
 *   rule 1, top-k: the min(k, I+1) highest scores, equal scores lowest J first;
 *   rule 2, top-p: every J with s[J] >= t, t the highest score such that the
 *                  scores >= t sum to at least p * sum_J s[J];
 * rule 0 is the threshold rule above.  Sink and local blocks are kept under
 * every rule.  flag[J] marks decisions that sit within rounding of the
 * boundary: |s[J] - t| <= 1e-5 (the scores lie in (0, 1]), and for top-p a
 * running mass (descending order, before or after J) within 1e-4 * total of
 * the target.
 */
static const double *g_sort_scores;

static int by_score_desc(const void *a, const void *b)
{
    long i = *(const long *)a, j = *(const long *)b;
    double si = g_sort_scores[i], sj = g_sort_scores[j];
    if (si > sj) return -1;
    if (si < sj) return 1;
    return (i > j) - (i < j);
}

void oracle_select_row_rule(const double *score, long I, int rule, double alpha, int top_k,
                            double top_p, int B, int sink, int local, unsigned char *keep,
                            unsigned char *flag)
{
    if (rule == 0) {
        oracle_select_row(score, I, alpha, B, sink, local, keep, flag);
        return;
    }
    long n = I + 1;
    long *order = malloc((size_t)n * sizeof(long));
    for (long J = 0; J < n; ++J) order[J] = J;
    g_sort_scores = score;             /* the oracle runs rows one at a time here */
    qsort(order, (size_t)n, sizeof(long), by_score_desc);
    for (long J = 0; J < n; ++J) keep[J] = flag[J] = 0;
    double t;
    if (rule == 1) {
        long k = top_k < n ? top_k : n;
        t = score[order[k - 1]];
        for (long q = 0; q < k; ++q) keep[order[q]] = 1;
    } else {
        double total = 0.0;
        for (long J = 0; J < n; ++J) total += score[J];
        double target = top_p * total, cum = 0.0;
        long q = 0;
        while (q < n - 1 && cum + score[order[q]] < target) cum += score[order[q++]];
        t = score[order[q]];
        for (long J = 0; J < n; ++J) keep[J] = score[J] >= t;
        cum = 0.0;
        for (q = 0; q < n; ++q) {
            double before = cum;
            cum += score[order[q]];
            if (fabs(before - target) <= 1e-4 * total || fabs(cum - target) <= 1e-4 * total)
                flag[order[q]] = 1;
        }
    }
    long sink_blocks = ceil_div(sink, B);
    long local_blocks = ceil_div(local, B);
    for (long J = 0; J < n; ++J) {
        if (fabs(score[J] - t) <= 1e-5) flag[J] = 1;
        if (J < sink_blocks || J >= I - local_blocks + 1) keep[J] = 1;
    }
    free(order);
}

/*
 * Sparse attention with block-mean correction for selected query rows
 * [V2 4.1; V2p mean correction], written as the plain ratio of sums:
 *
 *   O(q) = [ sum_{kept J} sum_{t in J, t <= p} e^{s_t - m} v_t
 *            + sum_{skipped J < I} n_J e^{sbar_J - m} vbar_J ]
 *        / [ the same sums without v ],
 *   s_t = scale q.k_t,  sbar_J = scale q.kbar_J,  m = max of all exponents,
 *   LSE = m + ln(denominator).
 *
 * keep == NULL means every causal block is kept (dense causal attention).
 * keep[(i_local*hkv + h)*nkb + J] is the selection of row (I, h).
 * qi[k] is a local query index, qh[k] a query head; results go to
 * o[k*d ...] and lse[k].  A row with no terms gets O = 0, LSE = -inf.
 */
void oracle_attn_rows(const double *q, long lq, long start, int hq, int hkv, int d,
                      int B, double scale, const double *kx, const double *vx, long lk,
                      const double *kbar, const double *vbar, long nkb,
                      const unsigned char *keep, int mean_corr,
                      const long *qi, const int *qh, long n, double *o, double *lse)
{
    int g = hq / hkv;
#pragma omp parallel for schedule(dynamic, 4)
    for (long k = 0; k < n; ++k) {
        long i = qi[k];
        int hh = qh[k];
        int h = hh / g;
        long p = start + i;
        long I = p / B;
        long il = I - start / B;
        const double *qv = q + (i * hq + hh) * d;
        /* every term: its exponent and a pointer to its value vector and weight */
        long cap = p + 1 + I + 1;
        double *e = malloc((size_t)cap * sizeof(double));
        const double **val = malloc((size_t)cap * sizeof(double *));
        long nt = 0;
        for (long J = 0; J <= I && J < nkb; ++J) {
            int kept = keep ? keep[(il * hkv + h) * nkb + J] : 1;
            if (kept) {
                long t1 = (J + 1) * B - 1;
                if (t1 > p) t1 = p;
                for (long t = J * B; t <= t1; ++t) {
                    e[nt] = scale * dot(qv, kx + (t * hkv + h) * d, d);
                    val[nt++] = vx + (t * hkv + h) * d;
                }
            } else if (mean_corr && J < I) {
                long nJ = lk - J * B < B ? lk - J * B : B;
                e[nt] = scale * dot(qv, kbar + (J * hkv + h) * d, d) + log((double)nJ);
                val[nt++] = vbar + (J * hkv + h) * d;
            }
        }
        double m = -INFINITY;
        for (long t = 0; t < nt; ++t)
            if (e[t] > m) m = e[t];
        double den = 0.0;
        double *num = calloc((size_t)d, sizeof(double));
        for (long t = 0; t < nt; ++t) {
            double w = exp(e[t] - m);
            den += w;
            for (int c = 0; c < d; ++c) num[c] += w * val[t][c];
        }
        for (int c = 0; c < d; ++c) o[k * d + c] = nt ? num[c] / den : 0.0;
        lse[k] = nt ? m + log(den) : -INFINITY;
        free(num);
        free(e);
        free(val);
    }
}
