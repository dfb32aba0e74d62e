/*
 * oracle.c -- plain, slow, scalar CPU oracle for batch speculative-decoding
 * verification and the ragged-to-rectangular realignment it forces.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may link,
 * load or call this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant with the
 * CUDA path: every definition below is restated from the pages it cites.
 *
 * Pages cited (by title and section):
 *   [CF]  "Correctness Forensics for Batch Speculative Decoding: Diagnosing the
 *         Ragged Tensor Problem" (source-linked summary of arXiv 2510.22876v4)
 *   [ZS]  "Chapter 10 Speculative Decoding (Code Walkthrough)" (zero-to-sglang)
 *   [SDR] "Design Document -- speculative-decoding-real"
 *   [AL]  "Speculative decoding: proposals and verified output" (Atlas lesson)
 *
 * Arithmetic: probabilities in fp64 (double); logits are read exactly from
 * their storage type (fp32, bf16 or fp16 bit patterns) into double.  The
 * loops over sequences and cache slabs may run on several threads
 * (oracle_set_threads), with results identical to one thread.
 *
 * Pins: every function here is checked in tests/test_oracle_*.py against
 * values the pages print, closed forms, brute force on tiny inputs and planted
 * mistakes (the oracle_set_mutant switch below).  The length-grouping policy
 * (oracle_group_by_length) is this project's own construction because the
 * pages give the EXSPEC scheduling appendix as a heading with no body: its
 * parity is UNPINNED by the pages (it is only checked against an independent
 * brute-force restatement of the same policy).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads for the loops over sequences and cache slabs (OpenMP when built
   with it; 1 by default).  Every sequence and every slab is computed exactly
   as on one thread -- nothing is reduced across them -- so the results do
   not depend on the thread count. */
static int g_threads = 1;
void oracle_set_threads(int n) { g_threads = n > 0 ? n : 1; }
int oracle_threads_available(void)
{
#ifdef _OPENMP
    return omp_get_num_procs();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* storage types of the logits                                         */
/* ------------------------------------------------------------------ */
enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2 };

/* IEEE binary16 -> double, from the format's definition (1 sign bit, 5
   exponent bits with bias 15, 10 fraction bits; exponent 0 = subnormal,
   exponent 31 = inf / NaN). */
static double half_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m | 0x400), e - 25);
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double logit_at(const void *x, int dtype, int64_t i)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)x)[i];
    if (dtype == ORACLE_BF16)
        return bf16_bits_to_double(((const uint16_t *)x)[i]);
    return half_bits_to_double(((const uint16_t *)x)[i]);
}

/* ------------------------------------------------------------------ */
/* planted mistakes, used only by the tests to show that the pins catch */
/* them; 0 = the correct oracle                                          */
/* ------------------------------------------------------------------ */
enum {
    MUT_NONE = 0,
    MUT_TIE_HIGHEST = 1,      /* argmax keeps the highest index among ties  */
    MUT_ROW_SHIFT = 2,        /* proposal j checked against row j+1         */
    MUT_RESAMPLE_FROM_P = 3,  /* correction drawn from p, not the residual  */
    MUT_BONUS_FROM_DRAFT = 4, /* bonus drawn from the last draft row        */
    MUT_NO_CLAMP = 5,         /* residual p-q without the positive part     */
    MUT_CDF_GE = 6,           /* inverse CDF tests C_i >= target            */
    MUT_SKIP_KV_SHIFT = 7,    /* realign updates lengths but moves no KV    */
    MUT_STALE_POSITIONS = 8,  /* position/mask rebuild writes nothing       */
    MUT_BONUS_ALWAYS = 9,     /* bonus appended even after a rejection      */
    MUT_SHIFT_ONE_SHORT = 10, /* KV run moved one row short                 */
    MUT_TOPK_STRICT = 11,     /* top-k drops the ties at the k-th value     */
    MUT_TOPP_BELOW = 12,      /* nucleus = largest top set of mass <= top_p */
    MUT_RATIO_UNFILTERED = 13,/* ratio test on p before the transforms      */
    MUT_RESID_UNFILTERED = 14,/* residual built from p before the transforms*/
    MUT_TOPP_FIRST = 15,      /* top-p applied before top-k                 */
    MUT_ZERO_SIGN_ORDER = 16  /* cut compares -0 as smaller than +0         */
};
static int g_mutant = MUT_NONE;
void oracle_set_mutant(int m) { g_mutant = m; }

/* ------------------------------------------------------------------ */
/* O1  greedy verification                                              */
/* ------------------------------------------------------------------ */

/* Index of the largest value of row x[off .. off+V): the lowest index among
   equal maxima, and a NaN counts as larger than every number (the first NaN
   wins).  The pages name tie-breaking as a source of divergence without fixing
   it ([CF] §4.2); lowest-index is the reading taken here. */
static int argmax_row(const void *x, int dtype, int64_t off, int V)
{
    int best = 0;
    double bv = logit_at(x, dtype, off);
    for (int v = 1; v < V; ++v) {
        if (isnan(bv))
            break;
        double xv = logit_at(x, dtype, off + v);
        int better = isnan(xv) || xv > bv;
        if (g_mutant == MUT_TIE_HIGHEST)
            better = better || xv == bv;
        if (better) {
            best = v;
            bv = xv;
        }
    }
    return best;
}

/*
 * Greedy commitment of one verification round for every sequence of a batch,
 * restating the teaching function greedy_commit ([ZS] §4.1) and steps 4-6 of
 * the standard greedy algorithm ([SDR] "Standard Greedy Algorithm"):
 *   - row j of sequence b (j < k_b) verifies proposal j; row k_b gives the
 *     bonus ([ZS] §3.3: with confirmed prefix L, rows L-1 .. L+k-2 verify and
 *     row L+k-1 gives the extra token; here those rows arrive as j = 0..k);
 *   - the argmax t of row j is committed; the round stops after it when t is
 *     EOS, when the output budget is reached, or when t differs from the
 *     proposal (t is then the correction);
 *   - after all k_b proposals are accepted the argmax of row k_b is the bonus,
 *     drawn from the target ([CF] App. D).
 *
 * logits       [B, k+1, V] in `dtype`
 * draft_tokens [B, k]
 * draft_len    [B] or NULL (NULL: every sequence has k proposals)
 * eos_id       token that ends a sequence, or negative for none
 * remaining    [B] output budget or NULL (NULL: unlimited); 0 commits nothing
 * out_tokens   [B, k+1] committed tokens, -1 after the last one
 * n_accept     [B] committed tokens that are accepted proposals
 * n_emit       [B] committed tokens (accepted + correction/bonus)
 */
void oracle_verify_greedy(const void *logits, int dtype, int B, int k, int V,
                          const int32_t *draft_tokens, const int32_t *draft_len,
                          int32_t eos_id, const int32_t *remaining,
                          int32_t *out_tokens, int32_t *n_accept, int32_t *n_emit)
{
#pragma omp parallel for num_threads(g_threads) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        int kb = draft_len ? draft_len[b] : k;
        int64_t rem = remaining ? remaining[b] : INT64_MAX;
        int32_t *out = out_tokens + (int64_t)b * (k + 1);
        int ne = 0, na = 0, stopped = 0;
        for (int i = 0; i <= k; ++i)
            out[i] = -1;
        if (rem > 0) {
            for (int j = 0; j < kb; ++j) {
                int row = (g_mutant == MUT_ROW_SHIFT) ? j + 1 : j;
                int t = argmax_row(logits, dtype, ((int64_t)b * (k + 1) + row) * V, V);
                int match = (t == draft_tokens[(int64_t)b * k + j]);
                out[ne++] = t;
                if (match)
                    na++;
                if ((eos_id >= 0 && t == eos_id) || ne == rem || !match) {
                    stopped = 1;
                    break;
                }
            }
            if (!stopped || g_mutant == MUT_BONUS_ALWAYS) {
                if (ne < k + 1 && ne < rem)
                    out[ne++] = argmax_row(logits, dtype, ((int64_t)b * (k + 1) + kb) * V, V);
            }
        }
        n_accept[b] = na;
        n_emit[b] = ne;
    }
}

/* ------------------------------------------------------------------ */
/* O2  stochastic verification                                           */
/* ------------------------------------------------------------------ */

/* p = softmax(x / T) of one row in fp64: m = max z, p_v = e^(z_v - m) / sum.
   A -inf logit is a masked token with probability 0.  Returns 1 when the
   distribution is undefined: a NaN or +inf logit, or no finite logit at all. */
static int softmax_row(const void *x, int dtype, int64_t off, int V, double T, double *p)
{
    int bad = 0;
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double z = logit_at(x, dtype, off + v) / T;
        p[v] = z;
        if (isnan(z) || z == INFINITY)
            bad = 1;
        if (z > m)
            m = z;
    }
    double s = 0.0;
    for (int v = 0; v < V; ++v) {
        p[v] = exp(p[v] - m);
        s += p[v];
    }
    for (int v = 0; v < V; ++v)
        p[v] /= s;
    if (!isfinite(s) || s <= 0.0)
        bad = 1;
    return bad;
}

/* ------------------------------------------------------------------ */
/* O2b  sampling transforms: temperature, top-k, top-p                  */
/* ------------------------------------------------------------------ */

/*
 * The ratio test, the residual and the bonus use the distribution the sampler
 * actually draws from: "if temperature, Top-k, or Top-p is applied, retain the
 * processed probabilities" ([ZS] §5.1), the same transforms on the same
 * events ([AL] "The mechanism" step 1).  The pages name the transforms
 * without defining them; this oracle takes the usual definitions, applied in
 * the order temperature, top-k, top-p:
 *
 *   top-k (k >= 1, off when k <= 0 or k >= V): keep the tokens whose logit is
 *     at least the k-th largest logit (counting repeats), so tokens tied with
 *     the k-th value are all kept;
 *   top-p (off when top_p >= 1 or NaN): among the top-k survivors, keep token
 *     v iff the mass of the tokens with a strictly larger logit is below
 *     top_p * (total mass) -- the smallest set of top values whose mass
 *     reaches top_p, with ties at the boundary kept; the most probable value
 *     is always kept (so top_p <= 0 keeps only it);
 *   then p = softmax(x / T) renormalised over the kept tokens (fp64).
 *
 * The top-p decision is taken on that definition in real arithmetic.  The
 * masses are m_v = e^{(x_v - x_max) / T} (x_max the largest kept logit, so
 * the top mass is exactly 1), computed in fp64: x_v - x_max and the division
 * by T are rounded once each (|a| u of relative error for the exponent a,
 * u = 2^-53), exp within one ulp, so each mass is within (2 + |a|) u of its
 * exact value relative, and |a| e^a <= 1/e bounds the second part by u/e in
 * absolute terms.  Sums are compensated (Neumaier), within 2u of the exact
 * sum of their terms.  A partial mass A and the total M are therefore
 * within 4u M + n u / e of their exact values (n kept tokens), and the
 * comparison A < top_p * M (top_p the fp32 value as given, the product
 * rounded once) is exact whenever |A - top_p M| exceeds
 *   eps = (10 M + n) u.
 * A decision inside that band is taken as computed and reported (the
 * "undecided" output of oracle_filter_cut); at the sizes used here the band
 * is ~1e-15 of the total.
 */

/* compensated (Neumaier) running sum */
typedef struct {
    double s, c;
} CSum;
static void csum_add(CSum *a, double v)
{
    double t = a->s + v;
    if (fabs(a->s) >= fabs(v))
        a->c += (a->s - t) + v;
    else
        a->c += (v - t) + a->s;
    a->s = t;
}
static double csum_val(const CSum *a) { return a->s + a->c; }

typedef struct {
    double x;
    int v;
} ValIdx;

/* descending by value; equal values in index order (irrelevant to the result) */
static int cmp_desc(const void *a, const void *b)
{
    const ValIdx *p = (const ValIdx *)a, *q = (const ValIdx *)b;
    if (p->x > q->x)
        return -1;
    if (p->x < q->x)
        return 1;
    return (p->v > q->v) - (p->v < q->v);
}

/* the value the cut compares: the logit itself (the planted mistake orders
   -0 below +0, as a comparison of bit patterns would) */
static double cut_value(double x)
{
    return (g_mutant == MUT_ZERO_SIGN_ORDER && x == 0.0 && signbit(x)) ? -DBL_MIN : x;
}

/* Smallest kept logit (the keep test is x >= cut) of a row after top-k and
   top-p; -inf when nothing is filtered.  vals is scratch of V entries.
   Optional outputs: *margin = min |A - top_p M| over the two top-p decisions
   next to the cut (masses in units of the top mass; +inf without top-p),
   *total = M, *undecided = 1 when a decision of the row fell inside the
   error band eps. */
static double filter_cut(const void *x, int dtype, int64_t off, int V, float T, int top_k, float top_p,
                         ValIdx *vals, double *margin, double *total_out, int *undecided)
{
    int use_k = top_k > 0 && top_k < V;
    int use_p = top_p < 1.0f;
    if (margin)
        *margin = INFINITY;
    if (total_out)
        *total_out = 0.0;
    if (undecided)
        *undecided = 0;
    if (!use_k && !use_p)
        return -INFINITY;
    for (int v = 0; v < V; ++v) {
        vals[v].x = cut_value(logit_at(x, dtype, off + v));
        vals[v].v = v;
    }
    qsort(vals, (size_t)V, sizeof *vals, cmp_desc);
    double cut_k = -INFINITY;
    if (use_k && g_mutant != MUT_TOPP_FIRST)
        cut_k = vals[top_k - 1].x;
    /* top-k survivors are vals[0 .. nk) */
    int nk = 0;
    while (nk < V && vals[nk].x >= cut_k && !(g_mutant == MUT_TOPK_STRICT && use_k && vals[nk].x == cut_k))
        ++nk;
    if (!use_p) {
        if (nk == 0)
            return INFINITY;
        return vals[nk - 1].x;
    }
    const double Td = (double)T;
    const double xmax = vals[0].x;
    CSum tot = {0.0, 0.0};
    for (int i = 0; i < nk; ++i)
        csum_add(&tot, exp((vals[i].x - xmax) / Td));
    const double M = csum_val(&tot);
    const double bound = (double)top_p * M;
    const double eps = (10.0 * M + (double)nk) * 0x1p-53;
    CSum above = {0.0, 0.0};
    double prev_gap = INFINITY, last_gap = INFINITY;
    int i = 0, und = 0;
    double cut = vals[0].x;
    while (i < nk) {
        int e = i; /* the group of values equal to vals[i] */
        CSum gm = {0.0, 0.0};
        while (e < nk && vals[e].x == vals[i].x) {
            csum_add(&gm, exp((vals[e].x - xmax) / Td));
            ++e;
        }
        const double a = csum_val(&above);
        int keep = (i == 0) || (a < bound);
        if (g_mutant == MUT_TOPP_BELOW)
            keep = (i == 0) || (a + csum_val(&gm) <= bound);
        const double gap = fabs(a - bound);
        if (i > 0 && gap <= eps)
            und = 1;
        if (!keep) {
            last_gap = gap; /* the first dropped group */
            break;
        }
        if (i > 0)
            prev_gap = gap; /* the last kept group (so far) */
        cut = vals[i].x;
        csum_add(&above, csum_val(&gm));
        i = e;
    }
    if (margin)
        *margin = fmin(prev_gap, last_gap);
    if (total_out)
        *total_out = M;
    if (undecided)
        *undecided = und;
    if (g_mutant == MUT_TOPP_FIRST && use_k) {
        /* mistaken order: the top-k cut taken after the nucleus */
        double ck = vals[top_k - 1].x;
        if (ck > cut)
            cut = ck;
    }
    return cut;
}

/* p = the processed distribution of one row: softmax(x / T) restricted to the
   tokens top-k and top-p keep, renormalised, in fp64.  Returns the undefined
   flag of softmax_row (no filtering is applied to an undefined row). */
static int processed_row(const void *x, int dtype, int64_t off, int V, double T, int top_k, float top_p, double *p,
                         ValIdx *vals)
{
    int bad = softmax_row(x, dtype, off, V, T, p);
    if (bad)
        return bad;
    double cut = filter_cut(x, dtype, off, V, (float)T, top_k, top_p, vals, NULL, NULL, NULL);
    if (cut == -INFINITY)
        return 0;
    double s = 0.0;
    for (int v = 0; v < V; ++v) {
        if (!(cut_value(logit_at(x, dtype, off + v)) >= cut))
            p[v] = 0.0;
        s += p[v];
    }
    for (int v = 0; v < V; ++v)
        p[v] /= s;
    return 0;
}

/* Inverse CDF of the weights w[0..V) at uniform u in [0,1): the smallest i
   whose sequential fp64 prefix sum C_i exceeds u * sum(w).  If rounding leaves
   no such i, the last index with positive weight.  A zero-weight index is
   therefore never returned. */
static int inverse_cdf(const double *w, int V, double u)
{
    double total = 0.0;
    for (int i = 0; i < V; ++i)
        total += w[i];
    double target = u * total;
    double c = 0.0;
    for (int i = 0; i < V; ++i) {
        c += w[i];
        int hit = (g_mutant == MUT_CDF_GE) ? (c >= target) : (c > target);
        if (hit)
            return i;
    }
    for (int i = V - 1; i >= 0; --i)
        if (w[i] > 0.0)
            return i;
    return V - 1;
}

/*
 * Stochastic verification of one round ([ZS] §5.1; [AL] "The mechanism" steps
 * 2-4 and "Acceptance and rejection correction"):
 *   - p_j = softmax(x_j / T) of target row j; q_j = draft_probs[b, j, :];
 *   - proposal y = d_j is accepted iff u_{b,j} < p_j(y) / q_j(y), which is
 *     acceptance with probability min(1, p/q) since u < 1;
 *   - on the first rejection the correction is drawn from the normalised
 *     positive residual r = max(0, p_j - q_j) / sum(...) and the round stops;
 *     the residual is used only when its sum is positive ([AL] "Assumptions";
 *     [ZS] "check numerical validity"); otherwise the draw is from p_j and
 *     flag bit 2 is set;
 *   - after k_b acceptances the bonus is drawn from p_{k_b}, the target
 *     ([CF] App. D), never from the draft;
 *   - one uniform per ratio test (columns 0..k-1) and a single uniform for
 *     the one draw of the round (column k) -- this layout is this project's
 *     reading: the page draws them with separate torch.rand / multinomial;
 *   - EOS and the output budget stop the round as in greedy commitment.
 * Flags per sequence: 1 = a tested proposal had q(y) = 0 (the page says such a
 * symbol cannot be proposed; IEEE then gives +inf -> accept when p > 0, or
 * NaN -> reject when p = 0), 2 = zero residual mass, 4 = a used row whose
 * softmax is undefined (a NaN or +inf logit, or every logit -inf; a -inf
 * logit alone is a masked token of probability 0), 8 = a proposal outside
 * [0, V) (rejected).
 *
 * out_residual [B, V] (or NULL): the normalised distribution the final draw
 * came from (residual, or p on zero residual, or the bonus row's p); rows of
 * sequences that drew nothing are left untouched.
 */
/* sequence b of oracle_verify_sample; p, w, praw, vals: V-sized scratch */
static void sample_sequence(int b, const void *logits, int dtype, double temperature,
                            const float *draft_probs, const int32_t *draft_tokens,
                            const float *uniforms, int k, int V,
                            const int32_t *draft_len, int32_t eos_id,
                            const int32_t *remaining, int32_t *out_tokens,
                            int32_t *n_accept, int32_t *n_emit, double *out_residual,
                            uint32_t *flags, const int32_t *top_k, const float *top_p,
                            double *p, double *w, double *praw, ValIdx *vals)
{
    {
        int tk = top_k ? top_k[b] : 0;
        float tp = top_p ? top_p[b] : 1.0f;
        int kb = draft_len ? draft_len[b] : k;
        int64_t rem = remaining ? remaining[b] : INT64_MAX;
        int32_t *out = out_tokens + (int64_t)b * (k + 1);
        const float *u = uniforms + (int64_t)b * (k + 1);
        uint32_t fl = 0;
        int ne = 0, na = 0, stopped = 0, draw_row = -1, draw_residual = 0;
        for (int i = 0; i <= k; ++i)
            out[i] = -1;
        if (rem > 0) {
            for (int j = 0; j < kb; ++j) {
                int y = draft_tokens[(int64_t)b * k + j];
                const float *q = draft_probs + ((int64_t)b * k + j) * V;
                const int64_t roff = ((int64_t)b * (k + 1) + j) * V;
                if (processed_row(logits, dtype, roff, V, temperature, tk, tp, p, vals))
                    fl |= 4;
                if (g_mutant == MUT_RATIO_UNFILTERED || g_mutant == MUT_RESID_UNFILTERED)
                    softmax_row(logits, dtype, roff, V, temperature, praw);
                /* a proposal outside the vocabulary has no probability under
                   either model: flag 8 and treat it as rejected */
                int valid = y >= 0 && y < V;
                if (!valid)
                    fl |= 8;
                if (valid && q[y] == 0.0f)
                    fl |= 1;
                const double *pr = (g_mutant == MUT_RATIO_UNFILTERED) ? praw : p;
                double ratio = valid ? pr[y] / (double)q[y] : 0.0;
                if (valid && (double)u[j] < ratio) {
                    out[ne++] = y;
                    na++;
                    if ((eos_id >= 0 && y == eos_id) || ne == rem) {
                        stopped = 1;
                        break;
                    }
                    continue;
                }
                /* first rejection: correction from the positive residual */
                double total = 0.0;
                const double *pw = (g_mutant == MUT_RESID_UNFILTERED) ? praw : p;
                for (int v = 0; v < V; ++v) {
                    double d = pw[v] - (double)q[v];
                    w[v] = (g_mutant == MUT_NO_CLAMP) ? d : (d > 0.0 ? d : 0.0);
                    total += w[v];
                }
                if (g_mutant == MUT_RESAMPLE_FROM_P || !(total > 0.0)) {
                    if (!(total > 0.0))
                        fl |= 2;
                    memcpy(w, p, sizeof(double) * (size_t)V);
                }
                draw_row = j;
                draw_residual = 1;
                stopped = 1;
                break;
            }
            if (!stopped) {
                /* bonus from the target row k_b */
                if (g_mutant == MUT_BONUS_FROM_DRAFT && kb > 0) {
                    const float *q = draft_probs + ((int64_t)b * k + kb - 1) * V;
                    for (int v = 0; v < V; ++v)
                        w[v] = (double)q[v];
                } else {
                    if (processed_row(logits, dtype, ((int64_t)b * (k + 1) + kb) * V, V, temperature, tk, tp, p,
                                      vals))
                        fl |= 4;
                    memcpy(w, p, sizeof(double) * (size_t)V);
                }
                draw_row = kb;
            }
            if (draw_row >= 0) {
                out[ne++] = inverse_cdf(w, V, (double)u[k]);
                if (out_residual) {
                    double total = 0.0;
                    for (int v = 0; v < V; ++v)
                        total += w[v];
                    for (int v = 0; v < V; ++v)
                        out_residual[(int64_t)b * V + v] = w[v] / total;
                }
            }
        }
        (void)draw_residual;
        n_accept[b] = na;
        n_emit[b] = ne;
        if (flags)
            flags[b] = fl;
    }
}

void oracle_verify_sample(const void *logits, int dtype, double temperature,
                          const float *draft_probs, const int32_t *draft_tokens,
                          const float *uniforms, int B, int k, int V,
                          const int32_t *draft_len, int32_t eos_id,
                          const int32_t *remaining, int32_t *out_tokens,
                          int32_t *n_accept, int32_t *n_emit, double *out_residual,
                          uint32_t *flags, const int32_t *top_k, const float *top_p)
{
    size_t nv = (size_t)(V > 0 ? V : 1);
#pragma omp parallel num_threads(g_threads)
    {
        double *p = (double *)malloc(sizeof(double) * nv);
        double *w = (double *)malloc(sizeof(double) * nv);
        double *praw = (double *)malloc(sizeof(double) * nv);
        ValIdx *vals = (ValIdx *)malloc(sizeof(ValIdx) * nv);
#pragma omp for schedule(dynamic, 1)
        for (int b = 0; b < B; ++b)
            sample_sequence(b, logits, dtype, temperature, draft_probs, draft_tokens, uniforms, k, V, draft_len,
                            eos_id, remaining, out_tokens, n_accept, n_emit, out_residual, flags, top_k, top_p, p, w,
                            praw, vals);
        free(p);
        free(w);
        free(praw);
        free(vals);
    }
}

/* fp64 processed distribution of one logits row (top_k <= 0 and top_p >= 1:
   plain softmax), exported for the tests' tolerance accounting (they
   recompute p/q and CDF boundaries next to a mismatch). */
int oracle_softmax_row(const void *logits, int dtype, int64_t row, int V, double T, int top_k, float top_p,
                       double *p)
{
    ValIdx *vals = (ValIdx *)malloc(sizeof(ValIdx) * (size_t)(V > 0 ? V : 1));
    int bad = processed_row(logits, dtype, row * V, V, T, top_k, top_p, p, vals);
    free(vals);
    return bad;
}

/* The smallest kept logit of a row after top-k / top-p (-inf: no filter);
   info (or NULL) receives [margin, total mass, undecided] of the top-p
   decision (filter_cut). */
double oracle_filter_cut(const void *logits, int dtype, int64_t row, int V, float T, int top_k, float top_p,
                         double *info)
{
    ValIdx *vals = (ValIdx *)malloc(sizeof(ValIdx) * (size_t)(V > 0 ? V : 1));
    double margin, total;
    int und;
    double cut = filter_cut(logits, dtype, row * V, V, T, top_k, top_p, vals, &margin, &total, &und);
    free(vals);
    if (info) {
        info[0] = margin;
        info[1] = total;
        info[2] = (double)und;
    }
    return cut;
}

/* ------------------------------------------------------------------ */
/* O3  realignment plan and KV shift                                      */
/* ------------------------------------------------------------------ */

/*
 * Unpad-append-repad ([CF] §3.2 and App. B), stated on per-sequence lengths.
 * Layout: sequence b is left-padded, its confirmed tokens occupy slots
 * pad_b .. pad_b + len_b - 1 of a common width W = pad_b + len_b (rectangular
 * alignment, invariant I1), and min_b pad_b = 0.  After a round that commits
 * n_b tokens: len'_b = len_b + n_b, the new width is W' = max_b len'_b (repad to
 * the new maximum length) and pad'_b = W' - len'_b.
 * Returns 0, or 2 when I1 does not hold on input (or a length is < 1), 3 when
 * a run would start beyond the buffer (W + n_b - 1 > S or n_b < 0), 1 when the
 * new width does not fit (W' > S).  Outputs are written only on 0.
 */
int oracle_realign_plan(int B, int S, const int32_t *len, const int32_t *pad,
                        const int32_t *n_emit, int32_t *len_new, int32_t *pad_new,
                        int32_t *width_new)
{
    if (B <= 0)
        return 0;
    int64_t W = (int64_t)pad[0] + len[0];
    int64_t min_pad = pad[0];
    for (int b = 0; b < B; ++b) {
        if (len[b] < 1 || pad[b] < 0 || (int64_t)pad[b] + len[b] != W)
            return 2;
        if (pad[b] < min_pad)
            min_pad = pad[b];
    }
    if (min_pad != 0)
        return 2;
    int64_t Wn = 0;
    for (int b = 0; b < B; ++b) {
        if (n_emit[b] < 0 || W + n_emit[b] - 1 > S)
            return 3;
        int64_t ln = (int64_t)len[b] + n_emit[b];
        if (ln > Wn)
            Wn = ln;
    }
    if (Wn > S)
        return 1;
    for (int b = 0; b < B; ++b) {
        int64_t ln = (int64_t)len[b] + n_emit[b];
        int64_t pn = Wn - ln;
        len_new[b] = (int32_t)ln;
        pad_new[b] = (int32_t)pn;
    }
    *width_new = (int32_t)Wn;
    return 0;
}

/*
 * Move the KV run of one (layer, K/V, sequence, head) slab.  A slab is S rows
 * of row_bytes each.  After the round, sequence b's valid KV covers positions
 * 0 .. len'_b - 2: the rows that were there, the row of the previous last token
 * and the rows of the accepted proposals, all target-computed; the committed
 * correction or bonus token has no KV until the next forward ([CF] App. D;
 * [ZS] §5.2).  The run of len'_b - 1 rows moves from slot pad_b to slot pad'_b
 * with memmove semantics; no other byte changes (stale slots stay as they are
 * and are masked).  Relocating retained entries and dropping rejected ones is
 * [CF] App. B's description of EQSPEC realignment.
 */
void oracle_shift_slab(uint8_t *slab, int64_t row_bytes, int pad_old, int pad_new, int n_rows)
{
    if (g_mutant == MUT_SKIP_KV_SHIFT)
        return;
    if (g_mutant == MUT_SHIFT_ONE_SHORT && n_rows > 0)
        n_rows -= 1;
    if (pad_old == pad_new || n_rows <= 0)
        return;
    memmove(slab + (int64_t)pad_new * row_bytes, slab + (int64_t)pad_old * row_bytes,
            (size_t)((int64_t)n_rows * row_bytes));
}

/* Plan and shift on a contiguous left-padded cache kv[L, 2, B, H, S, D] whose
   elements are elt_bytes wide.  Returns the plan's status; kv is untouched
   unless it is 0. */
int oracle_realign_kv(void *kv, int elt_bytes, int L, int B, int H, int S, int D,
                      const int32_t *len, const int32_t *pad, const int32_t *n_emit,
                      int32_t *len_new, int32_t *pad_new, int32_t *width_new)
{
    if (B <= 0)
        return 0;
    int32_t *ln = (int32_t *)malloc(sizeof(int32_t) * (size_t)B);
    int32_t *pn = (int32_t *)malloc(sizeof(int32_t) * (size_t)B);
    int32_t *po = (int32_t *)malloc(sizeof(int32_t) * (size_t)B);
    int32_t wn = 0;
    memcpy(po, pad, sizeof(int32_t) * (size_t)B); /* outputs may alias inputs */
    int st = oracle_realign_plan(B, S, len, pad, n_emit, ln, pn, &wn);
    if (st == 0) {
        int64_t row_bytes = (int64_t)D * elt_bytes;
        int64_t slab_bytes = row_bytes * S;
        int64_t n_slabs = (int64_t)L * 2 * B * H;
        /* slabs are disjoint: each is moved exactly as on one thread */
#pragma omp parallel for num_threads(g_threads) schedule(dynamic, 16)
        for (int64_t slab = 0; slab < n_slabs; ++slab) {
            int b = (int)((slab / H) % B);
            oracle_shift_slab((uint8_t *)kv + slab * slab_bytes, row_bytes, po[b], pn[b], ln[b] - 1);
        }
        memcpy(len_new, ln, sizeof(int32_t) * (size_t)B);
        memcpy(pad_new, pn, sizeof(int32_t) * (size_t)B);
        *width_new = wn;
    }
    free(ln);
    free(pn);
    free(po);
    return st;
}

/* ------------------------------------------------------------------ */
/* O4  position IDs and attention mask                                    */
/* ------------------------------------------------------------------ */

/* Recompute the mask and the positions of every row from the new padding:
   mask[b, s] = 1 for s >= pad'_b (0 in the left padding), and positions are
   recomputed from the mask ([CF] App. B) as cumsum(mask) - 1, clamped at 0 in
   the padding.  Slots at or beyond the new width keep counting, so the next
   round's query slots need no rewrite. */
void oracle_rebuild_pos_mask(int B, int S, const int32_t *pad_new, int32_t *pos, uint8_t *mask)
{
    if (g_mutant == MUT_STALE_POSITIONS)
        return;
    for (int b = 0; b < B; ++b) {
        int64_t csum = 0;
        for (int s = 0; s < S; ++s) {
            uint8_t m = (s >= pad_new[b]) ? 1 : 0;
            mask[(int64_t)b * S + s] = m;
            csum += m;
            int64_t p = csum - 1;
            pos[(int64_t)b * S + s] = (int32_t)(p < 0 ? 0 : p);
        }
    }
}

/* ------------------------------------------------------------------ */
/* O5  same-length grouping (policy UNPINNED by the pages)                  */
/* ------------------------------------------------------------------ */

/*
 * EXSPEC keeps sequences ragged and batches sequences of identical current
 * length so realignment can be skipped ([CF] §3.2).  The pages give no
 * algorithm (the appendix is a bare heading), so this policy is this project's
 * construction:
 *   - L* = the most frequent length among active sequences, ties to the
 *     smaller length;
 *   - members: active sequences of length L* in ascending index, at most B;
 *     count_equal = their number;
 *   - the remaining slots are filled with the other active sequences in
 *     ascending (|len - L*|, index);
 *   - slots beyond the number of active sequences hold -1;
 *   - group_len = L*, or -1 when no sequence is active.
 */
void oracle_group_by_length(int N, const int32_t *len, const uint8_t *active, int B,
                            int32_t *out_idx, int32_t *count_equal, int32_t *group_len)
{
    int64_t best_len = -1, best_cnt = 0;
    for (int i = 0; i < N; ++i) {
        if (active && !active[i])
            continue;
        int64_t cnt = 0;
        for (int j = 0; j < N; ++j)
            if ((!active || active[j]) && len[j] == len[i])
                cnt++;
        if (cnt > best_cnt || (cnt == best_cnt && len[i] < best_len)) {
            best_cnt = cnt;
            best_len = len[i];
        }
    }
    for (int s = 0; s < B; ++s)
        out_idx[s] = -1;
    *group_len = (int32_t)best_len;
    int n = 0;
    uint8_t *taken = (uint8_t *)calloc((size_t)(N > 0 ? N : 1), 1);
    for (int i = 0; i < N && n < B; ++i)
        if ((!active || active[i]) && len[i] == best_len) {
            out_idx[n++] = i;
            taken[i] = 1;
        }
    *count_equal = n;
    while (n < B) {
        int pick = -1;
        int64_t pick_d = 0;
        for (int i = 0; i < N; ++i) {
            if ((active && !active[i]) || taken[i])
                continue;
            int64_t d = llabs((int64_t)len[i] - best_len);
            if (pick < 0 || d < pick_d) {
                pick = i;
                pick_d = d;
            }
        }
        if (pick < 0)
            break;
        out_idx[n++] = pick;
        taken[pick] = 1;
    }
    free(taken);
}

/* ------------------------------------------------------------------ */
/* O7  ragged pool (EXSPEC) -- repad, unpad, commit                        */
/* ------------------------------------------------------------------ */

/*
 * EXSPEC keeps sequences ragged ([CF] §3.2): here a pool cache
 * pool[L, 2, N, H, S, D] holds sequence n left-aligned at slot 0, positions
 * 0 .. pool_len[n] - 2 with KV (the last token has none).  Position = slot, so
 * rectangular alignment is never needed for a group of equal lengths, and a
 * round's rejected proposals need no movement: their rows lie past the new
 * length (the "rollback of rejected tokens" of variable-length layouts, [CF]
 * §2, is the length update).  When no same-length group forms, EXSPEC falls
 * back to unpad-append-repad ([CF] §3.2): the chosen sequences are repadded
 * into a contiguous left-padded batch, realigned there round by round, and
 * unpadded back into the pool.
 */

/* pool_len[idx[b]] += n_emit[b].  Returns 0, 2 for a bad or repeated index
   (or a negative count), 1 when a length would exceed S; nothing changes
   unless it returns 0. */
int oracle_commit_ragged(int N, int32_t *pool_len, int B, const int32_t *idx, const int32_t *n_emit, int S)
{
    for (int b = 0; b < B; ++b) {
        if (idx[b] < 0 || idx[b] >= N || n_emit[b] < 0)
            return 2;
        for (int c = 0; c < b; ++c)
            if (idx[c] == idx[b])
                return 2;
    }
    for (int b = 0; b < B; ++b)
        if ((int64_t)pool_len[idx[b]] + n_emit[b] > S)
            return 1;
    for (int b = 0; b < B; ++b)
        pool_len[idx[b]] += n_emit[b];
    return 0;
}

/* Repad: batch slab (l, c, b, h) receives the pool slab (l, c, idx[b], h)'s
   rows 0 .. pool_len[idx[b]] - 2 at slot pad_b = W - pool_len[idx[b]], with
   W = max_b pool_len[idx[b]]; no other batch byte changes.  Outputs the
   batch lengths, paddings and width.  Returns 0, or 2 for a bad or repeated
   index or a length < 1 (nothing written). */
int oracle_repad_gather(const void *pool, void *batch, int elt_bytes, int L, int N, int B, int H, int S, int D,
                        const int32_t *idx, const int32_t *pool_len, int32_t *len_out, int32_t *pad_out,
                        int32_t *width_out)
{
    int64_t W = 0;
    for (int b = 0; b < B; ++b) {
        if (idx[b] < 0 || idx[b] >= N || pool_len[idx[b]] < 1 || pool_len[idx[b]] > S)
            return 2;
        for (int c = 0; c < b; ++c)
            if (idx[c] == idx[b])
                return 2;
        if (pool_len[idx[b]] > W)
            W = pool_len[idx[b]];
    }
    const int64_t row = (int64_t)D * elt_bytes, slab = row * S;
    for (int l = 0; l < L; ++l)
        for (int c = 0; c < 2; ++c)
            for (int b = 0; b < B; ++b)
                for (int h = 0; h < H; ++h) {
                    const int n = idx[b];
                    const int64_t len = pool_len[n], pad = W - len;
                    const uint8_t *src = (const uint8_t *)pool + ((((int64_t)l * 2 + c) * N + n) * H + h) * slab;
                    uint8_t *dst = (uint8_t *)batch + ((((int64_t)l * 2 + c) * B + b) * H + h) * slab;
                    memcpy(dst + pad * row, src, (size_t)((len - 1) * row));
                }
    for (int b = 0; b < B; ++b) {
        len_out[b] = pool_len[idx[b]];
        pad_out[b] = (int32_t)(W - pool_len[idx[b]]);
    }
    *width_out = (int32_t)W;
    return 0;
}

/* Unpad: the batch slab (l, c, b, h)'s rows pad[b] .. pad[b] + len[b] - 2 go
   back to slot 0 of the pool slab (l, c, idx[b], h), and pool_len[idx[b]] =
   len[b]; no other pool byte changes.  Returns 0, or 2 for a bad or repeated
   index, a length < 1 or a run past S (nothing written). */
int oracle_unpad_scatter(const void *batch, void *pool, int elt_bytes, int L, int N, int B, int H, int S, int D,
                         const int32_t *idx, const int32_t *len, const int32_t *pad, int32_t *pool_len)
{
    for (int b = 0; b < B; ++b) {
        if (idx[b] < 0 || idx[b] >= N || len[b] < 1 || pad[b] < 0 || (int64_t)pad[b] + len[b] - 1 > S)
            return 2;
        for (int c = 0; c < b; ++c)
            if (idx[c] == idx[b])
                return 2;
    }
    const int64_t row = (int64_t)D * elt_bytes, slab = row * S;
    for (int l = 0; l < L; ++l)
        for (int c = 0; c < 2; ++c)
            for (int b = 0; b < B; ++b)
                for (int h = 0; h < H; ++h) {
                    const int n = idx[b];
                    const uint8_t *src = (const uint8_t *)batch + ((((int64_t)l * 2 + c) * B + b) * H + h) * slab;
                    uint8_t *dst = (uint8_t *)pool + ((((int64_t)l * 2 + c) * N + n) * H + h) * slab;
                    memcpy(dst, src + (int64_t)pad[b] * row, (size_t)(((int64_t)len[b] - 1) * row));
                }
    for (int b = 0; b < B; ++b)
        pool_len[idx[b]] = len[b];
    return 0;
}
