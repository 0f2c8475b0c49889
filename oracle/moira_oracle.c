/*
 * moira_oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, fp64 CPU restatement of what the MOIRA sparse-decode hot
 * path computes.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load this library; the product path (the CUDA
 * library) never calls it and shares no code, header or table with it.
 *
 * Sources (the method is described only in prose, so every step below is the
 * plainest reading of that prose; readings are listed beside each function):
 *   [MOIRA]  "MOIRA: Mass-Oriented Indexing with Ragged Attention for
 *            Long-Context Decoding" (arXiv 2610.04313), abstract: at every
 *            decode step and for each request, layer and KV head, the fewest
 *            KV-cache pages whose estimated share of the attention adds up to
 *            gamma are picked, and attention reads only those pages.
 *   [FFD]    "Faster Flash Decoding" (FFD, arXiv 2609.00097; the page is a
 *            Chinese translation), section 2 (related work): metadata
 *            estimators summarise a block by its mean vector (Quest/SparQ);
 *            section 1 and figure 1: top-p selection needs a global softmax to
 *            form the cumulative probability, top-k keeps a fixed budget, and
 *            top-delta keeps the blocks within a relative threshold of the
 *            local maximum.
 *
 * The estimator is not fixed by the pages; this oracle and the CUDA library
 * both use the same stated choice: a page's summary is the mean of its keys,
 * stored as bf16; its score for query head h is sm_scale * q_h . kbar; the
 * page mass is the average over the GQA group of the per-head softmax over
 * the full pages.
 *
 * Every floating-point step is fp64; bf16 inputs are widened exactly.
 * Nothing here is blocked, fused or reordered beyond the definitions.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- bf16 <-> double ---------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (ties to even), in one rounding step.
 * bf16 carries 8 significant bits; normal numbers have exponent >= -126 and
 * below that the spacing stays at 2^-133 (subnormals). */
static uint16_t double_to_bf16_rne(double x)
{
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isinf(a)) return sign | 0x7F80;
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1) */
    int unbiased = e - 1;               /* a = 1.xxx * 2^unbiased */
    int quantum = (unbiased >= -126 ? unbiased : -126) - 7;
    double r = nearbyint(ldexp(a, -quantum));   /* ties to even */
    double v = ldexp(r, quantum);               /* exact */
    if (v > 0x1.FEp127) return sign | 0x7F80;   /* beyond the largest finite bf16 */
    float fv = (float)v;                        /* exact: v has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &fv, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* Exposed so the tests can pin the rounding helper on its own. */
uint16_t oracle_round_bf16(double x) { return double_to_bf16_rne(x); }

/* ---- page summaries ----------------------------------------------------- */

/* Summary of each (page, KV head) block: the mean of its S key vectors
 * ([FFD] section 2: "mean vectors" as block metadata), summed in fp64 in token
 * order and rounded once to bf16.
 *   k_blocks : [n_blocks][S][d] bf16 bit patterns
 *   summ_out : [n_blocks][d]    bf16 bit patterns */
void oracle_summaries(const uint16_t *k_blocks, int64_t n_blocks, int32_t S,
                      int32_t d, uint16_t *summ_out)
{
    for (int64_t b = 0; b < n_blocks; ++b) {
        for (int32_t i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int32_t t = 0; t < S; ++t)
                acc += bf16_to_double(k_blocks[((size_t)b * S + t) * d + i]);
            summ_out[(size_t)b * d + i] = double_to_bf16_rne(acc / (double)S);
        }
    }
}

/* ---- low-bit page summaries ------------------------------------------- */

/* The same mean-key summary stored in `bits` bits per element, after the
 * low-bit key "thumbnails" of "Faster Flash Decoding" (section 3.1: a
 * symmetric mid-rise quantiser, which has no zero level, so every element
 * keeps its sign).  Applied here to the page's mean key, not to each token:
 *   mean_i = (1/S) sum_t K[t][i]            fp64, token order (no bf16 rounding)
 *   a      = max_i |mean_i|
 *   step   = a / (2^(bits-1) - 1/2), rounded once to fp32
 *   code_i = floor(mean_i / step), clamped to [-2^(bits-1), 2^(bits-1) - 1]
 *   value  = (code_i + 1/2) * step
 * so the outermost levels sit at +-a.  A block with a non-finite mean element,
 * with a == 0 or with a step that rounds to 0 gets step 0 and codes 0 (value
 * 0).  bits is 8 or 2.
 *   k_blocks  : [n_blocks][S][d] bf16 bit patterns
 *   codes_out : [n_blocks][d]    one code per element (unpacked)
 *   step_out  : [n_blocks]       fp32 step */
void oracle_summaries_lowbit(const uint16_t *k_blocks, int64_t n_blocks, int32_t S, int32_t d,
                             int32_t bits, int8_t *codes_out, float *step_out)
{
    const double half_levels = ldexp(1.0, bits - 1);            /* 2^(bits-1) */
    double *mean = (double *)malloc(sizeof(double) * (size_t)d);
    for (int64_t b = 0; b < n_blocks; ++b) {
        double a = 0.0;
        int finite = 1;
        for (int32_t i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int32_t t = 0; t < S; ++t)
                acc += bf16_to_double(k_blocks[((size_t)b * S + t) * d + i]);
            mean[i] = acc / (double)S;
            if (!isfinite(mean[i])) finite = 0;
            else if (fabs(mean[i]) > a) a = fabs(mean[i]);
        }
        float step = finite ? (float)(a / (half_levels - 0.5)) : 0.0f;
        step_out[b] = step;
        for (int32_t i = 0; i < d; ++i) {
            double c = 0.0;
            if (step > 0.0f) {
                c = floor(mean[i] / (double)step);
                if (c < -half_levels) c = -half_levels;
                if (c > half_levels - 1.0) c = half_levels - 1.0;
            }
            codes_out[(size_t)b * d + i] = (int8_t)c;
        }
    }
    free(mean);
}

/* The value a low-bit summary stands for (exact in fp64). */
static double lowbit_value(int8_t code, float step)
{
    return ((double)code + 0.5) * (double)step;
}

/* ---- estimated page mass ------------------------------------------------ */

/* Scores and masses for one (request, KV head) unit.
 *   q_group : [G][d] bf16, the G query heads that share this KV head
 *   summ    : [F][d] bf16, summaries of the F full pages in logical order
 *   scores  : [G][F] out (nullable): s_{h,p} = sm_scale * q_h . kbar_p
 *   mass    : [F] out: m_p = (1/G) sum_h softmax_p(s_{h,.})
 * The softmax runs over the full pages only (the partial tail page has no
 * summary until it fills). */
void oracle_page_mass(const uint16_t *q_group, const uint16_t *summ, int32_t G,
                      int32_t F, int32_t d, double sm_scale, double *scores,
                      double *mass)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)(F > 0 ? F : 1));
    for (int32_t p = 0; p < F; ++p) mass[p] = 0.0;
    for (int32_t h = 0; h < G; ++h) {
        double smax = -INFINITY;
        for (int32_t p = 0; p < F; ++p) {
            double dot = 0.0;
            for (int32_t i = 0; i < d; ++i)
                dot += bf16_to_double(q_group[(size_t)h * d + i]) *
                       bf16_to_double(summ[(size_t)p * d + i]);
            s[p] = sm_scale * dot;
            if (scores) scores[(size_t)h * F + p] = s[p];
            if (s[p] > smax) smax = s[p];
        }
        double z = 0.0;
        for (int32_t p = 0; p < F; ++p) z += exp(s[p] - smax);
        for (int32_t p = 0; p < F; ++p) mass[p] += exp(s[p] - smax) / z / (double)G;
    }
    free(s);
}

/* ---- coverage rule ------------------------------------------------------ */

typedef struct { double m; int32_t p; } mass_idx;

/* Order of the coverage rule: larger mass first; equal masses by lower
 * logical page index. */
static int by_mass_desc_then_index(const void *a, const void *b)
{
    const mass_idx *x = (const mass_idx *)a, *y = (const mass_idx *)b;
    if (x->m > y->m) return -1;
    if (x->m < y->m) return 1;
    return (x->p > y->p) - (x->p < y->p);
}

/* [MOIRA] abstract: pick the fewest pages whose estimated mass adds up to
 * gamma.  Sorting by mass and taking the shortest prefix whose running
 * sum is >= gamma gives a smallest such set (any k pages have no more mass
 * than the k largest).  gamma >= 1 keeps every page.  If rounding keeps the
 * running sum below gamma, every page is kept.
 *   mass      : [F]
 *   keep      : [F] out, 1 for kept pages
 *   order     : [F] out (nullable), logical indices in rule order
 *   cum       : [F] out (nullable), running sums in rule order
 * Returns the number of kept pages. */
int32_t oracle_cover(const double *mass, int32_t F, double gamma,
                     uint8_t *keep, int32_t *order, double *cum)
{
    mass_idx *v = (mass_idx *)malloc(sizeof(mass_idx) * (size_t)(F > 0 ? F : 1));
    for (int32_t p = 0; p < F; ++p) { v[p].m = mass[p]; v[p].p = p; }
    qsort(v, (size_t)F, sizeof(mass_idx), by_mass_desc_then_index);
    int32_t k = F;
    double run = 0.0;
    for (int32_t i = 0; i < F; ++i) {
        run += v[i].m;
        if (order) order[i] = v[i].p;
        if (cum) cum[i] = run;
        if (k == F && gamma < 1.0 && run >= gamma) k = i + 1;
    }
    for (int32_t p = 0; p < F; ++p) keep[p] = 0;
    for (int32_t i = 0; i < k; ++i) keep[v[i].p] = 1;
    free(v);
    return k;
}

/* [FFD] section 1, figure 1 (a): a fixed budget keeps the k pages of largest
 * estimated mass, equal masses by lower logical index (the coverage rule's
 * order).  k >= F keeps every page; k <= 0 keeps none.
 *   keep : [F] out, 1 for kept pages
 * Returns the number of kept pages. */
int32_t oracle_topk(const double *mass, int32_t F, int32_t k, uint8_t *keep)
{
    mass_idx *v = (mass_idx *)malloc(sizeof(mass_idx) * (size_t)(F > 0 ? F : 1));
    for (int32_t p = 0; p < F; ++p) { v[p].m = mass[p]; v[p].p = p; }
    qsort(v, (size_t)F, sizeof(mass_idx), by_mass_desc_then_index);
    int32_t n = k < 0 ? 0 : (k > F ? F : k);
    for (int32_t p = 0; p < F; ++p) keep[p] = 0;
    for (int32_t i = 0; i < n; ++i) keep[v[i].p] = 1;
    free(v);
    return n;
}

/* [FFD] section 1, figure 1 (c) and its list of contributions: top-delta keeps
 * the blocks whose estimated contribution is within a relative threshold delta
 * of the local maximum.  The formula itself is cut from the page; the reading
 * taken: keep page p when mass_p >= delta * max_q mass_q (the same estimated
 * masses as the coverage rule, the maximum over the unit's full pages).
 * delta <= 0 keeps every page.
 *   keep : [F] out, 1 for kept pages
 * Returns the number of kept pages. */
int32_t oracle_topdelta(const double *mass, int32_t F, double delta, uint8_t *keep)
{
    double mx = 0.0;
    for (int32_t p = 0; p < F; ++p)
        if (mass[p] > mx) mx = mass[p];
    const double thr = delta * mx;
    int32_t n = 0;
    for (int32_t p = 0; p < F; ++p) {
        keep[p] = mass[p] >= thr;
        n += keep[p];
    }
    return n;
}

/* One unit's selection: estimator + coverage + the partial tail page.
 *   summ_pool : [*][Hkv][d] bf16 summaries by physical page; page_row maps
 *               logical page p to its physical page
 *   seq_len   : tokens of the request; F = seq_len / S full pages, and a tail
 *               page (logical index F) when seq_len % S != 0.  The tail is
 *               always kept (it has no summary yet) and, being the highest
 *               logical index, is the last entry.
 *   list_out  : [F + 1] out, kept logical page indices, ascending
 *   mass/order/cum : optional [F] outputs as in the functions above
 * Returns the list length. */
int32_t oracle_select_unit(const uint16_t *q_group, const uint16_t *summ_pool,
                           int32_t Hkv, int32_t j, const int32_t *page_row,
                           int32_t seq_len, int32_t S, int32_t G, int32_t d,
                           double gamma, double sm_scale, int32_t *list_out,
                           double *mass_out, int32_t *order_out, double *cum_out)
{
    int32_t F = seq_len / S, T = (seq_len % S) != 0;
    int32_t n = 0;
    if (gamma >= 1.0 || F == 0) {
        for (int32_t p = 0; p < F + T; ++p) list_out[n++] = p;
        return n;
    }
    uint16_t *summ = (uint16_t *)calloc((size_t)F * d, sizeof(uint16_t));
    for (int32_t p = 0; p < F; ++p)
        memcpy(summ + (size_t)p * d,
               summ_pool + ((size_t)page_row[p] * Hkv + j) * d, sizeof(uint16_t) * d);
    double *mass = (double *)malloc(sizeof(double) * (size_t)F);
    uint8_t *keep = (uint8_t *)malloc((size_t)F);
    oracle_page_mass(q_group, summ, G, F, d, sm_scale, NULL, mass);
    oracle_cover(mass, F, gamma, keep, order_out, cum_out);
    for (int32_t p = 0; p < F; ++p)
        if (keep[p]) list_out[n++] = p;
    if (T) list_out[n++] = F;
    if (mass_out) memcpy(mass_out, mass, sizeof(double) * (size_t)F);
    free(summ);
    free(mass);
    free(keep);
    return n;
}

/* oracle_select_unit with the rule chosen by `rule`: 0 = coverage (param =
 * gamma), 1 = top-k (param = k, a whole number), 2 = top-delta (param =
 * delta).  The estimator, the tail page and the list order are the same for
 * every rule.  Returns the list length. */
int32_t oracle_select_unit_rule(const uint16_t *q_group, const uint16_t *summ_pool,
                                int32_t Hkv, int32_t j, const int32_t *page_row,
                                int32_t seq_len, int32_t S, int32_t G, int32_t d,
                                int32_t rule, double param, double sm_scale,
                                int32_t *list_out)
{
    if (rule == 0)
        return oracle_select_unit(q_group, summ_pool, Hkv, j, page_row, seq_len, S, G, d,
                                  param, sm_scale, list_out, NULL, NULL, NULL);
    int32_t F = seq_len / S, T = (seq_len % S) != 0;
    int32_t n = 0;
    if (F == 0) {
        for (int32_t p = 0; p < T; ++p) list_out[n++] = p;
        return n;
    }
    uint16_t *summ = (uint16_t *)calloc((size_t)F * d, sizeof(uint16_t));
    for (int32_t p = 0; p < F; ++p)
        memcpy(summ + (size_t)p * d,
               summ_pool + ((size_t)page_row[p] * Hkv + j) * d, sizeof(uint16_t) * d);
    double *mass = (double *)malloc(sizeof(double) * (size_t)F);
    uint8_t *keep = (uint8_t *)malloc((size_t)F);
    oracle_page_mass(q_group, summ, G, F, d, sm_scale, NULL, mass);
    if (rule == 1) oracle_topk(mass, F, (int32_t)param, keep);
    else oracle_topdelta(mass, F, param, keep);
    for (int32_t p = 0; p < F; ++p)
        if (keep[p]) list_out[n++] = p;
    if (T) list_out[n++] = F;
    free(summ);
    free(mass);
    free(keep);
    return n;
}

/* Scores and masses of one unit from low-bit summaries: oracle_page_mass
 * with kbar_p[i] = (code + 1/2) * step.
 *   codes : [F][d] (logical order), steps : [F] */
void oracle_page_mass_lowbit(const uint16_t *q_group, const int8_t *codes, const float *steps,
                             int32_t G, int32_t F, int32_t d, double sm_scale, double *scores,
                             double *mass)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)(F > 0 ? F : 1));
    for (int32_t p = 0; p < F; ++p) mass[p] = 0.0;
    for (int32_t h = 0; h < G; ++h) {
        double smax = -INFINITY;
        for (int32_t p = 0; p < F; ++p) {
            double dot = 0.0;
            for (int32_t i = 0; i < d; ++i)
                dot += bf16_to_double(q_group[(size_t)h * d + i]) *
                       lowbit_value(codes[(size_t)p * d + i], steps[p]);
            s[p] = sm_scale * dot;
            if (scores) scores[(size_t)h * F + p] = s[p];
            if (s[p] > smax) smax = s[p];
        }
        double z = 0.0;
        for (int32_t p = 0; p < F; ++p) z += exp(s[p] - smax);
        for (int32_t p = 0; p < F; ++p) mass[p] += exp(s[p] - smax) / z / (double)G;
    }
    free(s);
}

/* One unit's selection from low-bit summaries under `rule` (0 = coverage,
 * 1 = top-k, 2 = top-delta, as oracle_select_unit_rule): the estimator reads
 * (code + 1/2) * step instead of the bf16 mean; the tail page and the list
 * order are unchanged.
 *   codes_pool : [*][Hkv][d] by physical page, steps_pool : [*][Hkv]
 *   mass_out   : [F] out (nullable; left untouched when no estimate is made)
 * Returns the list length. */
int32_t oracle_select_unit_lowbit(const uint16_t *q_group, const int8_t *codes_pool,
                                  const float *steps_pool, int32_t Hkv, int32_t j,
                                  const int32_t *page_row, int32_t seq_len, int32_t S, int32_t G,
                                  int32_t d, int32_t rule, double param, double sm_scale,
                                  int32_t *list_out, double *mass_out)
{
    int32_t F = seq_len / S, T = (seq_len % S) != 0;
    int32_t n = 0;
    if (F == 0 || (rule == 0 && param >= 1.0)) {
        for (int32_t p = 0; p < F + T; ++p) list_out[n++] = p;
        return n;
    }
    int8_t *codes = (int8_t *)malloc((size_t)F * d);
    float *steps = (float *)malloc(sizeof(float) * (size_t)F);
    for (int32_t p = 0; p < F; ++p) {
        size_t blk = (size_t)page_row[p] * Hkv + j;
        memcpy(codes + (size_t)p * d, codes_pool + blk * d, (size_t)d);
        steps[p] = steps_pool[blk];
    }
    double *mass = (double *)malloc(sizeof(double) * (size_t)F);
    uint8_t *keep = (uint8_t *)malloc((size_t)F);
    oracle_page_mass_lowbit(q_group, codes, steps, G, F, d, sm_scale, NULL, mass);
    if (rule == 0) oracle_cover(mass, F, param, keep, NULL, NULL);
    else if (rule == 1) oracle_topk(mass, F, (int32_t)param, keep);
    else oracle_topdelta(mass, F, param, keep);
    for (int32_t p = 0; p < F; ++p)
        if (keep[p]) list_out[n++] = p;
    if (T) list_out[n++] = F;
    if (mass_out) memcpy(mass_out, mass, sizeof(double) * (size_t)F);
    free(codes);
    free(steps);
    free(mass);
    free(keep);
    return n;
}

/* ---- exact attention over the kept tokens ------------------------------ */

/* Softmax attention of the G query heads over the tokens of the listed pages.
 *   k_pool, v_pool : [*][Hkv][S][d] bf16 by physical page; page_row maps
 *                    logical page p to its physical page
 *   list           : [len] logical page indices
 *   seq_len        : page p holds tokens [p*S, min((p+1)*S, seq_len))
 *   out            : [G][d]; zero when no token is listed */
void oracle_attend_unit(const uint16_t *q_group, const uint16_t *k_pool,
                        const uint16_t *v_pool, int32_t Hkv, int32_t j,
                        const int32_t *page_row, const int32_t *list,
                        int32_t len, int32_t seq_len, int32_t S, int32_t G,
                        int32_t d, double sm_scale, double *out)
{
    int64_t ntok = 0;
    for (int32_t e = 0; e < len; ++e) {
        int64_t lo = (int64_t)list[e] * S, hi = lo + S;
        if (hi > seq_len) hi = seq_len;
        if (hi > lo) ntok += hi - lo;
    }
    size_t blk = (size_t)S * d;
    double *logit = (double *)malloc(sizeof(double) * (size_t)(ntok > 0 ? ntok : 1));
    for (int32_t h = 0; h < G; ++h) {
        double *o = out + (size_t)h * d;
        for (int32_t i = 0; i < d; ++i) o[i] = 0.0;
        if (ntok == 0) continue;
        double lmax = -INFINITY;
        int64_t x = 0;
        for (int32_t e = 0; e < len; ++e) {
            int64_t p = list[e];
            const uint16_t *kb = k_pool + ((size_t)page_row[p] * Hkv + j) * blk;
            for (int32_t t = 0; t < S && p * S + t < seq_len; ++t) {
                double dot = 0.0;
                for (int32_t i = 0; i < d; ++i)
                    dot += bf16_to_double(q_group[(size_t)h * d + i]) *
                           bf16_to_double(kb[(size_t)t * d + i]);
                logit[x] = sm_scale * dot;
                if (logit[x] > lmax) lmax = logit[x];
                ++x;
            }
        }
        double z = 0.0;
        x = 0;
        for (int32_t e = 0; e < len; ++e) {
            int64_t p = list[e];
            const uint16_t *vb = v_pool + ((size_t)page_row[p] * Hkv + j) * blk;
            for (int32_t t = 0; t < S && p * S + t < seq_len; ++t) {
                double w = exp(logit[x] - lmax);
                z += w;
                for (int32_t i = 0; i < d; ++i)
                    o[i] += w * bf16_to_double(vb[(size_t)t * d + i]);
                ++x;
            }
        }
        for (int32_t i = 0; i < d; ++i) o[i] /= z;
    }
    free(logit);
}

/* ---- one decode-attention step over a pooled KV cache ------------------ */

/* Selection + attention for n_layers layers of a paged KV cache, every
 * (layer, request, KV head) unit independently (OpenMP over units).
 * Layouts (bf16 unless stated):
 *   q          : [n_layers][B][Hq][d]
 *   summ       : [n_layers][P][Hkv][d]      summaries of the physical pages
 *   k_pool     : [n_layers][P][Hkv][S][d], v_pool likewise
 *   page_table : int32 [B][max_pages], logical -> physical page
 *   seq_lens   : int32 [B]
 *   lengths    : int32 out [n_layers][B][Hkv]
 *   out        : double out [n_layers][B][Hq][d]
 * Query head h reads KV head h / G (G = Hq / Hkv).
 * Returns the number of threads used. */
int32_t oracle_decode_step(const uint16_t *q, const uint16_t *summ,
                           const uint16_t *k_pool, const uint16_t *v_pool,
                           const int32_t *page_table, const int32_t *seq_lens,
                           int32_t n_layers, int32_t B, int32_t Hq, int32_t Hkv,
                           int32_t d, int32_t S, int64_t P, int32_t max_pages,
                           double gamma, double sm_scale, int32_t *lengths,
                           double *out, int32_t n_threads)
{
    int32_t G = Hq / Hkv;
    int64_t units = (int64_t)n_layers * B * Hkv;
    int32_t used = 1;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
    {
#pragma omp single
        used = omp_get_num_threads();
    }
#else
    (void)n_threads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t u = 0; u < units; ++u) {
        int32_t l = (int32_t)(u / ((int64_t)B * Hkv));
        int32_t r = (int32_t)((u / Hkv) % B);
        int32_t j = (int32_t)(u % Hkv);
        int32_t L = seq_lens[r];
        const int32_t *row = page_table + (size_t)r * max_pages;
        const uint16_t *qg = q + (((size_t)l * B + r) * Hq + (size_t)j * G) * d;
        size_t lay_pages = (size_t)P * Hkv;
        int32_t *list = (int32_t *)malloc(sizeof(int32_t) * (size_t)(L / S + 2));
        int32_t len = oracle_select_unit(qg, summ + (size_t)l * lay_pages * d, Hkv, j,
                                         row, L, S, G, d, gamma, sm_scale, list,
                                         NULL, NULL, NULL);
        lengths[u] = len;
        oracle_attend_unit(qg, k_pool + (size_t)l * lay_pages * S * d,
                           v_pool + (size_t)l * lay_pages * S * d, Hkv, j, row,
                           list, len, L, S, G, d, sm_scale,
                           out + (((size_t)l * B + r) * Hq + (size_t)j * G) * d);
        free(list);
    }
    return used;
}
