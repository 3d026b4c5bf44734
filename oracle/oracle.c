/*
 * oracle.c -- plain fp64 CPU restatement of attention-score-driven prompt
 * KV-cache compression (SnapKV observation-window scoring, ZigZagKV MBA /
 * LMBA layer budgets, per-head top-K, K/V compaction, ThinK key-channel
 * magnitude pruning).
 *
 * TEST INFRASTRUCTURE ONLY.  The test-suite, the package smoke check and the
 * benchmark's CPU-baseline leg call this file; the CUDA library neither links
 * nor calls it and the two share no code.  It is deliberately slow and
 * direct: one loop per definition, library qsort for sorting, no blocking.
 *
 * Sources (page title, section):
 *  [SNAP]       ZigZagKV/SnapKV blog post "ZigZagKV, KVCache 80% compression
 *               near-lossless" (dis.qidao123.com), section "SnapKV": the last
 *               window's queries score every prefix token, the scores are
 *               averaged over the window rows per head, each head keeps its
 *               top-K prefix tokens plus every token of the last window.
 *  [ZZ-MBA]     same post, section "ZigZagKV's new observations": MBA is the
 *               fewest KV entries whose attention reaches 90% of the total
 *               attention score over the n tokens in the cache; LMBA is the
 *               mean of MBA over the heads of a layer.
 *  [ZZ-ALLOC]   same post, section "ZigZagKV space allocation": the total
 *               budget is split across layers in proportion to LMBA, with a
 *               minimum size reserved for every layer.
 *  [ZZ-SEL]     same post, section "ZigZagKV token selection": selection is
 *               SnapKV's, with each head's K set by its quota.
 *  [THINK-ATT]  "ThinK: Thinner Key Cache by Query-Driven Pruning", section
 *               "Method details", attention equation softmax(Q K^T / sqrt(D)) V.
 *  [THINK-MAG]  same page, "Magnitude-based pruning": M_{n,d} = ||K[n,:,d]||_p;
 *               keep floor((1-lambda) D) channels per head, Top_T of M.
 *  [THINK-IMPL] same page, "Implementation of THINK": recent tokens are not
 *               pruned.
 *  [THINK-QD]   same page, "Greedy algorithm" and "Observation window":
 *               channel score = Frobenius norm of Q[-S_obs:, j] K[:, j]^T.
 *  [THINK-V]    same page, appendix "Value cache pruning strategy": value
 *               channel score = norm of column j of softmax(Q[-S_obs:] K^T /
 *               sqrt(D)) V; keep the top T channels.
 *  [ZZ-HEAD]    ZigZagKV post: memory per attention head should follow the
 *               tokens that head needs; each head's K follows its quota.
 *  [KEYF]       "Keyformer: KV Cache reduction through key tokens selection"
 *               (moyutianzun.com): Gumbel noise on the logits, temperature
 *               softmax, recent w tokens plus the top k - w older ones.
 *  [THRESH]     ZigZagKV post, "SnapKV": scores above a threshold mark the
 *               important tokens; "NVIDIA AI presents KVzap" (kiadev.net):
 *               low-score entries are dropped, a sliding window of recent
 *               tokens is kept.
 *
 * Readings where the pages are silent or garbled:
 *  - GQA: query head h belongs to KV head h / G (G = H_q / H_kv); the score
 *    of a KV head is the mean over its G query heads and W window rows.
 *  - Causal mask inside the window: window row i sits at position P+i
 *    (P = T-W) and sees keys 0..P+i.
 *  - MBA is taken per KV head over all T scores (prefix and window); the
 *    mass is exact fixed point u_j = floor(c_j * 2^56) and "reaches" means
 *    den * (sum of the m largest u) >= num * (sum of all u).
 *  - Budgets count prefix tokens only; the W window rows are always kept.
 *  - Split: B_l = floor + largest-remainder share of (total - L*floor) by
 *    S_l = sum_k MBA_{l,k} (LMBA up to the common factor H_kv), ties to the
 *    lower layer; budgets above the prefix length P are capped and the excess
 *    is re-split over the uncapped layers until none exceeds P.
 *  - Top-K ties go to the lower token index; kept rows are written in
 *    ascending position order, then the window rows in order.
 *  - ThinK uses p = 2 over the kept prefix rows only (window rows stay
 *    full width); channel ties go to the lower channel index.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int32_t n_layers, n_q_heads, n_kv_heads, head_dim, seq_len, window;
    int32_t dtype; /* 0: fp32, 1: bf16 */
} ora_shape;

int ora_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void ora_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Exact widening of one stored element to fp64. bf16 is the top half of an
 * IEEE binary32, so shifting it up 16 bits gives the identical value. */
static double ora_elem(const void *base, int64_t i, int dtype)
{
    if (dtype == 0) return (double)((const float *)base)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static int ora_shape_ok(const ora_shape *s)
{
    if (!s) return 0;
    if (s->n_layers < 1 || s->n_q_heads < 1 || s->n_kv_heads < 1) return 0;
    if (s->n_q_heads % s->n_kv_heads) return 0;
    if (s->head_dim < 1 || s->window < 1 || s->seq_len <= s->window) return 0;
    if (s->dtype != 0 && s->dtype != 1) return 0;
    return 1;
}

/* ---------------------------------------------------------------------------
 * a1. Observation-window score of one (layer, KV head)   [SNAP], [THINK-ATT]
 *
 * For every query head h of the group and window row i (position t = P+i):
 *   x_j = (q_{h,i} . k_j) / sqrt(D)              for j = 0..t
 *   p_j = exp(x_j - max x) / sum_{j'<=t} exp(x_j' - max x)
 *   c_j += p_j / (G * W)
 * so c is the mean attention row over the G*W window queries; c sums to 1.
 * ------------------------------------------------------------------------- */
int ora_score_unit(const ora_shape *s, const void *q, const void *k,
                   int layer, int kv_head, double *c)
{
    if (!ora_shape_ok(s) || layer < 0 || layer >= s->n_layers ||
        kv_head < 0 || kv_head >= s->n_kv_heads)
        return -1;
    const int64_t D = s->head_dim, T = s->seq_len, W = s->window;
    const int64_t Hq = s->n_q_heads, Hkv = s->n_kv_heads, G = Hq / Hkv;
    const int64_t P = T - W;
    const double rows = (double)(G * W);
    const double root_d = sqrt((double)D);
    const int64_t k_base = ((int64_t)layer * Hkv + kv_head) * T * D;
    double *x = (double *)malloc(sizeof(double) * (size_t)T);
    double *qr = (double *)malloc(sizeof(double) * (size_t)D);
    if (!x || !qr) { free(x); free(qr); return -2; }
    for (int64_t j = 0; j < T; ++j) c[j] = 0.0;
    for (int64_t g = 0; g < G; ++g) {
        const int64_t h = (int64_t)kv_head * G + g;
        for (int64_t i = 0; i < W; ++i) {
            const int64_t q_base = (((int64_t)layer * Hq + h) * W + i) * D;
            for (int64_t d = 0; d < D; ++d) qr[d] = ora_elem(q, q_base + d, s->dtype);
            const int64_t t = P + i;
            double mu = -INFINITY;
            for (int64_t j = 0; j <= t; ++j) {
                double dot = 0.0;
                for (int64_t d = 0; d < D; ++d)
                    dot += qr[d] * ora_elem(k, k_base + j * D + d, s->dtype);
                x[j] = dot / root_d;
                if (x[j] > mu) mu = x[j];
            }
            double z = 0.0;
            for (int64_t j = 0; j <= t; ++j) {
                x[j] = exp(x[j] - mu);
                z += x[j];
            }
            for (int64_t j = 0; j <= t; ++j) c[j] += x[j] / z / rows;
        }
    }
    free(x);
    free(qr);
    return 0;
}

/* a1 over all (layer, KV head) units; scores laid out [L][H_kv][T]. */
int ora_score(const ora_shape *s, const void *q, const void *k, double *scores)
{
    if (!ora_shape_ok(s)) return -1;
    const int64_t units = (int64_t)s->n_layers * s->n_kv_heads;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t u = 0; u < units; ++u) {
        int l = (int)(u / s->n_kv_heads), h = (int)(u % s->n_kv_heads);
        if (ora_score_unit(s, q, k, l, h, scores + u * s->seq_len) != 0) bad = 1;
    }
    return bad ? -2 : 0;
}

/* ---------------------------------------------------------------------------
 * a2. MBA of one head                                        [ZZ-MBA]
 *
 * Mass in exact fixed point: u_j = floor(c_j * 2^56) (c_j in [0,1]).  With the
 * u sorted in descending order and U = sum u, MBA is the smallest m with
 *   den * sum_{r<m} u_(r) >= num * U        (num/den = 9/10 on the pages).
 * Returns -1 for a score outside [0,1] or NaN.
 * ------------------------------------------------------------------------- */
static int ora_cmp_u64_desc(const void *a, const void *b)
{
    uint64_t x = *(const uint64_t *)a, y = *(const uint64_t *)b;
    return (x < y) - (x > y);
}

int64_t ora_mba(int64_t n, const double *c, uint32_t num, uint32_t den)
{
    if (n < 0 || den == 0 || num > den) return -1;
    uint64_t *u = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(n ? n : 1));
    if (!u) return -2;
    for (int64_t j = 0; j < n; ++j) {
        if (!(c[j] >= 0.0 && c[j] <= 1.0)) { free(u); return -1; }
        u[j] = (uint64_t)floor(ldexp(c[j], 56));
    }
    qsort(u, (size_t)n, sizeof(uint64_t), ora_cmp_u64_desc);
    unsigned __int128 total = 0;
    for (int64_t j = 0; j < n; ++j) total += u[j];
    const unsigned __int128 need = (unsigned __int128)num * total;
    unsigned __int128 run = 0;
    int64_t m = 0;
    while ((unsigned __int128)den * run < need) {
        run += u[m];
        ++m;
    }
    free(u);
    return m;
}

int ora_mba_all(const ora_shape *s, const double *scores, uint32_t num, uint32_t den,
                int32_t *mba)
{
    if (!ora_shape_ok(s)) return -1;
    const int64_t units = (int64_t)s->n_layers * s->n_kv_heads;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t u = 0; u < units; ++u) {
        int64_t m = ora_mba(s->seq_len, scores + u * s->seq_len, num, den);
        if (m < 0) bad = 1;
        mba[u] = (int32_t)m;
    }
    return bad ? -1 : 0;
}

/* Same as ora_mba_all on fp32 scores (widened exactly). */
int ora_mba_all_f32(const ora_shape *s, const float *scores, uint32_t num, uint32_t den,
                    int32_t *mba)
{
    if (!ora_shape_ok(s)) return -1;
    const int64_t n = (int64_t)s->n_layers * s->n_kv_heads * s->seq_len;
    double *c = (double *)malloc(sizeof(double) * (size_t)n);
    if (!c) return -2;
    for (int64_t i = 0; i < n; ++i) c[i] = (double)scores[i];
    int r = ora_mba_all(s, c, num, den, mba);
    free(c);
    return r;
}

/* ---------------------------------------------------------------------------
 * a3. Layer budgets                                          [ZZ-ALLOC]
 *
 * Largest-remainder split of R units over the eligible entries in proportion
 * to w (equal weights if the eligible weights sum to zero).  Each entry gets
 * floor(R w_l / sum w); the units left over go one each to the largest
 * remainders R w_l mod sum w, ties to the lower index.
 * ------------------------------------------------------------------------- */
static void ora_split(int n, const int64_t *w, const unsigned char *eligible,
                      int64_t R, int64_t *add)
{
    int64_t sumw = 0;
    int any = 0;
    for (int l = 0; l < n; ++l)
        if (eligible[l]) { sumw += w[l]; any = 1; }
    for (int l = 0; l < n; ++l) add[l] = 0;
    if (!any || R <= 0) return;
    const int equal = (sumw == 0);
    if (equal)
        for (int l = 0; l < n; ++l) sumw += eligible[l] ? 1 : 0;
    int64_t *rem = (int64_t *)malloc(sizeof(int64_t) * (size_t)n);
    unsigned char *given = (unsigned char *)calloc((size_t)n, 1);
    int64_t handed = 0;
    for (int l = 0; l < n; ++l) {
        rem[l] = -1;
        if (!eligible[l]) continue;
        const __int128 prod = (__int128)R * (equal ? 1 : w[l]);
        add[l] = (int64_t)(prod / sumw);
        rem[l] = (int64_t)(prod % sumw);
        handed += add[l];
    }
    for (int64_t left = R - handed; left > 0; --left) {
        int best = -1;
        for (int l = 0; l < n; ++l)
            if (eligible[l] && !given[l] && (best < 0 || rem[l] > rem[best])) best = l;
        given[best] = 1;
        add[best] += 1;
    }
    free(rem);
    free(given);
}

/* mba: [L][H_kv]; budget: [L].  Returns -1 for invalid arguments. */
int ora_budget(int L, int Hkv, const int32_t *mba, int64_t prefix, int64_t total,
               int64_t floor_, int32_t *budget)
{
    if (L < 1 || Hkv < 1 || prefix < 1 || floor_ < 0 || floor_ > prefix ||
        total < (int64_t)L * floor_)
        return -1;
    if (total >= (int64_t)L * prefix) {
        for (int l = 0; l < L; ++l) budget[l] = (int32_t)prefix;
        return 0;
    }
    int64_t *S = (int64_t *)malloc(sizeof(int64_t) * (size_t)L);
    int64_t *B = (int64_t *)malloc(sizeof(int64_t) * (size_t)L);
    int64_t *add = (int64_t *)malloc(sizeof(int64_t) * (size_t)L);
    unsigned char *elig = (unsigned char *)malloc((size_t)L);
    for (int l = 0; l < L; ++l) {
        S[l] = 0;
        for (int k = 0; k < Hkv; ++k) S[l] += mba[(int64_t)l * Hkv + k];
        elig[l] = 1;
    }
    ora_split(L, S, elig, total - (int64_t)L * floor_, add);
    for (int l = 0; l < L; ++l) B[l] = floor_ + add[l];
    for (;;) {
        int64_t excess = 0;
        for (int l = 0; l < L; ++l)
            if (B[l] > prefix) { excess += B[l] - prefix; B[l] = prefix; }
        if (excess == 0) break;
        for (int l = 0; l < L; ++l) elig[l] = (unsigned char)(B[l] < prefix);
        ora_split(L, S, elig, excess, add);
        for (int l = 0; l < L; ++l) B[l] += add[l];
    }
    for (int l = 0; l < L; ++l) budget[l] = (int32_t)B[l];
    free(S); free(B); free(add); free(elig);
    return 0;
}

/* ---------------------------------------------------------------------------
 * a4. Per-head top-K of the prefix                           [SNAP], [ZZ-SEL]
 *
 * Order the prefix positions by (score descending, position ascending), keep
 * the first min(B, P), and return them in ascending position order.
 * ------------------------------------------------------------------------- */
typedef struct { double v; int64_t j; } ora_item;

static int ora_cmp_item(const void *a, const void *b)
{
    const ora_item *x = (const ora_item *)a, *y = (const ora_item *)b;
    if (x->v != y->v) return (x->v < y->v) ? 1 : -1;
    return (x->j > y->j) - (x->j < y->j);
}

static int ora_cmp_i32(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

static int64_t ora_kept(int64_t budget, int64_t prefix)
{
    return budget < 0 ? 0 : (budget > prefix ? prefix : budget);
}

int64_t ora_topk(int64_t P, const double *c, int64_t B, int32_t *idx)
{
    const int64_t n = ora_kept(B, P);
    ora_item *it = (ora_item *)malloc(sizeof(ora_item) * (size_t)(P ? P : 1));
    if (!it) return -2;
    for (int64_t j = 0; j < P; ++j) { it[j].v = c[j]; it[j].j = j; }
    qsort(it, (size_t)P, sizeof(ora_item), ora_cmp_item);
    for (int64_t r = 0; r < n; ++r) idx[r] = (int32_t)it[r].j;
    qsort(idx, (size_t)n, sizeof(int32_t), ora_cmp_i32);
    free(it);
    return n;
}

/* idx: [L][H_kv][k_max]; entries past the kept count are left untouched. */
int ora_topk_all(const ora_shape *s, const double *scores, const int32_t *budget,
                 int64_t k_max, int32_t *idx)
{
    if (!ora_shape_ok(s)) return -1;
    const int64_t T = s->seq_len, P = T - s->window, Hkv = s->n_kv_heads;
    for (int l = 0; l < s->n_layers; ++l)
        if (ora_kept(budget[l], P) > k_max) return -1;
    const int64_t units = (int64_t)s->n_layers * Hkv;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t u = 0; u < units; ++u) {
        if (ora_topk(P, scores + u * T, budget[u / Hkv], idx + u * k_max) < 0) bad = 1;
    }
    return bad ? -2 : 0;
}

int ora_topk_all_f32(const ora_shape *s, const float *scores, const int32_t *budget,
                     int64_t k_max, int32_t *idx)
{
    if (!ora_shape_ok(s)) return -1;
    const int64_t n = (int64_t)s->n_layers * s->n_kv_heads * s->seq_len;
    double *c = (double *)malloc(sizeof(double) * (size_t)n);
    if (!c) return -2;
    for (int64_t i = 0; i < n; ++i) c[i] = (double)scores[i];
    int r = ora_topk_all(s, c, budget, k_max, idx);
    free(c);
    return r;
}

/* ---------------------------------------------------------------------------
 * Optional: pooling of the prefix scores before top-K              [SNAP]
 *
 * The post pools each head's scores in 1D ("like a Gaussian blur") so that
 * the neighbours of an important token are kept with it; it names neither
 * the kernel's size nor its type.  Reading: an odd kernel k, "same" length
 * over the prefix j in [0,P): mode 0 averages the in-range entries
 * j-k/2 .. j+k/2 (dividing by how many lie inside [0,P)), mode 1 takes
 * their maximum.  Window positions j >= P are copied unchanged (they are
 * always kept and take no part in the ranking).  Output fp64 [L][H_kv][T].
 * ------------------------------------------------------------------------- */
int ora_pool(const ora_shape *s, const double *scores, int32_t kernel, int32_t mode,
             double *pooled)
{
    if (!ora_shape_ok(s) || kernel < 1 || kernel % 2 == 0 || (mode != 0 && mode != 1))
        return -1;
    const int64_t T = s->seq_len, P = T - s->window;
    const int64_t units = (int64_t)s->n_layers * s->n_kv_heads, half = kernel / 2;
#pragma omp parallel for schedule(static)
    for (int64_t u = 0; u < units; ++u) {
        const double *c = scores + u * T;
        double *o = pooled + u * T;
        for (int64_t j = 0; j < T; ++j) {
            if (j >= P) {
                o[j] = c[j];
                continue;
            }
            const int64_t lo = j - half < 0 ? 0 : j - half;
            const int64_t hi = j + half > P - 1 ? P - 1 : j + half;
            double acc = c[lo];
            for (int64_t t = lo + 1; t <= hi; ++t)
                acc = mode == 0 ? acc + c[t] : (c[t] > acc ? c[t] : acc);
            o[j] = mode == 0 ? acc / (double)(hi - lo + 1) : acc;
        }
    }
    return 0;
}

int ora_pool_f32(const ora_shape *s, const float *scores, int32_t kernel, int32_t mode,
                 double *pooled)
{
    if (!ora_shape_ok(s)) return -1;
    const int64_t n = (int64_t)s->n_layers * s->n_kv_heads * s->seq_len;
    double *c = (double *)malloc(sizeof(double) * (size_t)n);
    if (!c) return -2;
    for (int64_t i = 0; i < n; ++i) c[i] = (double)scores[i];
    int r = ora_pool(s, c, kernel, mode, pooled);
    free(c);
    return r;
}

/* ---------------------------------------------------------------------------
 * a5. Compaction                                             [SNAP]
 *
 * Layer l of the output holds [H_kv][n_l + W][D] with n_l = min(B_l, P): the
 * kept prefix rows in ascending position order, then the W window rows.
 * Layers follow each other; layer l starts at row H_kv * sum_{l'<l}(n_l'+W).
 * Returns the number of rows written per tensor, or -1.
 * ------------------------------------------------------------------------- */
int64_t ora_compact_rows(const ora_shape *s, const int32_t *budget)
{
    if (!ora_shape_ok(s)) return -1;
    const int64_t P = (int64_t)s->seq_len - s->window;
    int64_t rows = 0;
    for (int l = 0; l < s->n_layers; ++l)
        rows += (int64_t)s->n_kv_heads * (ora_kept(budget[l], P) + s->window);
    return rows;
}

int64_t ora_compact(const ora_shape *s, const void *src, const int32_t *idx,
                    const int32_t *budget, int64_t k_max, void *out)
{
    if (!ora_shape_ok(s)) return -1;
    const int64_t T = s->seq_len, W = s->window, P = T - W, Hkv = s->n_kv_heads;
    const size_t row_bytes = (size_t)s->head_dim * (s->dtype == 0 ? 4 : 2);
    const unsigned char *in = (const unsigned char *)src;
    unsigned char *o = (unsigned char *)out;
    int64_t row = 0;
    for (int l = 0; l < s->n_layers; ++l) {
        const int64_t n = ora_kept(budget[l], P);
        if (n > k_max) return -1;
        for (int64_t h = 0; h < Hkv; ++h) {
            const int64_t head = (int64_t)l * Hkv + h;
            const int32_t *sel = idx + head * k_max;
            for (int64_t r = 0; r < n + W; ++r) {
                const int64_t t = r < n ? (int64_t)sel[r] : P + (r - n);
                if (t < 0 || t >= T) return -1;
                memcpy(o + (size_t)row * row_bytes, in + (size_t)(head * T + t) * row_bytes,
                       row_bytes);
                ++row;
            }
        }
    }
    return row;
}

/* ---------------------------------------------------------------------------
 * a6. ThinK magnitude channel pruning                        [THINK-MAG]
 *
 * keep = floor((1 - lambda) * D).  Per (layer, KV head): M_d = sum over the
 * n_l kept prefix rows of K_out[r][d]^2 (the squared l2 norm ranks the same
 * channels as the norm), order channels by (M desc, d asc), keep the first
 * `keep`, list them ascending, and copy those channels of the kept prefix
 * rows into K_pruned.  The window rows are left full width [THINK-IMPL].
 * K_pruned layer l holds [H_kv][n_l][keep] starting at element
 * H_kv * keep * sum_{l'<l} n_l'.
 * ------------------------------------------------------------------------- */
int32_t ora_keep_channels(double lambda, int32_t D)
{
    return (int32_t)floor((1.0 - lambda) * (double)D);
}

typedef struct { double m; int32_t d; } ora_chan;

static int ora_cmp_chan(const void *a, const void *b)
{
    const ora_chan *x = (const ora_chan *)a, *y = (const ora_chan *)b;
    if (x->m != y->m) return (x->m < y->m) ? 1 : -1;
    return (x->d > y->d) - (x->d < y->d);
}

int ora_channel_prune(const ora_shape *s, const void *k_out, const int32_t *budget,
                      double lambda, int32_t *chan, double *norms, void *k_pruned)
{
    if (!ora_shape_ok(s)) return -1;
    const int64_t D = s->head_dim, W = s->window, P = (int64_t)s->seq_len - W;
    const int64_t Hkv = s->n_kv_heads, L = s->n_layers;
    const int32_t keep = ora_keep_channels(lambda, (int32_t)D);
    if (keep < 1 || keep > D) return -1;
    const size_t es = s->dtype == 0 ? 4 : 2;
    int64_t *in_row = (int64_t *)malloc(sizeof(int64_t) * (size_t)L);
    int64_t *out_el = (int64_t *)malloc(sizeof(int64_t) * (size_t)L);
    int64_t ir = 0, oe = 0;
    for (int64_t l = 0; l < L; ++l) {
        in_row[l] = ir;
        out_el[l] = oe;
        const int64_t n = ora_kept(budget[l], P);
        ir += Hkv * (n + W);
        oe += Hkv * n * keep;
    }
    const int64_t units = L * Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t u = 0; u < units; ++u) {
        const int64_t l = u / Hkv, h = u % Hkv;
        const int64_t n = ora_kept(budget[l], P);
        const int64_t row0 = in_row[l] + h * (n + W);
        ora_chan *ch = (ora_chan *)malloc(sizeof(ora_chan) * (size_t)D);
        for (int64_t d = 0; d < D; ++d) {
            double m = 0.0;
            for (int64_t r = 0; r < n; ++r) {
                const double x = ora_elem(k_out, (row0 + r) * D + d, s->dtype);
                m += x * x;
            }
            ch[d].m = m;
            ch[d].d = (int32_t)d;
            if (norms) norms[u * D + d] = m;
        }
        qsort(ch, (size_t)D, sizeof(ora_chan), ora_cmp_chan);
        int32_t *sel = chan + u * keep;
        for (int32_t i = 0; i < keep; ++i) sel[i] = ch[i].d;
        qsort(sel, (size_t)keep, sizeof(int32_t), ora_cmp_i32);
        if (k_pruned) {
            const unsigned char *src = (const unsigned char *)k_out;
            unsigned char *dst = (unsigned char *)k_pruned;
            const int64_t o0 = out_el[l] + h * n * keep;
            for (int64_t r = 0; r < n; ++r)
                for (int32_t i = 0; i < keep; ++i)
                    memcpy(dst + (size_t)(o0 + r * keep + i) * es,
                           src + (size_t)((row0 + r) * D + sel[i]) * es, es);
        }
        free(ch);
    }
    free(in_row);
    free(out_el);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Optional: ThinK value-channel pruning (THINKV)               [THINK-V]
 *
 * "ThinK: Thinner Key Cache by Query-Driven Pruning", appendix "Value cache
 * pruning strategy": channel j of a head's value cache scores the norm of
 * column j of the window queries' attention output,
 *   Score_v[j] = || softmax(Q[-S_obs:] K^T / sqrt(D)) V[:, j] ||_F,
 * and only the T channels with the largest scores are kept (T =
 * floor((1-lambda) D), the same count as for keys).
 * Readings: the attention is the window scoring's own (a1): window row i
 * (position P+i) attends to the whole prompt's keys 0..P+i with
 * softmax(q.k / sqrt(D)); with grouped-query attention the output column
 * stacks the G*W window rows of the KV head's query heads (as for the
 * query-driven key criterion); channels are ranked by the squared norm
 * (monotone in the norm, no rounding sqrt), ties to the lower channel.
 *
 * ora_value_scores: score_v [L][H_kv][D] = sum over the unit's G*W rows of
 * o_d^2, o = sum_j p_j v_j, one softmax row at a time.
 * ------------------------------------------------------------------------- */
int ora_value_scores(const ora_shape *s, const void *q, const void *k, const void *v,
                     double *score_v)
{
    if (!ora_shape_ok(s)) return -1;
    const int64_t D = s->head_dim, T = s->seq_len, W = s->window;
    const int64_t Hq = s->n_q_heads, Hkv = s->n_kv_heads, G = Hq / Hkv;
    const int64_t P = T - W, units = (int64_t)s->n_layers * Hkv;
    const double root_d = sqrt((double)D);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t u = 0; u < units; ++u) {
        const int64_t layer = u / Hkv, kv_head = u % Hkv;
        const int64_t kv_base = u * T * D;
        double *x = (double *)malloc(sizeof(double) * (size_t)T);
        double *qr = (double *)malloc(sizeof(double) * (size_t)D);
        double *o = (double *)malloc(sizeof(double) * (size_t)D);
        double *sv = score_v + u * D;
        if (!x || !qr || !o) { free(x); free(qr); free(o); bad = 1; continue; }
        for (int64_t d = 0; d < D; ++d) sv[d] = 0.0;
        for (int64_t g = 0; g < G; ++g) {
            const int64_t h = kv_head * G + g;
            for (int64_t i = 0; i < W; ++i) {
                const int64_t q_base = ((layer * Hq + h) * W + i) * D;
                for (int64_t d = 0; d < D; ++d) qr[d] = ora_elem(q, q_base + d, s->dtype);
                const int64_t t = P + i;
                double mu = -INFINITY;
                for (int64_t j = 0; j <= t; ++j) {
                    double dot = 0.0;
                    for (int64_t d = 0; d < D; ++d)
                        dot += qr[d] * ora_elem(k, kv_base + j * D + d, s->dtype);
                    x[j] = dot / root_d;
                    if (x[j] > mu) mu = x[j];
                }
                double z = 0.0;
                for (int64_t j = 0; j <= t; ++j) {
                    x[j] = exp(x[j] - mu);
                    z += x[j];
                }
                for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
                for (int64_t j = 0; j <= t; ++j) {
                    const double pj = x[j] / z;
                    for (int64_t d = 0; d < D; ++d)
                        o[d] += pj * ora_elem(v, kv_base + j * D + d, s->dtype);
                }
                for (int64_t d = 0; d < D; ++d) sv[d] += o[d] * o[d];
            }
        }
        free(x);
        free(qr);
        free(o);
    }
    return bad ? -2 : 0;
}

/* THINKV selection and copy: for every head keep the `keep` channels with the
 * largest score_v (ties to the lower channel), written ascending to chan
 * [L][H_kv][keep], and copy those channels of the head's n_l kept prefix rows
 * of the compacted values v_out (packed as kvc_compact writes them) to
 * v_pruned (layer l holds [H_kv][n_l][keep]); window rows are not pruned. */
int ora_channel_prune_value(const ora_shape *s, const double *score_v, const void *v_out,
                            const int32_t *budget, double lambda, int32_t *chan, void *v_pruned)
{
    if (!ora_shape_ok(s)) return -1;
    const int64_t D = s->head_dim, W = s->window, P = (int64_t)s->seq_len - W;
    const int64_t Hkv = s->n_kv_heads, L = s->n_layers;
    const int32_t keep = ora_keep_channels(lambda, (int32_t)D);
    if (keep < 1 || keep > D) return -1;
    const size_t es = s->dtype == 0 ? 4 : 2;
    int64_t ir = 0, oe = 0;
    for (int64_t l = 0; l < L; ++l) {
        const int64_t n = ora_kept(budget[l], P);
        for (int64_t h = 0; h < Hkv; ++h) {
            const int64_t u = l * Hkv + h;
            const int64_t row0 = ir + h * (n + W);
            ora_chan *ch = (ora_chan *)malloc(sizeof(ora_chan) * (size_t)D);
            if (!ch) return -2;
            for (int64_t d = 0; d < D; ++d) {
                ch[d].m = score_v[u * D + d];
                ch[d].d = (int32_t)d;
            }
            qsort(ch, (size_t)D, sizeof(ora_chan), ora_cmp_chan);
            int32_t *sel = chan + u * keep;
            for (int32_t i = 0; i < keep; ++i) sel[i] = ch[i].d;
            qsort(sel, (size_t)keep, sizeof(int32_t), ora_cmp_i32);
            free(ch);
            if (v_pruned) {
                const unsigned char *src = (const unsigned char *)v_out;
                unsigned char *dst = (unsigned char *)v_pruned;
                const int64_t o0 = oe + h * n * keep;
                for (int64_t r = 0; r < n; ++r)
                    for (int32_t i = 0; i < keep; ++i)
                        memcpy(dst + (size_t)(o0 + r * keep + i) * es,
                               src + (size_t)((row0 + r) * D + sel[i]) * es, es);
            }
        }
        ir += Hkv * (n + W);
        oe += Hkv * n * keep;
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Optional: ThinK query-driven key-channel pruning        [THINK-QD]
 *
 * "ThinK: Thinner Key Cache by Query-Driven Pruning", section "Greedy
 * algorithm" and "Observation window": channel j of a head scores the
 * Frobenius norm of the outer product of its query column (the last S_obs
 * window queries) and its key column, Q[-S_obs:, j] K[:, j]^T; the T
 * channels with the largest scores are kept.  The Frobenius norm of an outer
 * product is the product of the two column norms, so ranking by
 *   score_d = (sum over window query rows of q[d]^2) * (sum over kept key
 *              rows of k[d]^2)
 * (the squared norm, monotone in the norm) gives the same channels.
 * Readings: with grouped-query attention a KV head's query column stacks
 * the W window rows of each of its G query heads (all of them see this key
 * cache); the key column is the n_l kept prefix rows, as for the magnitude
 * criterion (window rows stay full width).  Ties go to the lower channel.
 * q is [L][H_q][W][D]; the other arguments and outputs are those of
 * ora_channel_prune, with `scores` receiving score_d.
 * ------------------------------------------------------------------------- */
int ora_channel_prune_query(const ora_shape *s, const void *q, const void *k_out,
                            const int32_t *budget, double lambda, int32_t *chan,
                            double *scores, void *k_pruned)
{
    if (!ora_shape_ok(s)) return -1;
    const int64_t D = s->head_dim, W = s->window, P = (int64_t)s->seq_len - W;
    const int64_t Hkv = s->n_kv_heads, Hq = s->n_q_heads, L = s->n_layers, G = Hq / Hkv;
    const int32_t keep = ora_keep_channels(lambda, (int32_t)D);
    if (keep < 1 || keep > D) return -1;
    const size_t es = s->dtype == 0 ? 4 : 2;
    int64_t *in_row = (int64_t *)malloc(sizeof(int64_t) * (size_t)L);
    int64_t *out_el = (int64_t *)malloc(sizeof(int64_t) * (size_t)L);
    int64_t ir = 0, oe = 0;
    for (int64_t l = 0; l < L; ++l) {
        in_row[l] = ir;
        out_el[l] = oe;
        const int64_t n = ora_kept(budget[l], P);
        ir += Hkv * (n + W);
        oe += Hkv * n * keep;
    }
    const int64_t units = L * Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t u = 0; u < units; ++u) {
        const int64_t l = u / Hkv, h = u % Hkv;
        const int64_t n = ora_kept(budget[l], P);
        const int64_t row0 = in_row[l] + h * (n + W);
        const int64_t qrow0 = (l * Hq + h * G) * W;   /* G*W consecutive window rows */
        ora_chan *ch = (ora_chan *)malloc(sizeof(ora_chan) * (size_t)D);
        for (int64_t d = 0; d < D; ++d) {
            double kk = 0.0, qq = 0.0;
            for (int64_t r = 0; r < n; ++r) {
                const double x = ora_elem(k_out, (row0 + r) * D + d, s->dtype);
                kk += x * x;
            }
            for (int64_t r = 0; r < G * W; ++r) {
                const double x = ora_elem(q, (qrow0 + r) * D + d, s->dtype);
                qq += x * x;
            }
            ch[d].m = qq * kk;
            ch[d].d = (int32_t)d;
            if (scores) scores[u * D + d] = qq * kk;
        }
        qsort(ch, (size_t)D, sizeof(ora_chan), ora_cmp_chan);
        int32_t *sel = chan + u * keep;
        for (int32_t i = 0; i < keep; ++i) sel[i] = ch[i].d;
        qsort(sel, (size_t)keep, sizeof(int32_t), ora_cmp_i32);
        if (k_pruned) {
            const unsigned char *src = (const unsigned char *)k_out;
            unsigned char *dst = (unsigned char *)k_pruned;
            const int64_t o0 = out_el[l] + h * n * keep;
            for (int64_t r = 0; r < n; ++r)
                for (int32_t i = 0; i < keep; ++i)
                    memcpy(dst + (size_t)(o0 + r * keep + i) * es,
                           src + (size_t)((row0 + r) * D + sel[i]) * es, es);
        }
        free(ch);
    }
    free(in_row);
    free(out_el);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Optional: per-head budgets inside a layer                   [ZZ-HEAD]
 *
 * Blog post "ZigZagKV, KVCache 80% compression near-lossless", opening of
 * the ZigZagKV part (memory should follow how many tokens each attention
 * head needs to keep most of its information, not be equal per head) and
 * "ZigZagKV token selection" (each head's K follows its quota).  Reading:
 * the layer's H_kv * B_l prefix tokens are split over its heads in
 * proportion to MBA_{l,k} with the same largest-remainder rule as the layer
 * split (ties to the lower head, equal shares when every MBA is zero), no
 * per-head minimum, each head capped at P with the excess re-split over the
 * uncapped heads until none exceeds P.  head_budget: [L][H_kv].
 * ------------------------------------------------------------------------- */
int ora_head_budget(int L, int Hkv, const int32_t *mba, const int32_t *budget, int64_t prefix,
                    int32_t *head_budget)
{
    if (L < 1 || Hkv < 1 || prefix < 1) return -1;
    int64_t *w = (int64_t *)malloc(sizeof(int64_t) * (size_t)Hkv);
    int64_t *B = (int64_t *)malloc(sizeof(int64_t) * (size_t)Hkv);
    int64_t *add = (int64_t *)malloc(sizeof(int64_t) * (size_t)Hkv);
    unsigned char *elig = (unsigned char *)malloc((size_t)Hkv);
    for (int l = 0; l < L; ++l) {
        const int64_t Bl = budget[l] < 0 ? 0 : (budget[l] > prefix ? prefix : budget[l]);
        for (int k = 0; k < Hkv; ++k) {
            w[k] = mba[(int64_t)l * Hkv + k];
            elig[k] = 1;
        }
        ora_split(Hkv, w, elig, (int64_t)Hkv * Bl, add);
        for (int k = 0; k < Hkv; ++k) B[k] = add[k];
        for (;;) {
            int64_t excess = 0;
            for (int k = 0; k < Hkv; ++k)
                if (B[k] > prefix) { excess += B[k] - prefix; B[k] = prefix; }
            if (excess == 0) break;
            for (int k = 0; k < Hkv; ++k) elig[k] = (unsigned char)(B[k] < prefix);
            ora_split(Hkv, w, elig, excess, add);
            for (int k = 0; k < Hkv; ++k) B[k] += add[k];
        }
        for (int k = 0; k < Hkv; ++k) head_budget[(int64_t)l * Hkv + k] = (int32_t)B[k];
    }
    free(w); free(B); free(add); free(elig);
    return 0;
}

/* Top-K with per-head budgets: head (l,k) keeps min(max(hb,0), P) prefix
 * positions by (score desc, index asc), written ascending.  idx:
 * [L][H_kv][k_max]; returns -1 if a head needs more than k_max. */
int ora_topk_heads(const ora_shape *s, const double *scores, const int32_t *head_budget,
                   int64_t k_max, int32_t *idx)
{
    if (!ora_shape_ok(s)) return -1;
    const int64_t T = s->seq_len, P = T - s->window;
    const int64_t units = (int64_t)s->n_layers * s->n_kv_heads;
    for (int64_t u = 0; u < units; ++u)
        if (ora_kept(head_budget[u], P) > k_max) return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t u = 0; u < units; ++u)
        if (ora_topk(P, scores + u * T, head_budget[u], idx + u * k_max) < 0) bad = 1;
    return bad ? -2 : 0;
}

/* ---------------------------------------------------------------------------
 * Optional: threshold selection with the recent window           [THRESH]
 *
 * Blog post above, section "SnapKV" (a token counts as important when its
 * attention score exceeds a set threshold) and "NVIDIA AI presents KVzap"
 * (entries with low scores are dropped while a sliding window of the most
 * recent tokens is always kept, so each head keeps as many tokens as its
 * context needs).  Reading: per head, keep every prefix position j < P with
 * c_j >= tau (fp32 scores compared as stored), ascending, plus the W window
 * rows; counts[l][k] is the number of prefix positions kept.  A head with
 * more than k_max such positions keeps the first k_max and the call
 * returns 1 (the counts still report the full number).
 * ------------------------------------------------------------------------- */
int ora_threshold_select(const ora_shape *s, const float *scores, float tau, int64_t k_max,
                         int32_t *idx, int32_t *counts)
{
    if (!ora_shape_ok(s) || k_max < 1) return -1;
    const int64_t T = s->seq_len, P = T - s->window;
    const int64_t units = (int64_t)s->n_layers * s->n_kv_heads;
    int over = 0;
    for (int64_t u = 0; u < units; ++u) {
        int64_t n = 0;
        for (int64_t j = 0; j < P; ++j) {
            if (scores[u * T + j] >= tau) {
                if (n < k_max) idx[u * k_max + n] = (int32_t)j;
                ++n;
            }
        }
        counts[u] = (int32_t)n;
        if (n > k_max) over = 1;
    }
    return over;
}

/* ---------------------------------------------------------------------------
 * Compaction with per-head counts                                  [SNAP]
 *
 * Head (l,k) contributes its n_{l,k} = min(max(counts,0), P, k_max) kept
 * rows idx[l][k][0..n) and then the W window rows; heads follow each other
 * in (l, k) order.  Returns the rows written, or -1.
 * ------------------------------------------------------------------------- */
int64_t ora_compact_heads(const ora_shape *s, const void *src, const int32_t *idx,
                          const int32_t *counts, int64_t k_max, void *out)
{
    if (!ora_shape_ok(s)) return -1;
    const int64_t D = s->head_dim, T = s->seq_len, W = s->window, P = T - W;
    const size_t es = s->dtype == 0 ? 4 : 2;
    const int64_t units = (int64_t)s->n_layers * s->n_kv_heads;
    const unsigned char *in = (const unsigned char *)src;
    unsigned char *o = (unsigned char *)out;
    int64_t row = 0;
    for (int64_t u = 0; u < units; ++u) {
        int64_t n = ora_kept(counts[u], P);
        if (n > k_max) n = k_max;
        for (int64_t r = 0; r < n; ++r, ++row)
            memcpy(o + (size_t)row * D * es, in + (size_t)(u * T + idx[u * k_max + r]) * D * es,
                   (size_t)D * es);
        for (int64_t w = 0; w < W; ++w, ++row)
            memcpy(o + (size_t)row * D * es, in + (size_t)(u * T + P + w) * D * es, (size_t)D * es);
    }
    return row;
}

/* ---------------------------------------------------------------------------
 * Optional: Keyformer scoring with Gumbel noise                 [KEYF]
 *
 * "Keyformer: KV Cache reduction through key tokens selection" (notes on
 * moyutianzun.com): the logits x_i = q.k_i / sqrt(d) get Gumbel noise,
 * y_i = x_i + zeta_i, and a temperature, f(y_i) = softmax(y / tau); in the
 * prompt phase the w most recent tokens are kept and the other k - w are the
 * highest-scoring older tokens.  Readings: the page's prompt-phase tau is
 * "infinite", which would make every score equal, so tau is a parameter; the
 * queries are the W window rows (as for SnapKV) and the score of a key is the
 * mean of f over them, causal inside the window, GQA rows averaged; the
 * recent tokens are the window, and the older tokens are chosen by the same
 * top-K step.  zeta = -ln(-ln u) with u uniform on (0,1) from the
 * counter-based generator below, one draw per (unit, row, key).
 *
 * Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
 * easy as 1, 2, 3", SC 2011): a 4 x 32-bit counter and a 2 x 32-bit key;
 * each of ten rounds multiplies counter words 0 and 2 by two constants into
 * 64-bit products, and the new counter is (hi(c2*M1) ^ c1 ^ k0, lo(c2*M1),
 * hi(c0*M0) ^ c3 ^ k1, lo(c0*M0)); the key gains the Weyl increments after
 * every round but the last.
 * ------------------------------------------------------------------------- */
void ora_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        const uint64_t p0 = (uint64_t)M0 * c0, p1 = (uint64_t)M1 * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        const uint32_t n1 = (uint32_t)p1;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        const uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        if (round < 9) { k0 += W0; k1 += W1; }
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The uniform draw for (unit u, row r, key j): word j mod 4 of Philox4x32-10
 * at counter (floor(j / 4), r, u, 0) with key (seed low, seed high) -- one
 * output block serves four consecutive keys of a row; its top 24 bits b give
 * u = (b + 1/2) * 2^-24, exactly representable and strictly inside (0,1). */
double ora_keyformer_uniform(uint64_t seed, int64_t unit, int64_t row, int64_t key)
{
    const uint32_t ctr[4] = {(uint32_t)(key >> 2), (uint32_t)row, (uint32_t)unit, 0u};
    const uint32_t k[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t o[4];
    ora_philox4x32_10(ctr, k, o);
    return ((double)(o[key & 3] >> 8) + 0.5) * (1.0 / 16777216.0);
}

int ora_score_keyformer(const ora_shape *s, const void *q, const void *k, uint64_t seed,
                        double tau, double *scores)
{
    if (!ora_shape_ok(s) || !(tau > 0.0)) return -1;
    const int64_t D = s->head_dim, T = s->seq_len, W = s->window;
    const int64_t Hq = s->n_q_heads, Hkv = s->n_kv_heads, G = Hq / Hkv, L = s->n_layers;
    const int64_t P = T - W;
    const double rows = (double)(G * W);
    const double root_d = sqrt((double)D);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t u = 0; u < L * Hkv; ++u) {
        const int64_t layer = u / Hkv, kv_head = u % Hkv;
        double *c = scores + u * T;
        const int64_t k_base = u * T * D;
        double *y = (double *)malloc(sizeof(double) * (size_t)T);
        double *qr = (double *)malloc(sizeof(double) * (size_t)D);
        if (!y || !qr) { free(y); free(qr); bad = 1; continue; }
        for (int64_t j = 0; j < T; ++j) c[j] = 0.0;
        for (int64_t g = 0; g < G; ++g) {
            const int64_t h = kv_head * G + g;
            for (int64_t i = 0; i < W; ++i) {
                const int64_t r = g * W + i;
                const int64_t q_base = ((layer * Hq + h) * W + i) * D;
                for (int64_t d = 0; d < D; ++d) qr[d] = ora_elem(q, q_base + d, s->dtype);
                const int64_t t = P + i;
                double mu = -INFINITY;
                for (int64_t j = 0; j <= t; ++j) {
                    double dot = 0.0;
                    for (int64_t d = 0; d < D; ++d)
                        dot += qr[d] * ora_elem(k, k_base + j * D + d, s->dtype);
                    const double zeta = -log(-log(ora_keyformer_uniform(seed, u, r, j)));
                    y[j] = (dot / root_d + zeta) / tau;
                    if (y[j] > mu) mu = y[j];
                }
                double z = 0.0;
                for (int64_t j = 0; j <= t; ++j) {
                    y[j] = exp(y[j] - mu);
                    z += y[j];
                }
                for (int64_t j = 0; j <= t; ++j) c[j] += y[j] / z / rows;
            }
        }
        free(y);
        free(qr);
    }
    return bad ? -2 : 0;
}

/* ---------------------------------------------------------------------------
 * The whole path for one prompt: score -> MBA -> budgets -> top-K -> compact
 * (-> channel prune when lambda >= 0).  Output buffers as above; scores are
 * returned in fp64.  Returns 0, or a negative code from the failing step.
 * ------------------------------------------------------------------------- */
int ora_compress(const ora_shape *s, const void *q, const void *k, const void *v,
                 uint32_t num, uint32_t den, int64_t total, int64_t floor_,
                 double lambda, int64_t k_max,
                 double *scores, int32_t *mba, int32_t *budget, int32_t *idx,
                 void *k_out, void *v_out, int32_t *chan, void *k_pruned)
{
    int r;
    if ((r = ora_score(s, q, k, scores)) != 0) return r;
    if ((r = ora_mba_all(s, scores, num, den, mba)) != 0) return r;
    if ((r = ora_budget(s->n_layers, s->n_kv_heads, mba, (int64_t)s->seq_len - s->window,
                        total, floor_, budget)) != 0)
        return r;
    if ((r = ora_topk_all(s, scores, budget, k_max, idx)) != 0) return r;
    if (ora_compact(s, k, idx, budget, k_max, k_out) < 0) return -3;
    if (ora_compact(s, v, idx, budget, k_max, v_out) < 0) return -3;
    if (lambda >= 0.0)
        if ((r = ora_channel_prune(s, k_out, budget, lambda, chan, NULL, k_pruned)) != 0)
            return r;
    return 0;
}
