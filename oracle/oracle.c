/*
 * oracle.c -- plain, slow CPU oracle for neuron-level activation-sparse FFN
 * inference (SelectInfer selection + SpAx three-tier down-projection).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do. It shares no code, header, table or helper with the CUDA
 * path.
 *
 * Precision: every floating-point value the method produces (scores,
 * activations, FFN outputs) is computed in double from the bf16 inputs
 * widened exactly. Where a float decides an integer (a ranking, a top-k, a
 * quantised code) the decision is taken on the float32 values the caller
 * hands in, with float32 arithmetic, which is the precision the GPU path
 * decides in.
 *
 * Notation follows the pages: neuron n has gate row Wg[n,:], up row Wu[n,:]
 * (HF layout [N x d]) and down column Wd[:,n] (HF layout [d x N]);
 * a_n(x) = silu(Wg[n].x) * (Wu[n].x), silu(z) = z / (1 + e^-z).
 *
 * Pins (what each function is checked against, besides itself), see tests:
 *   oracle_profile_scores  brute force per token + closed form silu values
 *   oracle_merge_scores    hand-computed file merges
 *   oracle_sparse_layers   Table 1's values read as words ("first layer 5",
 *                          "skip last 2") at several depths
 *   oracle_down_norms      closed forms (constant columns) and numpy.linalg.norm
 *   oracle_expand_clusters hand-worked expansions, S_c = 1 identity, brute force
 *   oracle_rank_loaded     subset enumeration on tiny N, Table 1 / Eq. 2 counts
 *   oracle_topk_rows       subset enumeration on tiny rows with forced ties
 *   oracle_select          subset enumeration of the top-beta step, counting
 *   oracle_sparse_ffn      dense numpy/scipy FFN when every neuron is kept
 *   oracle_absact          numpy/scipy activations
 *   oracle_dense_act       numpy/scipy activations
 *   oracle_spax_encode     error bound |w - w^| <= scale/2, constant and ramp groups
 *   oracle_spax_tiers      subset enumeration on tiny N
 *   oracle_spax_down       dense numpy product when top = 100% / mid = 100%
 *   oracle_swiglu          closed-form silu values; with spax_down, the dense
 *                          activations when every input channel is top tier
 *   oracle_bf16_round      the definition's properties on every kind of
 *                          input (exact values, ties both ways, halfway
 *                          carries into the exponent, signs, inf) and the
 *                          nearest-value property on random floats
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ basics */

static double bf(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* a_n(x) for one neuron: the input of down_proj, i.e. the output of the
 * SwiGLU activation (SelectInfer, section 3 "LLM Profiler"). */
static double act(const uint16_t *wg_row, const uint16_t *wu_row, const uint16_t *x, int d)
{
    double g = 0.0, u = 0.0;
    for (int k = 0; k < d; ++k) {
        double xk = bf(x[k]);
        g += bf(wg_row[k]) * xk;
        u += bf(wu_row[k]) * xk;
    }
    return silu(g) * u;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Neuron counts from the pages' ratios: round to nearest, in double.
 * (SelectInfer section 4 / Table 1 give the ratios; a count of 20% of 1024
 * neurons is 205.) */
long long oracle_cnt(double r, long long n) { return (long long)floor(r * (double)n + 0.5); }

/* ------------------------------------------------------------- ordering */

typedef struct {
    float key;
    int idx;
} kf;

/* descending key, ties to the lower index */
static int cmp_kf(const void *pa, const void *pb)
{
    const kf *a = (const kf *)pa, *b = (const kf *)pb;
    if (a->key > b->key) return -1;
    if (a->key < b->key) return 1;
    return (a->idx < b->idx) ? -1 : (a->idx > b->idx);
}

typedef struct {
    uint32_t key;
    int idx;
} ku;

static int cmp_ku(const void *pa, const void *pb)
{
    const ku *a = (const ku *)pa, *b = (const ku *)pb;
    if (a->key > b->key) return -1;
    if (a->key < b->key) return 1;
    return (a->idx < b->idx) ? -1 : (a->idx > b->idx);
}

static int cmp_int(const void *pa, const void *pb)
{
    int a = *(const int *)pa, b = *(const int *)pb;
    return (a > b) - (a < b);
}

/* ------------------------------------------------------------ a1 profile */

/* Profiler score, SelectInfer section 3, Eq. (1): s_n = sum over tokens t of
 * |a_n(t)|. Accumulates into s (double), so several calls over batches of
 * calibration tokens add up. */
void oracle_profile_scores(const uint16_t *Wg, const uint16_t *Wu, int d, int N,
                           const uint16_t *X, int T, double *s)
{
    #pragma omp parallel for schedule(dynamic, 16)
    for (int n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int t = 0; t < T; ++t)
            acc += fabs(act(Wg + (size_t)n * d, Wu + (size_t)n * d, X + (size_t)t * d, d));
        s[n] += acc;
    }
}

/* Merging score files, SelectInfer section 3: each file's scores are
 * normalised by its token count and the normalised values are summed.
 * float32, files in the given order: out[n] = sum_f (s_f[n] / (float)T_f).
 * The result feeds a ranking, so it is formed in float32 like the GPU's. */
void oracle_merge_scores(const float *const *s, const long long *tokens, int nfiles, int N, float *out)
{
    for (int n = 0; n < N; ++n) {
        float acc = 0.0f;
        for (int f = 0; f < nfiles; ++f) {
            float q = s[f][n] / (float)tokens[f];
            acc = acc + q;
        }
        out[n] = acc;
    }
}

/* Layer range, SelectInfer section 6.4, Table 1 ("First layer 5", "Last layer
 * -2 (skip last 2)"): selection runs on layers first .. end-1 and every other
 * layer keeps its dense FFN. `last` reads as a slice end: end = L + last when
 * last <= 0 (so -2 skips the last two layers), else end = last; the range is
 * clipped to [0, L]. sparse[l] = 1 inside it, 0 outside. Returns the number
 * of sparse layers, or -1 for L < 0 or first < 0. */
int oracle_sparse_layers(int L, int first, int last, uint8_t *sparse)
{
    if (L < 0 || first < 0) return -1;
    int end = last <= 0 ? L + last : last;
    if (end > L) end = L;
    int count = 0;
    for (int l = 0; l < L; ++l) {
        sparse[l] = (uint8_t)(l >= first && l < end);
        count += sparse[l];
    }
    return count;
}

/* Weight-aware salience (WiSparse abstract: activation magnitudes combined
 * with precomputed weight norms). Read as the size of neuron n's contribution
 * to the FFN output: salience_n = |a_n| * ||Wd[:, n]||_2. This computes the
 * norms of the loaded neurons' down columns, norm[p] = sqrt(sum_j
 * Wd[j, loaded[p]]^2), in float64. */
void oracle_down_norms(const uint16_t *Wd, int d, int N, const int *loaded, int n, double *norm)
{
    for (int p = 0; p < n; ++p) {
        double acc = 0.0;
        for (int j = 0; j < d; ++j) {
            double w = bf(Wd[(size_t)j * N + loaded[p]]);
            acc += w * w;
        }
        norm[p] = sqrt(acc);
    }
}

/* Cluster-granular selection (PowerInfer-2 neuron clusters, quoted as prior
 * art on the pages: contiguous blocks C_k of S_c neuron indices, k*S_c ..
 * (k+1)*S_c - 1; when one neuron of a cluster is predicted active the whole
 * cluster is brought in). Applied to a computed set: out receives, in
 * ascending order, every packed position p (loaded neuron loaded[p]) whose
 * cluster loaded[p] / S_c holds the neuron of some selected position S[i].
 * Returns the count, or -1 for S_c < 1. */
int oracle_expand_clusters(const int *loaded, int n_loaded, const int *S, int n_sel, int N, int S_c, int *out)
{
    if (S_c < 1) return -1;
    int nc = (N + S_c - 1) / S_c;
    uint8_t *hit = (uint8_t *)calloc((size_t)(nc > 0 ? nc : 1), 1);
    for (int i = 0; i < n_sel; ++i) hit[loaded[S[i]] / S_c] = 1;
    int n = 0;
    for (int p = 0; p < n_loaded; ++p)
        if (hit[loaded[p] / S_c]) out[n++] = p;
    free(hit);
    return n;
}

/* ------------------------------------------------------------ a2 loading */

/* Selective loading, SelectInfer section 4 and Fig. 6: the base neurons are
 * the top-delta neurons by task-specific score; secondary neurons are then
 * added by model-specific score (among the rest) until the loaded fraction
 * gamma is reached. Rankings are by decreasing score, ties to the lower
 * neuron index. Output: the loaded neurons in ascending index order
 * (loaded[0..n_loaded)), and is_static[p] = 1 when loaded[p] is a base
 * neuron (static neurons are the base neurons, section 5). */
int oracle_rank_loaded(const float *task, const float *model, int N, double gamma, double delta,
                       int *loaded, uint8_t *is_static, int *n_loaded_out, int *n_static_out)
{
    int n_load = (int)oracle_cnt(gamma, N), n_base = (int)oracle_cnt(delta, N);
    if (n_base > n_load || n_load > N || n_base < 0) return -1;
    kf *v = (kf *)malloc(sizeof(kf) * (size_t)N);
    uint8_t *base = (uint8_t *)calloc((size_t)N, 1), *take = (uint8_t *)calloc((size_t)N, 1);
    for (int n = 0; n < N; ++n) { v[n].key = task[n]; v[n].idx = n; }
    qsort(v, (size_t)N, sizeof(kf), cmp_kf);
    for (int i = 0; i < n_base; ++i) { base[v[i].idx] = 1; take[v[i].idx] = 1; }
    int m = 0;
    for (int n = 0; n < N; ++n)
        if (!base[n]) { v[m].key = model[n]; v[m].idx = n; ++m; }
    qsort(v, (size_t)m, sizeof(kf), cmp_kf);
    for (int i = 0; i < n_load - n_base; ++i) take[v[i].idx] = 1;
    int p = 0;
    for (int n = 0; n < N; ++n)
        if (take[n]) { loaded[p] = n; is_static[p] = base[n]; ++p; }
    *n_loaded_out = p;
    *n_static_out = n_base;
    free(v); free(base); free(take);
    return 0;
}

/* Bytes kept in memory by selective loading for one layer: the gate row, up
 * row and down column of each loaded neuron, at s bytes per parameter
 * (SelectInfer section 6.6, Eq. (2) counts the complement). */
long long oracle_loaded_bytes(int d, int n_loaded, int s) { return 3LL * d * n_loaded * s; }

/* -------------------------------------------------- a3 prefill activations */

/* |A|[t, p] = |a_{loaded[p]}(x_t)| for every token row and every loaded
 * neuron ("for each token, we compute activation values for all loaded
 * neurons", SelectInfer section 5, Fig. 7). double output, row-major
 * [rows x n_loaded]. */
void oracle_absact(const uint16_t *Wg, const uint16_t *Wu, int d, const int *loaded, int n_loaded,
                   const uint16_t *X, int rows, double *out)
{
    #pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < rows; ++t)
        for (int p = 0; p < n_loaded; ++p) {
            int n = loaded[p];
            out[(size_t)t * n_loaded + p] =
                fabs(act(Wg + (size_t)n * d, Wu + (size_t)n * d, X + (size_t)t * d, d));
        }
}

/* ------------------------------------------------------------ a4 top-alpha */

/* Per row, the k entries with the largest value, ties to the lower index
 * ("sort these activations in descending order and select the top alpha",
 * SelectInfer section 5). A is float32 [rows x ld], only the first n columns
 * take part. sel is [rows x n] bytes, 1 = selected. */
void oracle_topk_rows(const float *A, int rows, int n, int ld, int k, uint8_t *sel)
{
    #pragma omp parallel
    {
        kf *v = (kf *)malloc(sizeof(kf) * (size_t)(n > 0 ? n : 1));
        #pragma omp for schedule(dynamic, 4)
        for (int r = 0; r < rows; ++r) {
            for (int i = 0; i < n; ++i) { v[i].key = fabsf(A[(size_t)r * ld + i]); v[i].idx = i; }
            qsort(v, (size_t)n, sizeof(kf), cmp_kf);
            memset(sel + (size_t)r * n, 0, (size_t)n);
            for (int i = 0; i < k && i < n; ++i) sel[(size_t)r * n + v[i].idx] = 1;
        }
        free(v);
    }
}

/* --------------------------------------------- a5 + a6 dynamic selection */

/* Dynamic neuron selection during prefill, SelectInfer section 5 / Fig. 7:
 *   a4  per token, the top-alpha loaded neurons by |a| (all loaded neurons,
 *       static ones included);
 *   a5  per sequence, count how often each loaded neuron occurs in the
 *       per-token lists;
 *   a6  keep the top-beta neurons by count among the loaded non-static
 *       neurons (ties to the lower index), beta = n_sel - n_static, and
 *       combine them with the static neurons, so that the computed set
 *       reaches phi = delta + epsilon.
 * absA is float32 [B*T x ld] (sequence-major rows), is_static [n_loaded].
 * Outputs: S [B x n_sel] ascending packed positions; optional counts
 * [B x n_loaded] (uint32) and sel [B*T x n_loaded] (bytes). Returns -1 when
 * beta does not fit. */
int oracle_select(const float *absA, int T, int B, int n_loaded, int ld, const uint8_t *is_static,
                  int alpha, int n_sel, int *S, uint32_t *counts_out, uint8_t *sel_out)
{
    int n_static = 0;
    for (int p = 0; p < n_loaded; ++p) n_static += is_static[p] ? 1 : 0;
    int beta = n_sel - n_static;
    if (beta < 0 || beta > n_loaded - n_static) return -1;
    uint8_t *sel = sel_out ? sel_out : (uint8_t *)malloc((size_t)B * T * n_loaded + 1);
    oracle_topk_rows(absA, B * T, n_loaded, ld, alpha, sel);
    uint32_t *cnt = (uint32_t *)calloc((size_t)n_loaded, sizeof(uint32_t));
    ku *v = (ku *)malloc(sizeof(ku) * (size_t)(n_loaded + 1));
    uint8_t *take = (uint8_t *)malloc((size_t)n_loaded + 1);
    for (int b = 0; b < B; ++b) {
        memset(cnt, 0, sizeof(uint32_t) * (size_t)n_loaded);
        for (int t = 0; t < T; ++t)
            for (int p = 0; p < n_loaded; ++p)
                cnt[p] += sel[((size_t)b * T + t) * n_loaded + p];
        if (counts_out) memcpy(counts_out + (size_t)b * n_loaded, cnt, sizeof(uint32_t) * (size_t)n_loaded);
        int m = 0;
        for (int p = 0; p < n_loaded; ++p)
            if (!is_static[p]) { v[m].key = cnt[p]; v[m].idx = p; ++m; }
        qsort(v, (size_t)m, sizeof(ku), cmp_ku);
        for (int p = 0; p < n_loaded; ++p) take[p] = is_static[p] ? 1 : 0;
        for (int i = 0; i < beta; ++i) take[v[i].idx] = 1;
        int q = 0;
        for (int p = 0; p < n_loaded; ++p)
            if (take[p]) S[(size_t)b * n_sel + q++] = p;
    }
    free(v); free(take); free(cnt);
    if (!sel_out) free(sel);
    return 0;
}

/* ------------------------------------------------------ a7 sparse decode */

/* Sparse decode FFN on the computed set (SelectInfer section 5: only the
 * selected neurons are computed at decode):
 *   y = sum over p in S (ascending) of a_{loaded[p]}(x) * Wd[:, loaded[p]].
 * Weights are the HF-layout originals; y is double [d]. */
void oracle_sparse_ffn(const uint16_t *Wg, const uint16_t *Wu, const uint16_t *Wd, int d, int N,
                       const int *loaded, const int *S, int n_sel, const uint16_t *x, double *y)
{
    double *a = (double *)malloc(sizeof(double) * (size_t)(n_sel > 0 ? n_sel : 1));
    #pragma omp parallel for schedule(dynamic, 16)
    for (int i = 0; i < n_sel; ++i) {
        int n = loaded[S[i]];
        a[i] = act(Wg + (size_t)n * d, Wu + (size_t)n * d, x, d);
    }
    for (int j = 0; j < d; ++j) y[j] = 0.0;
    #pragma omp parallel for schedule(static)
    for (int j = 0; j < d; ++j) {
        double acc = 0.0;
        for (int i = 0; i < n_sel; ++i) acc += a[i] * bf(Wd[(size_t)j * N + loaded[S[i]]]);
        y[j] = acc;
    }
    free(a);
}

/* ------------------------------------------------- a7 decode stack input */

/* bf16 value of a float32, rounded to nearest with ties to even: the input a
 * layer of an FFN-only stack reads from the fp32 residual stream (the decode
 * steps of SelectInfer section 5 run the layers one after another; with no
 * attention or norm between the FFNs, layer l+1 reads h + FFN_l(x_l)).
 * Written from the definition: of the two bf16 values around f (f with its low
 * 16 bits cleared, and that plus one bf16 step away from zero), the nearer
 * one; on an exact tie, the one whose last kept bit is 0. Inf stays inf; NaN
 * stays a NaN. */
uint16_t oracle_bf16_round(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u) {           /* inf or NaN */
        if (u & 0x007FFFFFu) return (uint16_t)((u >> 16) | 0x0040u);
        return (uint16_t)(u >> 16);
    }
    uint32_t lower = u >> 16;                          /* truncated toward zero */
    uint32_t rest = u & 0xFFFFu;                       /* the dropped bits */
    if (rest > 0x8000u || (rest == 0x8000u && (lower & 1u))) lower += 1u;
    return (uint16_t)lower;
}

void oracle_bf16_round_array(const float *f, int n, uint16_t *out)
{
    for (int i = 0; i < n; ++i) out[i] = oracle_bf16_round(f[i]);
}

/* a_n(x) for every neuron of a layer (dense gate/up pass that the SpAx
 * decode uses to rank columns by |a|). double [N]. */
void oracle_dense_act(const uint16_t *Wg, const uint16_t *Wu, int d, int N, const uint16_t *x, double *a)
{
    #pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) a[n] = act(Wg + (size_t)n * d, Wu + (size_t)n * d, x, d);
}

/* a_n = silu(g_n) * u_n from given projections (double): the last step of
 * the gate/up pass when the projections themselves come from a tiered
 * product (SpAx's tiers applied to gate/up by |x|, the pages' "ALL"
 * configuration for the FFN). */
void oracle_swiglu(const double *g, const double *u, int n, double *a)
{
    for (int i = 0; i < n; ++i) a[i] = silu(g[i]) * u[i];
}

/* --------------------------------------------------------- a8 SpAx encode */

/* SpAx offline encoding ("Activation Sparsity with Weight Approximation for
 * Faster LLM Decoding on Offloaded Weights", Fig. 2 offline encoding and
 * Fig. 3 reconstruction of a middle-tier column from its own b-bit codes).
 * Per column n of Wd and per group of `group` consecutive rows:
 *   mn, mx = min, max of the group (float32);
 *   scale  = (mx - mn) / (2^bits - 1)            (float32)
 *   q      = clamp(floor((w - mn) / scale + 0.5), 0, 2^bits - 1), q = 0 when scale == 0
 *   w^     = mn + q * scale.
 * codes: [N x d*bits/8] bytes holding each column's codes as one bit stream,
 * element i in bits i*bits .. i*bits + bits - 1, bit k of the stream being
 * bit k % 8 of byte k / 8 (so element 2i sits in the low nibble of byte i for
 * bits = 4, and a 3-bit code can straddle two bytes); bits in {2, 3, 4, 8},
 * d*bits a multiple of 8; params: [N x d/group x 2] float32 = (scale, min). */
int oracle_spax_encode(const uint16_t *Wd, int d, int N, int bits, int group, uint8_t *codes, float *params)
{
    if (!(bits == 2 || bits == 3 || bits == 4 || bits == 8) || group <= 0 || d % group || (d * bits) % 8) return -1;
    int ng = d / group, qmax = (1 << bits) - 1;
    size_t cb = (size_t)d * bits / 8;
    memset(codes, 0, cb * (size_t)N);
    for (int n = 0; n < N; ++n)
        for (int g = 0; g < ng; ++g) {
            float mn = INFINITY, mx = -INFINITY;
            for (int r = 0; r < group; ++r) {
                float w = (float)bf(Wd[(size_t)(g * group + r) * N + n]);
                if (w < mn) mn = w;
                if (w > mx) mx = w;
            }
            float scale = (mx - mn) / (float)qmax;
            params[((size_t)n * ng + g) * 2 + 0] = scale;
            params[((size_t)n * ng + g) * 2 + 1] = mn;
            for (int r = 0; r < group; ++r) {
                int i = g * group + r;
                float w = (float)bf(Wd[(size_t)i * N + n]);
                int q = 0;
                if (scale != 0.0f) {
                    float t = (w - mn) / scale;
                    t = t + 0.5f;
                    q = (int)floorf(t);
                    if (q < 0) q = 0;
                    if (q > qmax) q = qmax;
                }
                for (int k = 0; k < bits; ++k) {
                    size_t bit = (size_t)i * bits + k;
                    codes[(size_t)n * cb + bit / 8] |= (uint8_t)(((q >> k) & 1) << (bit % 8));
                }
            }
        }
    return 0;
}

/* ---------------------------------------------------------- a9 SpAx tiers */

/* SpAx tier choice per decoded token (abstract; Fig. 2): columns with the
 * largest |a| are read in the original format (top tier, k_top columns), the
 * next k_mid are reconstructed from codes (middle tier), the rest skipped.
 * Ranking by |a| descending (float32), ties to the lower index. Both lists
 * are returned in ascending column order. */
int oracle_spax_tiers(const float *a, int N, int k_top, int k_mid, int *top, int *mid)
{
    if (k_top < 0 || k_mid < 0 || k_top + k_mid > N) return -1;
    kf *v = (kf *)malloc(sizeof(kf) * (size_t)(N > 0 ? N : 1));
    for (int n = 0; n < N; ++n) { v[n].key = fabsf(a[n]); v[n].idx = n; }
    qsort(v, (size_t)N, sizeof(kf), cmp_kf);
    for (int i = 0; i < k_top; ++i) top[i] = v[i].idx;
    for (int i = 0; i < k_mid; ++i) mid[i] = v[k_top + i].idx;
    qsort(top, (size_t)k_top, sizeof(int), cmp_int);
    qsort(mid, (size_t)k_mid, sizeof(int), cmp_int);
    free(v);
    return 0;
}

/* Tiered down-projection: y = sum_{n in top} a_n Wd[:, n]
 *                             + sum_{n in mid} a_n w^_n     (w^ from the codes).
 * a is float32 [N] (the activations that chose the tiers); y double [d]. */
void oracle_spax_down(const float *a, int N, int d, const uint16_t *Wd, const uint8_t *codes,
                      const float *params, int bits, int group, const int *top, int k_top,
                      const int *mid, int k_mid, double *y)
{
    int ng = d / group;
    size_t cb = (size_t)d * bits / 8;
    #pragma omp parallel for schedule(static)
    for (int j = 0; j < d; ++j) {
        double acc = 0.0;
        for (int i = 0; i < k_top; ++i) {
            int n = top[i];
            acc += (double)a[n] * bf(Wd[(size_t)j * N + n]);
        }
        int g = j / group;
        for (int i = 0; i < k_mid; ++i) {
            int n = mid[i];
            uint32_t q = 0;
            for (int k = 0; k < bits; ++k) {
                size_t bit = (size_t)j * bits + k;
                q |= (uint32_t)((codes[(size_t)n * cb + bit / 8] >> (bit % 8)) & 1u) << k;
            }
            double scale = params[((size_t)n * ng + g) * 2 + 0];
            double mn = params[((size_t)n * ng + g) * 2 + 1];
            acc += (double)a[n] * (mn + (double)q * scale);
        }
        y[j] = acc;
    }
}
