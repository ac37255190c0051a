/*
 * CPU oracle of the Mixture-of-Grouped-Experts (MoGE) layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header
 * or helper with the CUDA path and must never be used to produce a result of
 * the product path.
 *
 * Plain, slow and direct: every step is the definition written out, with
 * double accumulation and no blocking, fusion or reordering.  Loops over
 * tokens run in parallel (OpenMP) because tokens are independent; the
 * arithmetic of each token is the same as in a serial loop.
 *
 * Sources ("Pangu Pro MoE: Mixture of Grouped Experts for Efficient Sparsity"
 * as retold on the pages):
 *   [EXPL-1] Pangu Pro MoE explainer (lsdiaocha.cn), section 1 "innovative
 *            architecture": N experts split evenly into M groups of N/M; for
 *            each token a global softmax over all N expert scores, then a
 *            local top-K' with K' = K/M inside every group; the imbalance score
 *            is the load difference between the busiest and the idlest device
 *            over a batch.
 *   [EXPL-6] same page, section 6 "expert analysis": no co-activation of two
 *            experts of one group (K'=1).
 *   [CSDN]   CSDN post "突破千亿参数瓶颈…", "MoGE架构的革命性改进": 64 experts in
 *            8 groups of 8, a fixed number of experts chosen per group.
 * Readings where the pages are silent (SwiGLU expert FFN, unrenormalised
 * gates, lower-index tie break, bias added before softmax, contiguous
 * groups, stable by-token row order, imbalance normalised by T) are the
 * plainest ones consistent with the above; each is marked "reading" below.
 *
 * Data types: activations/weights are fp32 (dtype 0) or raw bf16 bits
 * (dtype 1), read as exact values.  Layouts: x [T,d], W_r [N,d],
 * W_gate/W_up [N,I,d], W_down [N,d,I], all row-major.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static inline double val(const void *p, int dtype, int64_t i) {
    if (dtype == 0) return (double)((const float *)p)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)p)[i] << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Router scores [EXPL-1: "scores for all experts"]:
 *   logit[t,e] = fp32( sum_i x[t,i] * W_r[e,i]  (double)  + b[e] ).
 * Reading: the bias is a per-expert additive term before the softmax. */
void oracle_router_logits(int64_t T, int64_t d, int64_t N, int dtype, const void *x,
                          const void *w_r, const float *bias, float *logits) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t e = 0; e < N; ++e) {
            double s = 0.0;
            for (int64_t i = 0; i < d; ++i) s += val(x, dtype, t * d + i) * val(w_r, dtype, e * d + i);
            if (bias) s += (double)bias[e];
            logits[t * N + e] = (float)s;
        }
    }
}

/* Global softmax over all N experts [EXPL-1], in double:
 *   p[t,e] = exp(l[t,e] - m) / sum_e' exp(l[t,e'] - m),  m = max_e l[t,e]. */
void oracle_softmax(int64_t T, int64_t N, const float *logits, double *p) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * N;
        double m = (double)l[0];
        for (int64_t e = 1; e < N; ++e) m = fmax(m, (double)l[e]);
        double s = 0.0;
        for (int64_t e = 0; e < N; ++e) s += exp((double)l[e] - m);
        for (int64_t e = 0; e < N; ++e) p[t * N + e] = exp((double)l[e] - m) / s;
    }
}

/* "a ranks before b": higher score first, lower expert index on equal scores
 * (reading: ties go to the lower index). */
static inline int ranks_before(float la, int64_t a, float lb, int64_t b) {
    return (la > lb) || (la == lb && a < b);
}

/* Sort experts lo..hi-1 of one token by ranks_before (insertion sort, stable
 * by construction) and write the first k of them to out[0..k). */
static void top_k_of_range(const float *l, int64_t lo, int64_t hi, int64_t k, int32_t *out,
                           int32_t *scratch) {
    int64_t n = hi - lo;
    for (int64_t i = 0; i < n; ++i) {
        int32_t e = (int32_t)(lo + i);
        int64_t j = i;
        while (j > 0 && ranks_before(l[e], e, l[scratch[j - 1]], scratch[j - 1])) {
            scratch[j] = scratch[j - 1];
            --j;
        }
        scratch[j] = e;
    }
    for (int64_t r = 0; r < k; ++r) out[r] = scratch[r];
}

/* Group-local top-K' [EXPL-1, CSDN].  Group g holds experts [gG, (g+1)G)
 * (reading: contiguous ranges, "split evenly").  Selection compares the fp32
 * logits, which orders experts exactly as the softmax probabilities do since
 * the softmax is strictly increasing.  Slot order (reading): group ascending,
 * then rank ascending: idx[t, g*K' + r] = r-th best expert of group g. */
void oracle_select_grouped(int64_t T, int64_t N, int64_t M, int64_t kpg, const float *logits,
                           int32_t *idx) {
    const int64_t G = N / M, K = M * kpg;
#pragma omp parallel
    {
        int32_t *scratch = (int32_t *)malloc(sizeof(int32_t) * (size_t)G);
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t)
            for (int64_t g = 0; g < M; ++g)
                top_k_of_range(logits + t * N, g * G, (g + 1) * G, kpg, idx + t * K + g * kpg, scratch);
        free(scratch);
    }
}

/* Conventional MoE routing that ignores placement [EXPL-1]: top-K over all N
 * experts, slots in rank order.  The same rank rule with one group. */
void oracle_select_global(int64_t T, int64_t N, int64_t K, const float *logits, int32_t *idx) {
#pragma omp parallel
    {
        int32_t *scratch = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) top_k_of_range(logits + t * N, 0, N, K, idx + t * K, scratch);
        free(scratch);
    }
}

/* Gates: the global-softmax probability of each selected expert, not
 * renormalised over the selection (reading).  gate32 = fp32(gate64). */
void oracle_gates(int64_t T, int64_t N, int64_t K, const int32_t *idx, const double *p,
                  float *gate32, double *gate64) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = 0; k < K; ++k) {
            double g = p[t * N + idx[t * K + k]];
            if (gate64) gate64[t * K + k] = g;
            if (gate32) gate32[t * K + k] = (float)g;
        }
}

/* Permutation of (token, slot) pairs to expert-contiguous rows.
 *   counts[e]  = #{(t,k) : idx[t,k] = e}
 *   offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e]
 *   pair_row[t,k] = offsets[e] + #{t' < t : e in idx[t',:]}   (e = idx[t,k])
 *   row_token[pair_row[t,k]] = t
 * i.e. a stable counting sort by expert of the pairs taken in (t,k) order
 * (reading: ascending token order inside an expert; no capacity limit). */
void oracle_permute(int64_t T, int64_t K, int64_t N, const int32_t *idx, int32_t *counts,
                    int32_t *offsets, int32_t *pair_row, int32_t *row_token) {
    for (int64_t e = 0; e < N; ++e) counts[e] = 0;
    for (int64_t i = 0; i < T * K; ++i) counts[idx[i]] += 1;
    offsets[0] = 0;
    for (int64_t e = 0; e < N; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t *next = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
    for (int64_t e = 0; e < N; ++e) next[e] = offsets[e];
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = 0; k < K; ++k) {
            int32_t e = idx[t * K + k];
            int32_t row = next[e]++;
            pair_row[t * K + k] = row;
            if (row_token) row_token[row] = (int32_t)t;
        }
    free(next);
}

/* Per-group load and imbalance score [EXPL-1]: load_g = sum of counts over
 * the experts of group g (one group = one device); score = (max_g load_g -
 * min_g load_g) / T (reading: normalised by the token count). */
double oracle_imbalance(int64_t T, int64_t N, int64_t M, const int32_t *counts, int32_t *group_load) {
    const int64_t G = N / M;
    int64_t mx = 0, mn = 0;
    for (int64_t g = 0; g < M; ++g) {
        int64_t s = 0;
        for (int64_t e = g * G; e < (g + 1) * G; ++e) s += counts[e];
        if (group_load) group_load[g] = (int32_t)s;
        if (g == 0 || s > mx) mx = s;
        if (g == 0 || s < mn) mn = s;
    }
    return (double)(mx - mn) / (double)T;
}

/* One expert's SwiGLU FFN on one token (reading: SwiGLU form), all double:
 *   a = W_gate[e] x,  u = W_up[e] x,  h = a * sigmoid(a) * u,  o = W_down[e] h. */
static void expert_ffn_token(int64_t d, int64_t I, int dtype, const void *x, int64_t t, int64_t e,
                             const void *w_gate, const void *w_up, const void *w_down, double *h,
                             double *o) {
    for (int64_t f = 0; f < I; ++f) {
        double a = 0.0, u = 0.0;
        const int64_t wrow = (e * I + f) * d;
        for (int64_t i = 0; i < d; ++i) {
            double xi = val(x, dtype, t * d + i);
            a += val(w_gate, dtype, wrow + i) * xi;
            u += val(w_up, dtype, wrow + i) * xi;
        }
        h[f] = a / (1.0 + exp(-a)) * u;
    }
    for (int64_t j = 0; j < d; ++j) {
        double s = 0.0;
        const int64_t wrow = (e * d + j) * I;
        for (int64_t f = 0; f < I; ++f) s += val(w_down, dtype, wrow + f) * h[f];
        o[j] = s;
    }
}

/* Expert outputs of chosen (token, expert) pairs: o[p, :] = FFN_{expert[p]}(x[token[p]]). */
void oracle_expert_ffn_pairs(int64_t n_pairs, const int32_t *token, const int32_t *expert, int64_t d,
                             int64_t I, int dtype, const void *x, const void *w_gate, const void *w_up,
                             const void *w_down, double *o) {
#pragma omp parallel
    {
        double *h = (double *)malloc(sizeof(double) * (size_t)I);
#pragma omp for schedule(dynamic, 1)
        for (int64_t p = 0; p < n_pairs; ++p)
            expert_ffn_token(d, I, dtype, x, token[p], expert[p], w_gate, w_up, w_down, h, o + p * d);
        free(h);
    }
}

/* Weighted combine of listed tokens [EXPL-1 routing + reading: gates weight
 * the expert outputs, summed in slot order]:
 *   y[t] = sum_{k=0..K-1} gate[t,k] * FFN_{idx[t,k]}(x[t])   (double). */
void oracle_combine_tokens(int64_t n_tok, const int32_t *tokens, int64_t K, const int32_t *idx,
                           const double *gate64, int64_t d, int64_t I, int dtype, const void *x,
                           const void *w_gate, const void *w_up, const void *w_down, double *y) {
#pragma omp parallel
    {
        double *h = (double *)malloc(sizeof(double) * (size_t)I);
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t n = 0; n < n_tok; ++n) {
            const int64_t t = tokens[n];
            double *yt = y + n * d;
            for (int64_t j = 0; j < d; ++j) yt[j] = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                expert_ffn_token(d, I, dtype, x, t, idx[t * K + k], w_gate, w_up, w_down, h, o);
                const double g = gate64[t * K + k];
                for (int64_t j = 0; j < d; ++j) yt[j] += g * o[j];
            }
        }
        free(h);
        free(o);
    }
}

/* The combine step alone, on given expert-output rows (reading: gates weight
 * the expert outputs, summed in slot order):
 *   y[t,:] = sum_k gate[t,k] * rows[pair_row[t,k], :]   (double; rows of any dtype). */
void oracle_combine_rows(int64_t T, int64_t K, int64_t d, int dtype, const void *rows, const int32_t *pair_row,
                         const double *gate64, double *y) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double *yt = y + t * d;
        for (int64_t j = 0; j < d; ++j) yt[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const int64_t r = pair_row[t * K + k];
            const double g = gate64[t * K + k];
            for (int64_t j = 0; j < d; ++j) yt[j] += g * val(rows, dtype, r * d + j);
        }
    }
}
