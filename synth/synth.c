/*
 * Seeded synthetic inputs for the MoGE layer (input generation only).
 *
 * This file holds no arithmetic of the layer itself: it only draws numbers.
 * Both the CPU oracle and the CUDA path consume the arrays it writes, so the
 * two sides always see identical inputs.
 *
 * Generator (counter based, so the output does not depend on thread count):
 *   key(seed, tensor) = splitmix64(seed XOR tensor_id)
 *   word(i)           = splitmix64(key + i)
 * splitmix64 is the 64-bit mixer of Steele, Lea and Flood ("Fast splittable
 * pseudorandom number generators", OOPSLA 2014), written here from that
 * definition: add the golden-ratio increment, then two xor-shift-multiply
 * rounds and a final xor-shift.
 *
 * Normal draws use the Box-Muller transform (Box and Muller, 1958) on the pair
 * of words (2j, 2j+1): u1 in (0,1], u2 in [0,1), r = sqrt(-2 ln u1); element
 * 2j takes r*cos(2 pi u2) and element 2j+1 takes r*sin(2 pi u2). All of it in
 * double, then scaled by the requested standard deviation and rounded once to
 * fp32. bf16 values are the fp32 values rounded to nearest-even.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static inline uint64_t mix64(uint64_t z) {
    z += 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tensor_id) {
    return mix64(seed ^ tensor_id);
}

/* Both normals of pair j. */
static inline void normal_pair(uint64_t key, uint64_t j, double *z0, double *z1) {
    uint64_t w1 = mix64(key + 2 * j);
    uint64_t w2 = mix64(key + 2 * j + 1);
    double u1 = (double)((w1 >> 11) + 1) * 0x1p-53; /* (0, 1] */
    double u2 = (double)(w2 >> 11) * 0x1p-53;       /* [0, 1) */
    double r = sqrt(-2.0 * log(u1));
    double a = 6.283185307179586476925286766559 * u2;
    *z0 = r * cos(a);
    *z1 = r * sin(a);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u); /* finite inputs only */
    return (uint16_t)(u >> 16);
}

/* Writes element g of the stream (if it lies in [start, start+count)) to
 * out[g - start] through put(); pairs are computed once for both elements. */
#define SYNTH_NORMAL_LOOP(PUT)                                                         \
    const uint64_t key = stream_key(seed, tensor_id);                                  \
    if (count == 0) return;                                                            \
    const int64_t j0 = (int64_t)(start >> 1), j1 = (int64_t)((start + count - 1) >> 1); \
    _Pragma("omp parallel for schedule(static)")                                       \
    for (int64_t j = j0; j <= j1; ++j) {                                               \
        double z[2];                                                                   \
        normal_pair(key, (uint64_t)j, &z[0], &z[1]);                                   \
        for (int h = 0; h < 2; ++h) {                                                  \
            uint64_t g = 2 * (uint64_t)j + (uint64_t)h;                                \
            if (g < start || g >= start + count) continue;                             \
            PUT(out[g - start], (float)(stddev * z[h]));                               \
        }                                                                              \
    }

#define PUT_F32(dst, v) (dst) = (v)
#define PUT_BF16(dst, v) (dst) = f32_to_bf16_rne(v)

/* Elements [start, start+count) of the stream, as fp32 (std * N(0,1)). */
void synth_normal_f32(uint64_t seed, uint64_t tensor_id, uint64_t start, uint64_t count,
                      double stddev, float *out) {
    SYNTH_NORMAL_LOOP(PUT_F32)
}

/* Same stream, rounded on to bf16 (stored as raw uint16 bits). */
void synth_normal_bf16(uint64_t seed, uint64_t tensor_id, uint64_t start, uint64_t count,
                       double stddev, uint16_t *out) {
    SYNTH_NORMAL_LOOP(PUT_BF16)
}

/* fp32 -> bf16 (nearest-even) for an existing array. */
void synth_f32_to_bf16(const float *in, uint64_t count, uint16_t *out) {
    const int64_t n = (int64_t)count;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(in[i]);
}

/* Seeded permutation of 1..n (Fisher-Yates, descending i, j = word(i) mod (i+1)). */
void synth_rank_permutation(uint64_t seed, uint64_t tensor_id, int64_t n, int32_t *rank) {
    const uint64_t key = stream_key(seed, tensor_id);
    for (int64_t i = 0; i < n; ++i) rank[i] = (int32_t)(i + 1);
    for (int64_t i = n - 1; i > 0; --i) {
        int64_t j = (int64_t)(mix64(key + (uint64_t)i) % (uint64_t)(i + 1));
        int32_t t = rank[i];
        rank[i] = rank[j];
        rank[j] = t;
    }
}

/* Popularity skew of the router: b_e = scale * ln(1 / rank_e), rounded to fp32. */
void synth_rank_bias(const int32_t *rank, int64_t n, double scale, float *bias) {
    for (int64_t i = 0; i < n; ++i) bias[i] = (float)(scale * log(1.0 / (double)rank[i]));
}

/* Scores of the imbalance Monte-Carlo study: element i of the stream (i = (b*T + t)*N + e for
 * batch b, token t, expert e) is an Irwin-Hall approximation of N(0,1) built from three words,
 *   words w_j = word(3i + j), j = 0..2;  S = sum of the twelve 16-bit fields of w_0..w_2;
 *   z = (2S + 12) / 2^17 - 6  ( = sum of twelve uniforms (u + 1/2)/2^16, minus 6 ).
 * Every step is exact in fp32 (2S + 12 < 2^21), so any implementation of this definition
 * produces the same bits.  Writes batches [b0, b0 + nb) as [nb][T][N]. */
void synth_study_scores(uint64_t seed, uint64_t tensor_id, int64_t b0, int64_t nb, int64_t T, int64_t N,
                        float *out) {
    const uint64_t key = stream_key(seed, tensor_id);
    const int64_t n = nb * T * N;
    const uint64_t first = (uint64_t)b0 * (uint64_t)T * (uint64_t)N;
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < n; ++k) {
        const uint64_t i = first + (uint64_t)k;
        uint32_t S = 0;
        for (int j = 0; j < 3; ++j) {
            const uint64_t w = mix64(key + 3 * i + (uint64_t)j);
            S += (uint32_t)(w & 0xFFFFu) + (uint32_t)((w >> 16) & 0xFFFFu) + (uint32_t)((w >> 32) & 0xFFFFu) +
                 (uint32_t)(w >> 48);
        }
        out[k] = (float)(2u * S + 12u) * (1.0f / 131072.0f) - 6.0f;
    }
}

int synth_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
