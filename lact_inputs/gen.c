/*
 * Seeded synthetic inputs for the LaCT fast-weight chunk step.
 *
 * This file holds no arithmetic of the method itself: it only draws the
 * tensors that, in a LaCT block, the slow-weight projections would produce
 * (queries, keys, values, per-token learning rates) and the initial fast
 * weights. Both the CPU oracle and the CUDA path take their inputs from here,
 * so the two sides see bit-identical values.
 *
 * Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014; the 64-bit finaliser constants as in
 * Vigna's public-domain splitmix64.c), used in counter mode:
 *     key(seed, stream) = mix(seed + (stream + 1) * GAMMA)
 *     draw(seed, stream, i) = mix(key + (i + 1) * GAMMA)
 * so element i of a stream does not depend on how the work is split across
 * threads. Normals come from the Box-Muller transform on pairs of draws:
 * pair j = (draw 2j, draw 2j+1) gives elements 2j (cos branch) and 2j+1
 * (sin branch).
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (see build.py).
 * -ffp-contract=off keeps the arithmetic free of FMA contraction so the
 * values do not depend on the host compiler's choices.
 */
#include <stdint.h>
#include <math.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(seed + (stream + 1) * GAMMA);
}

static inline uint64_t draw(uint64_t key, uint64_t i) {
    return mix64(key + (i + 1) * GAMMA);
}

/* Standard normal number i of the stream with the given key (fp64). */
static inline double normal_at(uint64_t key, uint64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    uint64_t j = i >> 1;
    uint64_t x1 = draw(key, 2 * j), x2 = draw(key, 2 * j + 1);
    double u1 = ((double)(x1 >> 11) + 0.5) * (1.0 / 9007199254740992.0); /* (0,1) */
    double u2 = ((double)(x2 >> 11)) * (1.0 / 9007199254740992.0);       /* [0,1) */
    double r = sqrt(-2.0 * log(u1));
    return (i & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
}

/* fp32 -> bf16 bit pattern, round to nearest even (finite inputs). */
static inline uint16_t f32_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

static inline void store(void* out, int64_t idx, float f, int as_bf16) {
    if (as_bf16) ((uint16_t*)out)[idx] = f32_to_bf16_bits(f);
    else ((float*)out)[idx] = f;
}

/* Raw SplitMix64 draws of one stream (exposed for the generator's own tests). */
void lact_gen_draws(uint64_t seed, uint64_t stream, int64_t n, uint64_t* out) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = draw(key, (uint64_t)i);
}

/* Sequential SplitMix64 from a raw state (state += GAMMA; out = mix(state)),
 * i.e. the textbook form, exposed so tests can compare with published values. */
void lact_gen_splitmix_sequence(uint64_t state, int64_t n, uint64_t* out) {
    for (int64_t i = 0; i < n; ++i) { state += GAMMA; out[i] = mix64(state); }
}

/* out[i] = round_fp32(scale * N_i), i in [0, n); optionally stored as bf16
 * (the fp32 value rounded to nearest even). */
void lact_gen_normal(uint64_t seed, uint64_t stream, int64_t n, double scale,
                     int as_bf16, void* out) {
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        store(out, i, (float)(scale * normal_at(key, (uint64_t)i)), as_bf16);
}

/* rows x d normals, each row divided by its own L2 norm (fp64), rounded to
 * fp32, then optionally to bf16. This is the per-token normalisation of
 * queries and keys in the synthetic workloads. */
void lact_gen_unit_rows(uint64_t seed, uint64_t stream, int64_t rows, int64_t d,
                        int as_bf16, void* out) {
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double buf[1024];
        double ss = 0.0;
        for (int64_t c = 0; c < d; ++c) {
            double z = normal_at(key, (uint64_t)(r * d + c));
            buf[c] = z;
            ss += z * z;
        }
        double inv = 1.0 / sqrt(ss);
        for (int64_t c = 0; c < d; ++c) store(out, r * d + c, (float)(buf[c] * inv), as_bf16);
    }
}

/* Per-token learning rates: eta_i = round_fp32(0.01 * log1p(exp(z_i))). */
void lact_gen_eta(uint64_t seed, uint64_t stream, int64_t n, float* out) {
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double z = normal_at(key, (uint64_t)i);
        out[i] = (float)(0.01 * log1p(exp(z)));
    }
}
