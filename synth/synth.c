/*
 * Seeded synthetic inputs for the gpt-oss MoE layer (activations, router,
 * expert weights and biases, MXFP4 codes and block scales).
 *
 * This file holds no arithmetic of the MoE layer itself: it only draws random
 * numbers and rounds them to the storage formats. Both the CPU oracle (via the
 * tests) and the CUDA library (via the tests and the benchmark) read the
 * buffers it fills, so the two sides always see identical inputs.
 *
 * Generator: splitmix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014; the finaliser constants are
 * Vigna's public-domain ones) used in counter mode.  Draw i of stream s under
 * seed q is  mix(key(q, s) + (i + 1) * GOLDEN),  which is exactly the i-th
 * output of a splitmix64 sequence started at key(q, s).  Being counter-based,
 * every element is independent of the thread that computes it, so results do
 * not depend on the OpenMP thread count.
 *
 * Normals: Box-Muller on two 24-bit uniforms taken from one 64-bit draw,
 * u1 in (0, 1] (so log(u1) is finite) and u2 in [0, 1), evaluated in double.
 * bf16: round-to-nearest-even of the fp32 value.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ull

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(mix64(seed + GOLDEN) ^ (stream * 0xD1B54A32D192ED03ull));
}

static inline uint64_t draw(uint64_t key, uint64_t i) {
    return mix64(key + (i + 1) * GOLDEN);
}

static inline double normal_from(uint64_t r) {
    const double two24 = 16777216.0;
    double u1 = ((double)(r >> 40) + 1.0) / two24;        /* (0, 1] */
    double u2 = (double)(r & 0xFFFFFFull) / two24;        /* [0, 1) */
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

static inline double uniform01(uint64_t r) {             /* [0, 1) */
    return (double)(r >> 40) / 16777216.0;
}

uint16_t synth_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u) {               /* inf / nan */
        return (uint16_t)((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
    }
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* out[i] = fp32(mean + std * N(0,1)) for i in [0, n). */
void synth_normal_f32(float* out, size_t n, uint64_t seed, uint64_t stream,
                      double mean, double std) {
    const uint64_t key = stream_key(seed, stream);
    long long nn = (long long)n;
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < nn; ++i)
        out[i] = (float)(mean + std * normal_from(draw(key, (uint64_t)i)));
}

/* out[i] = bf16(mean + std * N(0,1)); when p_outlier > 0, an independent
 * Bernoulli(p_outlier) draw (stream + 0x1000) multiplies the value by
 * outlier_scale before rounding. */
void synth_normal_bf16(uint16_t* out, size_t n, uint64_t seed, uint64_t stream,
                       double mean, double std, double p_outlier,
                       double outlier_scale) {
    const uint64_t key = stream_key(seed, stream);
    const uint64_t okey = stream_key(seed, stream + 0x1000);
    long long nn = (long long)n;
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < nn; ++i) {
        double v = mean + std * normal_from(draw(key, (uint64_t)i));
        if (p_outlier > 0.0 && uniform01(draw(okey, (uint64_t)i)) < p_outlier)
            v *= outlier_scale;
        out[i] = synth_f32_to_bf16((float)v);
    }
}

/* out[i] uniform over the integers [lo, hi] (hi - lo < 2^32). */
void synth_uniform_u8(uint8_t* out, size_t n, uint64_t seed, uint64_t stream,
                      uint32_t lo, uint32_t hi) {
    const uint64_t key = stream_key(seed, stream);
    const uint64_t span = (uint64_t)(hi - lo) + 1u;
    long long nn = (long long)n;
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < nn; ++i) {
        uint64_t r = draw(key, (uint64_t)i) >> 32;
        out[i] = (uint8_t)(lo + ((r * span) >> 32));
    }
}

/* fp32 -> bf16 (round to nearest even), element-wise. */
void synth_round_bf16(const float* in, uint16_t* out, size_t n) {
    long long nn = (long long)n;
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < nn; ++i) out[i] = synth_f32_to_bf16(in[i]);
}
