/*
 * Seeded synthetic input generators shared by the oracle tests and the GPU
 * tests/bench.  This file holds no arithmetic of the tile-movement method or
 * of the GEMM: it only turns (seed, element index) into numbers.
 *
 * Every value is a pure function of (seed, i), built on the counter-based
 * form of SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014): the i-th output of a stream is the
 * SplitMix64 finaliser applied to seed + (i + 1) * golden_gamma.  Output is
 * therefore identical at any thread count.
 *
 * Derived distributions:
 *   uniform [0,1)   : (h >> 40) * 2^-24                    (24 random bits)
 *   int in [0, n)   : ((h >> 32) * n) >> 32                (Lemire 2019)
 *   N(0,1)          : Box-Muller (1958) in double on
 *                     u1 = ((h(2i) >> 11) + 1) * 2^-53, u2 = (h(2i+1) >> 11) * 2^-53
 *   permutation     : Fisher-Yates / Durstenfeld shuffle, draws from one stream
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t synth_h(uint64_t seed, uint64_t i) { return mix64(seed + (i + 1) * SYNTH_GAMMA); }

static inline double unit24(uint64_t h) { return (double)(h >> 40) * (1.0 / 16777216.0); }

/* Round a float to bf16 bits, round-to-nearest-even (NaN kept quiet). */
static inline uint16_t f32_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void synth_u64(uint64_t seed, int64_t n, uint64_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = synth_h(seed, (uint64_t)i);
}

/* x = lo + (hi - lo) * u, u uniform [0,1) on 24 bits; computed in double, stored fp32. */
void synth_uniform_f32(uint64_t seed, int64_t n, double lo, double hi, float* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(lo + (hi - lo) * unit24(synth_h(seed, (uint64_t)i)));
}

/* The same uniform numbers as synth_uniform_f32, in double. */
void synth_uniform_f64(uint64_t seed, int64_t n, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = unit24(synth_h(seed, (uint64_t)i));
}

static inline double normal_at(uint64_t seed, uint64_t i) {
    double u1 = (double)((synth_h(seed, 2 * i) >> 11) + 1) * (1.0 / 9007199254740992.0);
    double u2 = (double)(synth_h(seed, 2 * i + 1) >> 11) * (1.0 / 9007199254740992.0);
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

/* N(0,1) in double, rounded to fp32 (RNE) then to bf16 bits (RNE). */
void synth_normal_bf16(uint64_t seed, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_bits((float)normal_at(seed, (uint64_t)i));
}

void synth_normal_f32(uint64_t seed, int64_t n, float* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (float)normal_at(seed, (uint64_t)i);
}

/* lo + int in [0, n_range) for each element; n_range <= 2^32. */
void synth_int_below(uint64_t seed, int64_t n, uint64_t n_range, int64_t lo, int64_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = lo + (int64_t)(((synth_h(seed, (uint64_t)i) >> 32) * n_range) >> 32);
}

/* 1 with probability p (u < p on the 24-bit uniform), else 0. */
void synth_bernoulli_u8(uint64_t seed, int64_t n, double p, uint8_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = unit24(synth_h(seed, (uint64_t)i)) < p ? 1 : 0;
}

/* First n_out entries of a uniformly random permutation of [0, n_total),
 * Durstenfeld's in-place Fisher-Yates on one stream; work holds n_total int32. */
void synth_permutation_prefix(uint64_t seed, int64_t n_total, int64_t n_out, int32_t* work, int32_t* out) {
    for (int64_t i = 0; i < n_total; ++i) work[i] = (int32_t)i;
    uint64_t draw = 0;
    for (int64_t i = n_total - 1; i > 0; --i) {
        uint64_t j = ((synth_h(seed, draw++) >> 32) * (uint64_t)(i + 1)) >> 32;
        int32_t t = work[i];
        work[i] = work[j];
        work[j] = t;
    }
    memcpy(out, work, (size_t)n_out * sizeof(int32_t));
}
