/*
 * Seeded synthetic inputs: weights, token streams and uniform draws.
 *
 * This file holds only input generation. It computes nothing of the
 * speculative-decoding method; the oracle and the GPU path both consume the
 * arrays it writes.
 *
 * Definition (counter-based, so any element can be produced independently):
 *   key(seed, name) = mix64(seed ^ fnv1a64(name))
 *   u64(key, i)     = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)
 * where mix64 is the SplitMix64 output function (Steele, Lea and Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014; constants as
 * published by Vigna), and fnv1a64 is the 64-bit FNV-1a hash of the name.
 *
 *   normal(i)  : p = floor(i/2),
 *                u1 = ((u64(2p) >> 11) + 1) * 2^-53 in (0,1],
 *                u2 = (u64(2p+1) >> 11) * 2^-53 in [0,1),
 *                z  = sqrt(-2 ln u1) * (i even ? cos : sin)(2 pi u2)   (Box-Muller pair)
 *   weight(i)  : bf16_rne((float)(std * z))
 *   token(i)   : floor(u64(i) * V / 2^64)                      (multiply-high)
 *   unit(i)    : (u64(i) >> 11) * 2^-53 in [0,1)
 *   int(i)     : lo + floor(u64(i) * (hi - lo + 1) / 2^64)
 *
 * Portable C99: no intrinsics, no architecture flags; results are identical on
 * x86_64 and aarch64 up to the last-ulp behaviour of libm log/cos, which can
 * change a bf16 weight only when the fp64 value sits within one ulp of a bf16
 * rounding midpoint.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static uint64_t fnv1a64(const char *s) {
    uint64_t h = 0xcbf29ce484222325ULL;
    for (const unsigned char *p = (const unsigned char *)s; *p; ++p) {
        h ^= (uint64_t)(*p);
        h *= 0x100000001b3ULL;
    }
    return h;
}

uint64_t synth_key(uint64_t seed, const char *name) { return mix64(seed ^ fnv1a64(name)); }

uint64_t synth_u64(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

static uint64_t mulhi64(uint64_t a, uint64_t b) {
    /* floor(a*b / 2^64) without a 128-bit type: split into 32-bit halves. */
    uint64_t a_lo = a & 0xFFFFFFFFULL, a_hi = a >> 32;
    uint64_t b_lo = b & 0xFFFFFFFFULL, b_hi = b >> 32;
    uint64_t lo_lo = a_lo * b_lo;
    uint64_t hi_lo = a_hi * b_lo;
    uint64_t lo_hi = a_lo * b_hi;
    uint64_t hi_hi = a_hi * b_hi;
    uint64_t cross = (lo_lo >> 32) + (hi_lo & 0xFFFFFFFFULL) + lo_hi;
    return hi_hi + (hi_lo >> 32) + (cross >> 32);
}

static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

static const double TWO_PI = 6.283185307179586476925286766559;
static const double TWO_M53 = 1.0 / 9007199254740992.0;

double synth_normal_at(uint64_t key, uint64_t i) {
    uint64_t p = i >> 1;
    double u1 = (double)((synth_u64(key, 2 * p) >> 11) + 1) * TWO_M53;
    double u2 = (double)(synth_u64(key, 2 * p + 1) >> 11) * TWO_M53;
    double r = sqrt(-2.0 * log(u1));
    return (i & 1) ? r * sin(TWO_PI * u2) : r * cos(TWO_PI * u2);
}

/* bf16 bit patterns of std * N(0,1), elements [offset, offset + n). */
void synth_normal_bf16(uint64_t seed, const char *name, double stdev, uint64_t offset, uint64_t n,
                       uint16_t *out) {
    uint64_t key = synth_key(seed, name);
    if (n == 0) return;
    uint64_t first_pair = offset >> 1, last_pair = (offset + n - 1) >> 1;
    long long npairs = (long long)(last_pair - first_pair + 1);
#pragma omp parallel for schedule(static)
    for (long long q = 0; q < npairs; ++q) {
        uint64_t p = first_pair + (uint64_t)q;
        double u1 = (double)((synth_u64(key, 2 * p) >> 11) + 1) * TWO_M53;
        double u2 = (double)(synth_u64(key, 2 * p + 1) >> 11) * TWO_M53;
        double r = sqrt(-2.0 * log(u1));
        uint64_t i0 = 2 * p, i1 = 2 * p + 1;
        if (i0 >= offset && i0 < offset + n) out[i0 - offset] = f32_to_bf16_rne((float)(stdev * r * cos(TWO_PI * u2)));
        if (i1 >= offset && i1 < offset + n) out[i1 - offset] = f32_to_bf16_rne((float)(stdev * r * sin(TWO_PI * u2)));
    }
}

/* Tokens uniform in [0, vocab). */
void synth_tokens(uint64_t seed, const char *name, uint64_t offset, uint64_t n, uint32_t vocab,
                  int32_t *out) {
    uint64_t key = synth_key(seed, name);
    long long nn = (long long)n;
#pragma omp parallel for schedule(static)
    for (long long j = 0; j < nn; ++j)
        out[j] = (int32_t)mulhi64(synth_u64(key, offset + (uint64_t)j), (uint64_t)vocab);
}

/* Uniform doubles in [0, 1). */
void synth_unit(uint64_t seed, const char *name, uint64_t offset, uint64_t n, double *out) {
    uint64_t key = synth_key(seed, name);
    for (uint64_t j = 0; j < n; ++j) out[j] = (double)(synth_u64(key, offset + j) >> 11) * TWO_M53;
}

/* Integers uniform in [lo, hi] (inclusive). */
void synth_ints(uint64_t seed, const char *name, uint64_t offset, uint64_t n, int64_t lo, int64_t hi,
                int64_t *out) {
    uint64_t key = synth_key(seed, name);
    uint64_t span = (uint64_t)(hi - lo) + 1;
    for (uint64_t j = 0; j < n; ++j) out[j] = lo + (int64_t)mulhi64(synth_u64(key, offset + j), span);
}
