/*
 * Seeded synthetic input generator shared by the tests, the bench and the
 * oracle's callers.  It holds none of the attention arithmetic: it only turns
 * (seed, counter) pairs into pseudo-random bits.
 *
 *  - SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
 *    generators", OOPSLA 2014): state advances by the golden-ratio gamma and
 *    each output is the state passed through the published 64-bit finaliser.
 *    Output i of a stream seeded with s is mix(s + (i + 1) * gamma), so any
 *    element can be produced on its own (counter-based use).
 *  - Standard normals by the Box-Muller transform (1958), both branches used:
 *    element 2k is r*cos(2 pi u2), element 2k+1 is r*sin(2 pi u2) with
 *    r = sqrt(-2 ln u1), u1, u2 taken from outputs 2k and 2k+1.
 *  - Bounded integers by Lemire's multiply-shift with rejection ("Fast random
 *    integer generation in an interval", ACM TOMACS 2019).
 *
 * Compiled with -ffp-contract=off so x86-64 and aarch64 builds give the same
 * doubles.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define WL_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t wl_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Output i (0-based) of the SplitMix64 stream seeded with `seed`. */
uint64_t wl_splitmix64_at(uint64_t seed, uint64_t i) {
    return wl_mix(seed + (i + 1) * WL_GAMMA);
}

/* Fill out[0..count) with outputs start..start+count of the stream. */
void wl_splitmix64_fill(uint64_t seed, uint64_t start, int64_t count, uint64_t* out) {
    for (int64_t k = 0; k < count; ++k) out[k] = wl_splitmix64_at(seed, start + (uint64_t)k);
}

/* A sub-stream seed: the SplitMix64 output `tag` of the stream seeded by `base`. */
uint64_t wl_derive_seed(uint64_t base, uint64_t tag) { return wl_splitmix64_at(base, tag); }

/* Uniform double in (0, 1]: top 53 bits plus one, over 2^53. */
static inline double wl_u01(uint64_t x) { return (double)((x >> 11) + 1) * (1.0 / 9007199254740992.0); }

static inline double wl_normal_at(uint64_t seed, uint64_t e) {
    uint64_t k = e >> 1;
    double u1 = wl_u01(wl_splitmix64_at(seed, 2 * k));
    double u2 = wl_u01(wl_splitmix64_at(seed, 2 * k + 1));
    double r = sqrt(-2.0 * log(u1));
    double a = 6.283185307179586476925286766559 * u2;
    return (e & 1) ? r * sin(a) : r * cos(a);
}

/* Element e of the normal stream, as double (before any narrowing). */
double wl_normal_f64_at(uint64_t seed, uint64_t e) { return wl_normal_at(seed, e); }

/* float32 round-to-nearest-even from double is the C cast (IEEE default mode). */
static inline uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* float32 -> bfloat16 bits, round to nearest even (inputs here are finite). */
static inline uint16_t wl_f32_to_bf16(float f) {
    uint32_t u = f32_bits(f);
    uint32_t bias = 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)((u + bias) >> 16);
}

/* float32 -> binary16 bits, round to nearest even, finite inputs of modest size. */
static inline uint16_t wl_f32_to_f16(float f) {
    uint32_t u = f32_bits(f);
    uint32_t sign = (u >> 16) & 0x8000u;
    int32_t exp = (int32_t)((u >> 23) & 0xFF) - 127;
    uint32_t man = u & 0x7FFFFFu;
    if (exp > 15) return (uint16_t)(sign | 0x7C00u); /* overflow -> inf (never hit by N(0,1)) */
    if (exp >= -14) {                                 /* normal binary16 */
        uint32_t m = man >> 13, rest = man & 0x1FFFu;
        uint32_t h = ((uint32_t)(exp + 15) << 10) | m;
        if (rest > 0x1000u || (rest == 0x1000u && (m & 1u))) h += 1; /* carry may bump exponent */
        return (uint16_t)(sign | h);
    }
    if (exp < -25) return (uint16_t)sign;             /* below half the smallest subnormal */
    /* subnormal: value = man24 * 2^(exp-23), unit 2^-24 */
    uint32_t man24 = man | 0x800000u;
    int shift = -exp - 1; /* = 13 + (-14 - exp) */
    uint32_t m = man24 >> shift, rest = man24 & ((1u << shift) - 1u), half = 1u << (shift - 1);
    if (rest > half || (rest == half && (m & 1u))) m += 1;
    return (uint16_t)(sign | m);
}

/* dtype: 0 = float16, 1 = bfloat16 */
void wl_normal_bits(uint64_t seed, uint64_t start, int64_t count, int dtype, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < count; ++k) {
        float f = (float)wl_normal_at(seed, start + (uint64_t)k);
        out[k] = dtype ? wl_f32_to_bf16(f) : wl_f32_to_f16(f);
    }
}

/* The same normals, kept in float32. */
void wl_normal_f32(uint64_t seed, uint64_t start, int64_t count, float* out) {
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < count; ++k) out[k] = (float)wl_normal_at(seed, start + (uint64_t)k);
}

/* ---- sequential integer draws -------------------------------------------------- */

typedef struct { uint64_t seed; uint64_t i; } wl_seq;

static inline uint64_t wl_next(wl_seq* r) { return wl_splitmix64_at(r->seed, r->i++); }

/* Unbiased integer in [0, n), n >= 1 (Lemire). */
static uint64_t wl_bounded(wl_seq* r, uint64_t n) {
    unsigned __int128 m = (unsigned __int128)wl_next(r) * n;
    uint64_t lo = (uint64_t)m;
    if (lo < n) {
        uint64_t t = (0 - n) % n;
        while (lo < t) {
            m = (unsigned __int128)wl_next(r) * n;
            lo = (uint64_t)m;
        }
    }
    return (uint64_t)(m >> 64);
}

/* count integers uniform on [lo, hi] (inclusive). */
void wl_uniform_ints(uint64_t seed, int64_t count, int64_t lo, int64_t hi, int64_t* out) {
    wl_seq r = {seed, 0};
    uint64_t n = (uint64_t)(hi - lo) + 1;
    for (int64_t k = 0; k < count; ++k) out[k] = lo + (int64_t)wl_bounded(&r, n);
}

/* A uniformly random permutation of 0..n-1 (Fisher-Yates, Durstenfeld form). */
void wl_permutation(uint64_t seed, int64_t n, int64_t* out) {
    wl_seq r = {seed, 0};
    for (int64_t k = 0; k < n; ++k) out[k] = k;
    for (int64_t k = n - 1; k > 0; --k) {
        int64_t j = (int64_t)wl_bounded(&r, (uint64_t)k + 1);
        int64_t t = out[k]; out[k] = out[j]; out[j] = t;
    }
}
