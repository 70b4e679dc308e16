/*
 * Seeded synthetic inputs shared by the oracle side and the CUDA side.
 *
 * This file holds no arithmetic of the prefill method: it only draws numbers.
 * Every tensor is a pure function of (seed, name, layer, element index), so any
 * slice can be regenerated on its own and both sides see identical bits.
 *
 *   key(seed, name, layer) = mix64(seed * K1 ^ fnv1a64(name) ^ (layer + 1) * K2)
 *   draw(key, i)           = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)
 *
 * mix64 is the splitmix64 output finalizer (Steele, Lea and Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014), so draw(key, i) is
 * the i-th output of a splitmix64 stream started at `key`.
 *
 * Normals use the Box-Muller transform in fp64 (element 2j from the cosine and
 * 2j+1 from the sine of the pair drawn at 2j, 2j+1), then round to nearest even
 * into fp16 (or fp32).  Bounded integers use Lemire's multiply-shift on the top
 * 32 bits of a draw.  Bytes are the little-endian bytes of successive draws.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define K1 0xD1B54A32D192ED03ull
#define K2 0xABC98388FB8FAC03ull
#define GOLDEN 0x9E3779B97F4A7C15ull

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static uint64_t fnv1a64(const char *s) {
    uint64_t h = 0xCBF29CE484222325ull;
    for (; *s; ++s) {
        h ^= (uint64_t)(unsigned char)*s;
        h *= 0x100000001B3ull;
    }
    return h;
}

uint64_t synth_key(uint64_t seed, const char *name, int64_t layer) {
    return mix64(seed * K1 ^ fnv1a64(name) ^ (uint64_t)(layer + 1) * K2);
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

/* uniform in (0, 1]: never 0, so log() is finite */
static inline double unif_open0(uint64_t d) { return (double)((d >> 11) + 1) * 0x1.0p-53; }
static inline double unif(uint64_t d) { return (double)(d >> 11) * 0x1.0p-53; }

static inline double normal_at(uint64_t key, int64_t i) {
    int64_t j = i & ~(int64_t)1;
    double u1 = unif_open0(draw(key, (uint64_t)j));
    double u2 = unif(draw(key, (uint64_t)j + 1));
    double r = sqrt(-2.0 * log(u1));
    double a = 6.283185307179586476925 * u2;
    return (i & 1) ? r * sin(a) : r * cos(a);
}

/* IEEE binary16, round to nearest even, from a double (no double rounding). */
static uint16_t f64_to_f16(double x) {
    uint64_t b;
    memcpy(&b, &x, 8);
    uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
    int exp = (int)((b >> 52) & 0x7FF);
    uint64_t man = b & 0xFFFFFFFFFFFFFull;
    if (exp == 0x7FF) return sign | 0x7C00u | (man ? 0x200u : 0u);
    if (exp == 0 && man == 0) return sign;
    /* value = 1.man * 2^(exp-1023) for normal doubles; doubles that are
       subnormal are far below the fp16 range and round to zero. */
    if (exp == 0) return sign;
    int e = exp - 1023;
    uint64_t m = man | (1ull << 52); /* 53-bit significand */
    int shift;                       /* bits to drop from m */
    uint16_t hexp;
    if (e > 15) return sign | 0x7C00u;
    if (e >= -14) {
        hexp = (uint16_t)(e + 15);
        shift = 42; /* keep 11 bits */
    } else {
        hexp = 0;
        shift = 42 + (-14 - e); /* subnormal: fewer kept bits */
        if (shift > 63) return sign;
    }
    uint64_t kept = m >> shift;
    uint64_t rem = m & ((1ull << shift) - 1);
    uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (kept & 1))) kept++;
    if (hexp == 0) {
        /* subnormal (kept may have carried into the normal range: 0x400) */
        return sign | (uint16_t)kept;
    }
    if (kept == (1ull << 11)) { /* carry out of the significand */
        kept >>= 1;
        hexp++;
        if (hexp >= 31) return sign | 0x7C00u;
    }
    return sign | (uint16_t)(hexp << 10) | (uint16_t)(kept & 0x3FFu);
}

void synth_normal_f16(uint64_t seed, const char *name, int64_t layer, double mean, double std,
                      uint16_t *out, int64_t n) {
    uint64_t key = synth_key(seed, name, layer);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = f64_to_f16(mean + std * normal_at(key, i));
}

void synth_normal_f32(uint64_t seed, const char *name, int64_t layer, double mean, double std,
                      float *out, int64_t n) {
    uint64_t key = synth_key(seed, name, layer);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(mean + std * normal_at(key, i));
}

void synth_normal_f64(uint64_t seed, const char *name, int64_t layer, double mean, double std,
                      double *out, int64_t n) {
    uint64_t key = synth_key(seed, name, layer);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = mean + std * normal_at(key, i);
}

void synth_bytes(uint64_t seed, const char *name, int64_t layer, uint8_t *out, int64_t n) {
    uint64_t key = synth_key(seed, name, layer);
    int64_t nw = n / 8;
#pragma omp parallel for schedule(static)
    for (int64_t w = 0; w < nw; ++w) {
        uint64_t d = draw(key, (uint64_t)w);
        for (int b = 0; b < 8; ++b) out[w * 8 + b] = (uint8_t)(d >> (8 * b));
    }
    if (n % 8) {
        uint64_t d = draw(key, (uint64_t)nw);
        for (int64_t b = 0; b < n % 8; ++b) out[nw * 8 + b] = (uint8_t)(d >> (8 * b));
    }
}

/* uniform integers in [0, bound): Lemire multiply-shift of the top 32 bits */
void synth_uniform_int(uint64_t seed, const char *name, int64_t layer, uint32_t bound, int32_t *out,
                       int64_t n) {
    uint64_t key = synth_key(seed, name, layer);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t hi = draw(key, (uint64_t)i) >> 32;
        out[i] = (int32_t)((hi * (uint64_t)bound) >> 32);
    }
}

/* uniform 6-bit codes: the top 6 bits of each draw */
void synth_codes6(uint64_t seed, const char *name, int64_t layer, uint8_t *out, int64_t n) {
    uint64_t key = synth_key(seed, name, layer);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)(draw(key, (uint64_t)i) >> 58);
}

/* elements [start, start + count) of the same stream synth_normal_f16 would write */
void synth_normal_f16_range(uint64_t seed, const char *name, int64_t layer, double mean, double std,
                            uint16_t *out, int64_t start, int64_t count) {
    uint64_t key = synth_key(seed, name, layer);
#pragma omp parallel for schedule(static) if (count > 65536)
    for (int64_t i = 0; i < count; ++i) out[i] = f64_to_f16(mean + std * normal_at(key, start + i));
}
