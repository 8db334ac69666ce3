/*
 * inputgen.c — seeded synthetic inputs shared by the tests, the benchmark and
 * the oracle's callers.  It holds none of the weighted-sum or scaled-SiLU
 * arithmetic: it only draws numbers and rounds them to the storage type.
 *
 * Generator.  SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) used as a counter-based
 * generator: the k-th 64-bit word of stream s under seed `seed` is
 *
 *     key   = mix64(seed * GAMMA + s + 1)
 *     z_k   = mix64(key + (k + 1) * GAMMA)            (mod 2^64)
 *
 * with GAMMA = 0x9E3779B97F4A7C15 and mix64 the published SplitMix64
 * finaliser (xor-shift 30 / multiply / xor-shift 27 / multiply / xor-shift 31).
 * A word becomes a uniform double in (0,1) as ((z >> 11) + 0.5) * 2^-53.
 *
 * Distributions.
 *   uniform(a, b):  v_k = a + (b - a) * u_k
 *   normal(m, sd):  Box-Muller (G. Box, M. Muller, Ann. Math. Stat. 1958) on
 *                   the pair j = k / 2:  r = sqrt(-2 ln u_{2j}),
 *                   t = 2 pi u_{2j+1};  v_{2j} = m + sd r cos t,
 *                   v_{2j+1} = m + sd r sin t.
 * Every element depends only on (seed, stream, k), so any sub-range (a row,
 * a sample of rows) can be regenerated without the rest, and the result does
 * not depend on the number of threads.
 *
 * Storage.  The double v_k is rounded once, to nearest with ties to even, to
 * the storage type: binary32, binary16 or bfloat16.  The rounding below works
 * on the integer fields of the double; it is written independently of the
 * oracle's own conversions so that the two can check each other.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define IG_F32 0
#define IG_F16 1
#define IG_BF16 2

#define IG_NORMAL 0
#define IG_UNIFORM 1

static const uint64_t GAMMA = 0x9E3779B97F4A7C15ull;

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline double u01(uint64_t key, uint64_t k) {
    uint64_t z = mix64(key + (k + 1) * GAMMA);
    return ((double)(z >> 11) + 0.5) * 0x1.0p-53;
}

/* Round a double to a binary format with `ebits` exponent bits and `mbits`
 * stored mantissa bits, ties to even; returns the bit pattern. */
static uint32_t round_to_format(double v, int ebits, int mbits) {
    uint64_t b;
    memcpy(&b, &v, 8);
    const uint32_t sign = (uint32_t)(b >> 63) << (ebits + mbits);
    const int bias = (1 << (ebits - 1)) - 1;
    const uint32_t exp_all_ones = (uint32_t)((1 << ebits) - 1);
    const int E = (int)((b >> 52) & 0x7FF);
    const uint64_t M = b & 0xFFFFFFFFFFFFFull;
    if (E == 0x7FF) { /* inf or NaN */
        if (M) return sign | (exp_all_ones << mbits) | (1u << (mbits - 1));
        return sign | (exp_all_ones << mbits);
    }
    if (E == 0 && M == 0) return sign;
    /* value = sig * 2^(e - 52) with sig the 53-bit significand */
    uint64_t sig = (E == 0) ? M : (M | (1ull << 52));
    int e = (E == 0) ? -1022 : E - 1023;
    if (E == 0) { /* normalise a double subnormal */
        while (!(sig & (1ull << 52))) { sig <<= 1; e--; }
    }
    const int emin = 1 - bias;
    /* number of low significand bits to drop */
    int drop = 52 - mbits;
    if (e < emin) drop += emin - e; /* target subnormal: fewer bits survive */
    uint64_t kept;
    if (drop >= 64) {
        kept = 0; /* far below the smallest subnormal: rounds to zero */
    } else {
        kept = sig >> drop;
        const uint64_t rem = sig & ((1ull << drop) - 1);
        const uint64_t half = 1ull << (drop - 1);
        if (rem > half || (rem == half && (kept & 1))) kept++;
    }
    /* re-assemble: `kept` is the significand in units of the target ulp */
    int te = (e < emin) ? emin : e; /* exponent of the target quantum scale */
    if (e < emin) {
        /* subnormal range: kept may have carried into the normal range,
         * which the field encoding below handles naturally */
        if (kept >= (1ull << mbits)) return sign | (1u << mbits) | (uint32_t)(kept - (1ull << mbits));
        return sign | (uint32_t)kept;
    }
    if (kept >= (2ull << mbits)) { kept >>= 1; te++; } /* carry to next binade */
    if (te > bias) return sign | (exp_all_ones << mbits); /* overflow -> inf */
    return sign | ((uint32_t)(te + bias) << mbits) | (uint32_t)(kept & ((1ull << mbits) - 1));
}

static inline void store(void* out, int64_t i, int dtype, double v) {
    if (dtype == IG_F32) {
        ((float*)out)[i] = (float)v;
    } else if (dtype == IG_F16) {
        ((uint16_t*)out)[i] = (uint16_t)round_to_format(v, 5, 10);
    } else {
        ((uint16_t*)out)[i] = (uint16_t)round_to_format(v, 8, 7);
    }
}

static inline double draw(uint64_t key, int64_t k, int dist, double a, double b) {
    if (dist == IG_UNIFORM) return a + (b - a) * u01(key, (uint64_t)k);
    const int64_t j = k >> 1;
    const double r = sqrt(-2.0 * log(u01(key, (uint64_t)(2 * j))));
    const double t = 6.283185307179586476925286766559 * u01(key, (uint64_t)(2 * j + 1));
    return a + b * r * ((k & 1) ? sin(t) : cos(t));
}

/* Fill out[0..n) with elements first .. first+n-1 of (seed, stream).
 * dtype: 0 binary32, 1 binary16, 2 bfloat16.  dist: 0 normal(a, sd=b),
 * 1 uniform(a, b).  Returns 0, or -1 on a bad argument. */
int ig_fill(void* out, int64_t n, int dtype, int dist, double a, double b,
            uint64_t seed, uint64_t stream, int64_t first) {
    if (!out || n < 0 || first < 0 || dtype < 0 || dtype > 2 || dist < 0 || dist > 1) return -1;
    const uint64_t key = mix64(seed * GAMMA + stream + 1);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) store(out, i, dtype, draw(key, first + i, dist, a, b));
    return 0;
}

/* Fill a 2-D [rows, cols] block with row stride ld (elements) from the
 * logical row-major stream of a [*, cols] tensor starting at row first_row.
 * Padding between cols and ld is left untouched. */
int ig_fill_rows(void* out, int64_t rows, int64_t cols, int64_t ld, int dtype, int dist,
                 double a, double b, uint64_t seed, uint64_t stream, int64_t first_row) {
    if (!out || rows < 0 || cols < 0 || ld < cols || first_row < 0 || dtype < 0 || dtype > 2 ||
        dist < 0 || dist > 1)
        return -1;
    const uint64_t key = mix64(seed * GAMMA + stream + 1);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c++)
            store(out, r * ld + c, dtype, draw(key, (first_row + r) * cols + c, dist, a, b));
    return 0;
}

/* The raw 64-bit word z_k (for checking the generator against its
 * published definition). */
uint64_t ig_word(uint64_t seed, uint64_t stream, uint64_t k) {
    return mix64(mix64(seed * GAMMA + stream + 1) + (k + 1) * GAMMA);
}

/* The k-th output (k = 0, 1, ...) of the sequential SplitMix64 generator
 * whose state starts at state0: mix64(state0 + (k + 1) * GAMMA). */
uint64_t ig_splitmix64(uint64_t state0, uint64_t k) { return mix64(state0 + (k + 1) * GAMMA); }

/* Rounding helpers exposed for cross-checks: double -> binary16 / bfloat16 bits. */
uint32_t ig_round_f16(double v) { return round_to_format(v, 5, 10); }
uint32_t ig_round_bf16(double v) { return round_to_format(v, 8, 7); }
