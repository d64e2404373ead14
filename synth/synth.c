/*
 * synth.c - seeded synthetic BF16 weight and activation generator.
 *
 * This module only draws random numbers and rounds them to BF16.  It holds
 * none of the codec's arithmetic (no exponent split, palette, Huffman or
 * matmul), so both the oracle and the CUDA path can consume its output
 * without sharing method code.
 *
 * Recipe (all in fp64, then rounded fp64 -> fp32 (RNE) -> bf16 (RNE)):
 *   - Element i of a tensor belongs to page p = i / SYNTH_PAGE.  Each page has
 *     its own xoshiro256** state seeded by splitmix64 from (seed, stream, p),
 *     so generation is deterministic for any thread count.
 *   - Normal deviates use the Box-Muller transform (cosine branch only).
 *   - Student-t(nu=3) = Z / sqrt(chi2_3 / 3), chi2_3 the sum of three squared
 *     normals drawn from the same page stream after Z.
 *   - Outliers come from an independent stream (stream id 1): one uniform u
 *     per element; u < p1 multiplies the value by f1, else u < p1 + p2
 *     multiplies it by f2.
 *
 * The generators for splitmix64 and xoshiro256** follow their published
 * definitions (Vigna, "splitmix64.c" and "xoshiro256starstar.c").
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#define SYNTH_PAGE 4096

typedef struct { uint64_t s[4]; } xo_state;

static uint64_t splitmix64_next(uint64_t *x)
{
    uint64_t z = (*x += 0x9E3779B97F4A7C15ULL);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t rotl64(uint64_t x, int k) { return (x << k) | (x >> (64 - k)); }

static uint64_t xo_next(xo_state *st)
{
    uint64_t *s = st->s;
    uint64_t result = rotl64(s[1] * 5, 7) * 9;
    uint64_t t = s[1] << 17;
    s[2] ^= s[0];
    s[3] ^= s[1];
    s[1] ^= s[2];
    s[0] ^= s[3];
    s[2] ^= t;
    s[3] = rotl64(s[3], 45);
    return result;
}

static void xo_seed(xo_state *st, uint64_t seed, uint64_t stream, uint64_t page)
{
    uint64_t x = seed ^ (stream * 0xD1B54A32D192ED03ULL) ^ (page * 0x8CB92BA72F3D8DD7ULL);
    for (int i = 0; i < 4; i++) st->s[i] = splitmix64_next(&x);
}

/* uniform in (0, 1]: 53 random bits, never exactly zero */
static double xo_u01_open0(xo_state *st)
{
    return ((double)(xo_next(st) >> 11) + 1.0) * (1.0 / 9007199254740992.0);
}

static double xo_normal(xo_state *st)
{
    double u1 = xo_u01_open0(st);
    double u2 = xo_u01_open0(st);
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

static uint16_t f64_to_bf16(double v)
{
    float f = (float)v;
    uint32_t b;
    memcpy(&b, &f, 4);
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) return (uint16_t)((b >> 16) | 0x40u);
    b += 0x7FFFu + ((b >> 16) & 1u);
    return (uint16_t)(b >> 16);
}

enum { SYNTH_NORMAL = 0, SYNTH_STUDENT_T3 = 1 };

/*
 * Fill out[0..n) with bf16 bit patterns.
 *   kind  : SYNTH_NORMAL (scale * Z) or SYNTH_STUDENT_T3 (scale * t_3)
 *   p1,f1 : probability and multiplier of the first outlier class
 *   p2,f2 : probability and multiplier of the second outlier class
 */
void synth_fill_bf16(uint16_t *out, int64_t n, uint64_t seed, int kind, double scale,
                     double p1, double f1, double p2, double f2)
{
    int64_t n_pages = (n + SYNTH_PAGE - 1) / SYNTH_PAGE;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < n_pages; p++) {
        xo_state main_st, out_st;
        xo_seed(&main_st, seed, 0, (uint64_t)p);
        xo_seed(&out_st, seed, 1, (uint64_t)p);
        int64_t lo = p * SYNTH_PAGE, hi = lo + SYNTH_PAGE;
        if (hi > n) hi = n;
        for (int64_t i = lo; i < hi; i++) {
            double z = xo_normal(&main_st);
            double v;
            if (kind == SYNTH_STUDENT_T3) {
                double a = xo_normal(&main_st), b = xo_normal(&main_st), c = xo_normal(&main_st);
                v = z / sqrt((a * a + b * b + c * c) / 3.0);
            } else {
                v = z;
            }
            v *= scale;
            if (p1 > 0.0 || p2 > 0.0) {
                double u = (double)(xo_next(&out_st) >> 11) * (1.0 / 9007199254740992.0);
                if (u < p1) v *= f1;
                else if (u < p1 + p2) v *= f2;
            }
            out[i] = f64_to_bf16(v);
        }
    }
}

/* raw uniform 64-bit words from the page stream (used to draw random bit patterns) */
void synth_fill_u16_bits(uint16_t *out, int64_t n, uint64_t seed)
{
    int64_t n_pages = (n + SYNTH_PAGE - 1) / SYNTH_PAGE;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < n_pages; p++) {
        xo_state st;
        xo_seed(&st, seed, 2, (uint64_t)p);
        int64_t lo = p * SYNTH_PAGE, hi = lo + SYNTH_PAGE;
        if (hi > n) hi = n;
        for (int64_t i = lo; i < hi; i++) out[i] = (uint16_t)(xo_next(&st) >> 48);
    }
}
