/* exhaustive_encode.c -- test helper, not part of the library or the oracle.
 *
 * An FP8 encoder written from the two formats' bit layouts (E4M3: bias 7,
 * 3 mantissa bits, S.1111.111 the only NaN, largest finite 448; E5M2: bias
 * 15, 2 mantissa bits, IEEE-style inf/NaN, largest finite 57344 -- the
 * format table of "NVIDIA Transformer Engine and FP8 mixed precision:
 * implementation guide", section "What are Transformer Engine and FP8 mixed
 * precision"), rounding to nearest with ties to even by integer arithmetic on
 * the binary32 significand and saturating at the largest finite value.
 *
 * count_mismatches() runs every one of the 2^32 binary32 bit patterns
 * through this encoder and through an encoder passed in as a function
 * pointer (the oracle's value-table search), and counts the patterns whose
 * codes differ (NaN codes compared as a class).  Threads split the range.
 */
#include <pthread.h>
#include <stdint.h>
#include <string.h>

typedef uint8_t (*encode_fn)(float, int);

enum { E4M3 = 0, E5M2 = 1 };

static int is_nan_code(uint8_t c, int fmt)
{
    uint8_t m = c & 0x7f;
    return fmt == E4M3 ? m == 0x7f : m > 0x7c;
}

/* Round the integer m / 2^sh to nearest, ties to even. */
static uint32_t rne_shift(uint32_t m, int sh)
{
    if (sh <= 0)
        return m;
    if (sh >= 32)
        return 0;
    uint32_t q = m >> sh;
    uint32_t rem = m & ((1u << sh) - 1u);
    uint32_t half = 1u << (sh - 1);
    if (rem > half || (rem == half && (q & 1u)))
        ++q;
    return q;
}

static uint8_t encode_bits(float v, int fmt)
{
    uint32_t u;
    memcpy(&u, &v, 4);
    const uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
    const uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u)
        return 0xff;                                   /* NaN (a NaN code of both formats) */
    const int mbits = fmt == E4M3 ? 3 : 2;
    const int bias = fmt == E4M3 ? 7 : 15;
    const uint32_t top = fmt == E4M3 ? 0x7eu : 0x7bu; /* largest finite magnitude code */
    const int e32 = (int)(a >> 23);
    if (e32 == 0)
        return sign;          /* zero or binary32 subnormal: far below half the FP8 minimum */
    if (e32 == 255)
        return (uint8_t)(sign | top);                  /* infinity saturates */
    const uint32_t sig = (a & 0x7fffffu) | 0x800000u;  /* 24-bit significand */
    const int e = e32 - 127;                           /* value = sig * 2^(e - 23) */
    uint32_t code;
    if (e + bias >= 1) {
        /* normal range of the target: keep mbits fraction bits; a carry out
         * of the fraction moves into the exponent field by itself */
        const uint32_t frac = rne_shift(sig, 23 - mbits);            /* 1.f * 2^mbits */
        const int64_t c = ((int64_t)(e + bias) << mbits) + (int64_t)frac - (1 << mbits);
        code = c > (int64_t)top ? top + 1u : (uint32_t)c;
    } else {
        /* subnormal range: multiples of 2^(1 - bias - mbits) */
        const int sh = 23 - mbits + (1 - bias - e);
        code = rne_shift(sig, sh);
    }
    if (code > top)
        code = top;
    return (uint8_t)(sign | code);
}

struct job {
    encode_fn other;
    int fmt;
    uint64_t lo, hi;
    int64_t bad;
    uint32_t first_bad;
};

static void *run(void *p)
{
    struct job *j = (struct job *)p;
    for (uint64_t i = j->lo; i < j->hi; ++i) {
        const uint32_t u = (uint32_t)i;
        float v;
        memcpy(&v, &u, 4);
        const uint8_t x = encode_bits(v, j->fmt), y = j->other(v, j->fmt);
        if (x == y || (is_nan_code(x, j->fmt) && is_nan_code(y, j->fmt)))
            continue;
        if (j->bad == 0)
            j->first_bad = u;
        ++j->bad;
    }
    return NULL;
}

/* Number of the 2^32 patterns whose codes differ; *first_bad = the lowest
 * such pattern of the first thread that found one. */
int64_t count_mismatches(encode_fn other, int fmt, int nthreads, uint32_t *first_bad)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 64)
        nthreads = 64;
    struct job jobs[64];
    pthread_t th[64];
    const uint64_t total = 1ull << 32, per = (total + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].other = other;
        jobs[t].fmt = fmt;
        jobs[t].lo = per * t;
        jobs[t].hi = per * (t + 1) < total ? per * (t + 1) : total;
        jobs[t].bad = 0;
        jobs[t].first_bad = 0;
        pthread_create(&th[t], NULL, run, &jobs[t]);
    }
    int64_t bad = 0;
    *first_bad = 0;
    for (int t = 0; t < nthreads; ++t) {
        pthread_join(th[t], NULL);
        if (jobs[t].bad && bad == 0)
            *first_bad = jobs[t].first_bad;
        bad += jobs[t].bad;
    }
    return bad;
}

/* The bit-level encoder alone, for spot checks from the test. */
uint8_t encode_bits_one(float v, int fmt) { return encode_bits(v, fmt); }
