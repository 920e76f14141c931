/* recip_division_check.c -- host-side proof of the fp32 division used on the
 * fast path of kv_append_fp8 (test infrastructure, run by
 * test_append_division.py; not part of the library).
 *
 * The kernel divides a bf16 value a by the per-head scale b as
 *     y = RN(1/b),  q0 = RN(|a|*y),  r = RN(|a| - b*q0),  q = RN(q0 + r*y)
 * (the two last steps fused multiply-adds), then gives q the sign of a; it
 * does so only for 2^-30 <= b <= 2^30 and |a| <= 2^64.  This program checks
 * the same sequence in IEEE single precision on the host against the
 * correctly rounded quotient RN(a/b), computed as (float)((double)a/(double)b)
 * (a single rounding: 53 >= 2*24 + 2 bits makes the double rounding
 * innocuous), and the reciprocal likewise.
 *
 *  1. exhaustive: every bf16 significand of a (128) times every fp32
 *     significand of b (2^23), both in [1, 2);
 *  2. random pairs over the whole admitted exponent range, with signs;
 *  3. |a| < 2^-64 (zero and subnormals included): the result is finite,
 *     below 2^-33 in magnitude and carries a's sign (its e4m3 code is then
 *     the signed zero, as for the exact quotient).
 * Exit status 0 iff every case agrees. */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

static float rn_recip(float b) { return (float)(1.0 / (double)b); }
static float rn_div(float a, float b) { return (float)((double)a / (double)b); }

/* The kernel's sequence. */
static float recip_div(float a, float b, float y) {
    float m = fabsf(a);
    float q0 = m * y;
    float r = fmaf(-q0, b, m);
    float q = fmaf(r, y, q0);
    return from_bits(to_bits(q) | (to_bits(a) & 0x80000000u));
}

static uint64_t splitmix(uint64_t *s) {
    uint64_t z = (*s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

#define NTHREADS 8
struct part { uint32_t lo, hi; unsigned long long bad; };

static void *exhaustive(void *arg) {
    struct part *p = (struct part *)arg;
    for (uint32_t mb = p->lo; mb < p->hi; ++mb) {
        float b = from_bits(0x3F800000u | mb);
        float y = rn_recip(b);
        for (uint32_t ma = 0; ma < 128; ++ma) {
            float a = from_bits(0x3F800000u | (ma << 16));
            if (recip_div(a, b, y) != rn_div(a, b)) ++p->bad;
        }
    }
    return NULL;
}

int main(void) {
    /* 1. exhaustive over significands */
    pthread_t th[NTHREADS];
    struct part parts[NTHREADS];
    const uint32_t n = 1u << 23;
    for (int t = 0; t < NTHREADS; ++t) {
        parts[t].lo = (uint32_t)((uint64_t)n * t / NTHREADS);
        parts[t].hi = (uint32_t)((uint64_t)n * (t + 1) / NTHREADS);
        parts[t].bad = 0;
        pthread_create(&th[t], NULL, exhaustive, &parts[t]);
    }
    unsigned long long bad_exhaustive = 0;
    for (int t = 0; t < NTHREADS; ++t) {
        pthread_join(th[t], NULL);
        bad_exhaustive += parts[t].bad;
    }

    /* 2. random pairs across the admitted exponent range (and its ends) */
    uint64_t s = 12345;
    unsigned long long bad_scaled = 0, scaled = 0;
    for (int i = 0; i < (1 << 24); ++i) {
        uint64_t u = splitmix(&s);
        int ea = (int)(u % 129) - 64;                      /* |a| in [2^-64, 2^65) */
        int eb = (int)((u >> 8) % 61) - 30;                /* b in [2^-30, 2^31) */
        uint32_t abits = ((uint32_t)(ea + 127) << 23) | ((uint32_t)(u >> 16) & 0x007F0000u) |
                         ((uint32_t)(u >> 40) & 1u) << 31;
        uint32_t bbits = ((uint32_t)(eb + 127) << 23) | ((uint32_t)(u >> 41) & 0x007FFFFFu);
        float a = from_bits(abits), b = from_bits(bbits);
        if (fabsf(a) > 0x1p64f || b > 0x1p30f) continue;  /* outside the fast path */
        ++scaled;
        if (recip_div(a, b, rn_recip(b)) != rn_div(a, b)) ++bad_scaled;
    }
    const float ends_a[] = {0x1p-64f, 0x1p64f, 0x1.FEp63f, 0x1.02p-64f};
    const float ends_b[] = {0x1p-30f, 0x1p30f, 0x1.FFFFFEp29f, 0x1.000002p-30f};
    for (int i = 0; i < 4; ++i)
        for (int j = 0; j < 4; ++j)
            for (int sg = 0; sg < 2; ++sg) {
                float a = sg ? -ends_a[i] : ends_a[i], b = ends_b[j];
                ++scaled;
                if (recip_div(a, b, rn_recip(b)) != rn_div(a, b)) ++bad_scaled;
            }

    /* 3. |a| below 2^-64: finite, tiny, signed like a */
    unsigned long long bad_tiny = 0, tiny = 0;
    for (int i = 0; i < (1 << 20); ++i) {
        uint64_t u = splitmix(&s);
        uint32_t e = (uint32_t)(u % 64);                   /* biased exponent 0..63: |a| < 2^-64 */
        uint32_t abits = (e << 23) | ((uint32_t)(u >> 16) & 0x007F0000u) | ((uint32_t)(u >> 40) & 1u) << 31;
        int eb = (int)((u >> 8) % 61) - 30;
        float a = from_bits(abits), b = from_bits(((uint32_t)(eb + 127) << 23) | ((uint32_t)(u >> 41) & 0x7FFFFFu));
        if (b > 0x1p30f) continue;
        ++tiny;
        float q = recip_div(a, b, rn_recip(b));
        if (!isfinite(q) || fabsf(q) >= 0x1p-33f || signbit(q) != signbit(a)) ++bad_tiny;
    }
    ++tiny;                                               /* -0 stays -0 */
    if (to_bits(recip_div(-0.0f, 0.25f, rn_recip(0.25f))) != 0x80000000u) ++bad_tiny;

    printf("exhaustive_pairs=%llu bad=%llu\n", (unsigned long long)n * 128ull, bad_exhaustive);
    printf("scaled_pairs=%llu bad=%llu\n", scaled, bad_scaled);
    printf("tiny_pairs=%llu bad=%llu\n", tiny, bad_tiny);
    return (bad_exhaustive || bad_scaled || bad_tiny) ? 1 : 0;
}
