/* e4m3_encode_exhaustive.c -- the oracle's E4M3 encoder against a nearest-
 * value search, on every binary32 value where the result is not a signed
 * zero or the saturated magnitude, and on a sample of the rest.
 *
 * The reference here is built from the OCP FP8 definition of E4M3 alone (bias
 * 7, three mantissa bits, subnormals in steps of 2^-9, S.1111.111 NaN, 448 the
 * largest finite magnitude): the 127 non-negative finite values are listed
 * code by code, and a magnitude encodes to the listed value nearest to it,
 * ties to the even code, anything above 448 saturating to 448 (satfinite) and
 * NaN keeping its sign with code 0x7F.  The oracle instead takes the binary
 * exponent with frexp and rounds the scaled mantissa; the two share nothing
 * but the format.
 *
 * Exhaustive range: binary32 exponent fields 0x6F .. 0x88, both signs (|x| in
 * [2^-16, 2^10), 26 * 2^24 values).  Below 2^-10 every value is nearer to 0
 * than to 2^-9 (2^-10 itself is the tie, which goes to the even code 0), and
 * from 464 up everything saturates; the sample covers both ends, zeros,
 * infinities, NaNs and binary32 subnormals.
 *
 * Prints one "name count bad=N" line per part; exits 1 on any mismatch.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

uint8_t oracle_e4m3_encode(float xf);

#define NTHREADS 16

static double g_val[127];          /* value of code c, c = 0 .. 0x7E */

static float from_bits(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static void build_values(void) {
    for (int c = 0; c < 127; ++c) {
        int e = c >> 3, m = c & 7;
        g_val[c] = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    }
}

/* nearest listed value, ties to the even code; satfinite; NaN keeps its sign */
static uint8_t reference_encode(float xf) {
    uint8_t s = signbit(xf) ? 0x80 : 0x00;
    if (isnan(xf)) return s | 0x7F;
    double a = fabs((double)xf);
    if (a >= g_val[126]) return s | 0x7E;
    int lo = 0, hi = 126;                      /* g_val[lo] <= a < g_val[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (g_val[mid] <= a) lo = mid; else hi = mid;
    }
    double dl = a - g_val[lo], dh = g_val[hi] - a;   /* exact: both are binary64 sums of few bits */
    int c;
    if (dl < dh) c = lo;
    else if (dh < dl) c = hi;
    else c = (lo % 2 == 0) ? lo : hi;
    return s | (uint8_t)c;
}

struct part {
    uint32_t lo, hi;                /* range of binary32 bit patterns (sign bit added inside) */
    unsigned long long n, bad;
    uint32_t first_bad;
};

static void *sweep(void *arg) {
    struct part *p = (struct part *)arg;
    p->n = p->bad = 0;
    p->first_bad = 0;
    for (uint32_t u = p->lo; u < p->hi; ++u) {
        for (uint32_t sgn = 0; sgn < 2; ++sgn) {
            float x = from_bits(u | (sgn << 31));
            ++p->n;
            if (oracle_e4m3_encode(x) != reference_encode(x)) {
                if (!p->bad) p->first_bad = u | (sgn << 31);
                ++p->bad;
            }
        }
    }
    return NULL;
}

static uint64_t splitmix(uint64_t *s) {
    uint64_t z = (*s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

int main(void) {
    build_values();
    int fail = 0;

    /* 1. every binary32 with exponent field 0x6F .. 0x88 */
    const uint32_t lo = 0x6Fu << 23, hi = 0x89u << 23;
    pthread_t th[NTHREADS];
    struct part parts[NTHREADS];
    for (int t = 0; t < NTHREADS; ++t) {
        parts[t].lo = lo + (uint32_t)((uint64_t)(hi - lo) * t / NTHREADS);
        parts[t].hi = lo + (uint32_t)((uint64_t)(hi - lo) * (t + 1) / NTHREADS);
        pthread_create(&th[t], NULL, sweep, &parts[t]);
    }
    unsigned long long n = 0, bad = 0;
    uint32_t first = 0;
    for (int t = 0; t < NTHREADS; ++t) {
        pthread_join(th[t], NULL);
        n += parts[t].n;
        if (parts[t].bad && !bad) first = parts[t].first_bad;
        bad += parts[t].bad;
    }
    printf("exhaustive %llu bad=%llu\n", n, bad);
    if (bad) {
        printf("first_mismatch 0x%08x\n", first);
        fail = 1;
    }

    /* 2. the rest: a random sample of every other binary32, and the specials */
    uint64_t s = 20261202;
    unsigned long long ns = 0, bads = 0;
    for (int i = 0; i < (1 << 24); ++i) {
        uint32_t u = (uint32_t)splitmix(&s);
        uint32_t e = (u >> 23) & 0xFFu;
        if (e >= 0x6Fu && e <= 0x88u) continue;      /* covered above */
        float x = from_bits(u);
        ++ns;
        if (oracle_e4m3_encode(x) != reference_encode(x)) ++bads;
    }
    const uint32_t specials[] = {0x00000000u, 0x80000000u, 0x00000001u, 0x80000001u, 0x007FFFFFu, 0x3A800000u,
                                 0x3A800001u, 0xBA800000u, 0x43E00000u, 0x43E7FFFFu, 0x43E80000u, 0x43E80001u,
                                 0x7F7FFFFFu, 0xFF7FFFFFu, 0x7F800000u, 0xFF800000u, 0x7FC00000u, 0xFFC00000u,
                                 0x7F800001u};
    for (size_t i = 0; i < sizeof specials / sizeof specials[0]; ++i) {
        float x = from_bits(specials[i]);
        ++ns;
        if (oracle_e4m3_encode(x) != reference_encode(x)) ++bads;
    }
    printf("sampled %llu bad=%llu\n", ns, bads);
    if (bads) fail = 1;
    return fail;
}
