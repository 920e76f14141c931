/*
 * fkv_oracle.c -- CPU oracle for FP8 paged-KV decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * reference that the CUDA library is checked against.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the
 * library itself never calls it and has no CPU fallback.  It shares no code,
 * header, table or constant with the CUDA sources.
 *
 * Everything is scalar C in fp64, in the order the definitions state it, with
 * no blocking, fusion or reordering.
 *
 * Sources for what is computed (page title, then section):
 *   [CF]  "Cloudflare Workers AI Optimizes Large Model Serving with KV Cache
 *         Quantization, Weight Compression, and Integrity Checks" -- the
 *         extracted text of Cloudflare's post "Smaller, faster, safer": the KV
 *         cache is stored as 8-bit floating point (FP8, e4m3) instead of BF16;
 *         the FP8 attention kernel converts values as it reads them; every
 *         physical page carries a tag that changes when the page is
 *         reallocated, the server records the (page, tag) pairs each request
 *         expects, mappings are checked before decode reads the cache and a
 *         mismatching request is aborted.
 *   [GN]  "Kimi and GLM Reasoning Slimming: Hands-On Test", section
 *         "Giving Every Physical Cache Page a 'Generation Number'": the
 *         per-request loop over expected pages, comparing the allocator's
 *         current tag with the expected tag and aborting on mismatch
 *         (fail closed).
 *   [OFP8] The OCP "8-bit Floating Point Specification (OFP8)", E4M3 format:
 *         1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent
 *         field 0 is subnormal; S.1111.111 is NaN; no infinities; the largest
 *         finite magnitude is 1.75 * 2^8 = 448.  The pages name the format only.
 *
 * Readings taken where the pages are silent (each one is also listed in the
 * design notes):
 *   - quantize: code = e4m3_rne_satfinite( fl32( fl32(x_bf16) / scale ) ),
 *     an IEEE round-to-nearest fp32 division followed by one round-to-nearest-
 *     even to E4M3; magnitudes above 448 (and +-Inf) saturate to +-448; NaN
 *     stays NaN (sign kept); -0 encodes as 0x80.
 *   - scale granularity: one fp32 scale per KV head for K and one for V.
 *   - layout: K and V pools are [num_pages][num_kv_heads][page_size][head_dim].
 *   - page table: CSR (indptr[B+1], indices[nnz]); token t of request r lives
 *     in page indices[indptr[r] + t / S] at offset t % S.
 *   - GQA: query head i reads KV head i / G, G = Hq / Hkv.
 *   - tag check: a request aborts if any listed page id is outside [0, P),
 *     any live tag differs from the expected tag, or its CSR row is malformed.
 *   - attention: aborted, empty, or malformed requests (a CSR row outside
 *     [0, nnz], seq_len <= 0, seq_len > pages * S, or a page id read outside
 *     [0, P)) give an all-zero output row (fail closed).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Scalar formats                                                            */
/* ------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double oracle_bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* E4M3 decode, [OFP8]: subnormal m * 2^-9, normal (1 + m/8) * 2^(e-7). */
double oracle_e4m3_decode(uint8_t code)
{
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return s ? -NAN : NAN;
    if (e == 0)
        v = (double)m * ldexp(1.0, -9);
    else
        v = (1.0 + (double)m / 8.0) * ldexp(1.0, e - 7);
    return s ? -v : v;
}

/* Round-half-to-even of a double that is exactly representable. */
static double rne(double y)
{
    double f = floor(y);
    double d = y - f;
    if (d > 0.5)
        return f + 1.0;
    if (d < 0.5)
        return f;
    /* exact tie: pick the even neighbour */
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* E4M3 encode with round-to-nearest-even and saturation to +-448, [OFP8]. */
uint8_t oracle_e4m3_encode(float xf)
{
    double x = (double)xf;
    uint8_t s = signbit(x) ? 0x80 : 0x00;
    double a;
    int e2;
    if (isnan(x))
        return s | 0x7F;
    a = fabs(x);
    if (a > 448.0)               /* satfinite: the largest finite magnitude */
        return s | 0x7E;
    if (a < ldexp(1.0, -6)) {    /* subnormal range: steps of 2^-9 */
        double q = rne(a * 512.0);   /* 0 .. 8; 8 is the smallest normal, code 0x08 */
        return s | (uint8_t)q;
    }
    /* normal: a = f * 2^e2 with f in [0.5, 1), so floor(log2 a) = e2 - 1 */
    (void)frexp(a, &e2);
    {
        int e = e2 - 1;
        double m = rne((ldexp(a, -e) - 1.0) * 8.0);   /* exact in fp64 */
        if (m == 8.0) {
            m = 0.0;
            e += 1;
        }
        return s | (uint8_t)(((e + 7) << 3) | (int)m);
    }
}

/* fl32(x / scale) with a single IEEE round-to-nearest: the fp64 quotient of two
 * binary32 operands, rounded once more to binary32, is the correctly rounded
 * binary32 quotient (53 >= 2*24 + 2, so the double rounding is innocuous). */
float oracle_div_rn_f32(float x, float scale)
{
    return (float)((double)x / (double)scale);
}

/* ------------------------------------------------------------------------ */
/* Append: quantize each new token's K/V and write it into its page slot.    */
/* [CF]: K/V stored as FP8 e4m3 instead of BF16, one fp32 scale per KV head. */
/* ------------------------------------------------------------------------ */
void oracle_kv_append_fp8(const uint16_t *k_new, const uint16_t *v_new,
                          const int64_t *slot_mapping, int32_t n_tokens,
                          const float *k_scale, const float *v_scale,
                          uint8_t *k_cache, uint8_t *v_cache,
                          int32_t num_pages, int32_t num_kv_heads,
                          int32_t page_size, int32_t head_dim)
{
    for (int32_t n = 0; n < n_tokens; ++n) {
        int64_t slot = slot_mapping[n];
        int64_t page, off;
        if (slot < 0)
            continue;                       /* padding token: nothing to write */
        page = slot / page_size;
        off = slot % page_size;
        if (page >= num_pages)
            continue;                       /* outside the pool: not written */
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            for (int32_t d = 0; d < head_dim; ++d) {
                int64_t src = ((int64_t)n * num_kv_heads + h) * head_dim + d;
                int64_t dst = (((page * num_kv_heads) + h) * page_size + off) * head_dim + d;
                float kx = (float)oracle_bf16_to_double(k_new[src]);
                float vx = (float)oracle_bf16_to_double(v_new[src]);
                k_cache[dst] = oracle_e4m3_encode(oracle_div_rn_f32(kx, k_scale[h]));
                v_cache[dst] = oracle_e4m3_encode(oracle_div_rn_f32(vx, v_scale[h]));
            }
        }
    }
}

/* BF16 cache: the same placement, the value stored unchanged. */
void oracle_kv_append_bf16(const uint16_t *k_new, const uint16_t *v_new,
                           const int64_t *slot_mapping, int32_t n_tokens,
                           uint16_t *k_cache, uint16_t *v_cache,
                           int32_t num_pages, int32_t num_kv_heads,
                           int32_t page_size, int32_t head_dim)
{
    for (int32_t n = 0; n < n_tokens; ++n) {
        int64_t slot = slot_mapping[n];
        int64_t page, off;
        if (slot < 0)
            continue;
        page = slot / page_size;
        off = slot % page_size;
        if (page >= num_pages)
            continue;
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            for (int32_t d = 0; d < head_dim; ++d) {
                int64_t src = ((int64_t)n * num_kv_heads + h) * head_dim + d;
                int64_t dst = (((page * num_kv_heads) + h) * page_size + off) * head_dim + d;
                k_cache[dst] = k_new[src];
                v_cache[dst] = v_new[src];
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Integrity check, [GN] and [CF]: for each page a request expects, compare   */
/* the live tag with the expected one; any mismatch aborts the request.      */
/* ------------------------------------------------------------------------ */
void oracle_kv_page_tag_check(const uint32_t *page_tags, int32_t num_pages,
                              const int32_t *page_indptr, const int32_t *page_indices,
                              const uint32_t *expected_tags, int32_t batch, int64_t nnz,
                              uint8_t *abort_mask)
{
    for (int32_t r = 0; r < batch; ++r) {
        int64_t begin = page_indptr[r];
        int64_t end = page_indptr[r + 1];
        uint8_t abort_r = 0;
        if (begin < 0 || end < begin || end > nnz) {
            abort_mask[r] = 1;               /* malformed row: fail closed */
            continue;
        }
        for (int64_t j = begin; j < end; ++j) {
            int32_t page = page_indices[j];
            if (page < 0 || page >= num_pages) {
                abort_r = 1;                 /* no such page: fail closed */
                break;
            }
            if (page_tags[page] != expected_tags[j]) {
                abort_r = 1;                 /* stale or mismatched page */
                break;
            }
        }
        abort_mask[r] = abort_r;
    }
}

/* ------------------------------------------------------------------------ */
/* Attention                                                                 */
/* ------------------------------------------------------------------------ */

/* Dense softmax(q k^T * sm_scale) v for one query row over T keys, fp64.
 * k, v are [T][D] row-major.  T == 0 gives zeros. */
void oracle_dense_attn(const double *q, const double *k, const double *v,
                       int32_t T, int32_t D, double sm_scale, double *out)
{
    double *s;
    double mx = -INFINITY, l = 0.0;
    for (int32_t d = 0; d < D; ++d)
        out[d] = 0.0;
    if (T <= 0)
        return;
    s = (double *)malloc(sizeof(double) * (size_t)T);
    for (int32_t t = 0; t < T; ++t) {
        double acc = 0.0;
        for (int32_t d = 0; d < D; ++d)
            acc += q[d] * k[(int64_t)t * D + d];
        s[t] = acc * sm_scale;
        if (s[t] > mx)
            mx = s[t];
    }
    for (int32_t t = 0; t < T; ++t) {
        s[t] = exp(s[t] - mx);
        l += s[t];
    }
    for (int32_t t = 0; t < T; ++t)
        for (int32_t d = 0; d < D; ++d)
            out[d] += s[t] * v[(int64_t)t * D + d];
    for (int32_t d = 0; d < D; ++d)
        out[d] /= l;
    free(s);
}

/* Dequantized cache element in fp64: code value times the head's scale for
 * FP8, the bf16 value itself for BF16. */
static double cache_value(const void *cache, int kv_is_fp8, int64_t idx, const float *scale, int32_t h)
{
    if (kv_is_fp8)
        return oracle_e4m3_decode(((const uint8_t *)cache)[idx]) * (double)scale[h];
    return oracle_bf16_to_double(((const uint16_t *)cache)[idx]);
}

/* Paged decode attention: for every selected (request, query head) row,
 * gather the request's tokens through its page table, dequantize them and
 * take the dense fp64 attention.  `rows` lists flat indices r*Hq + i; NULL
 * means all B*Hq rows in order.  out is [nrows][D]. */
void oracle_paged_decode_attn(const uint16_t *q, int32_t batch, int32_t num_q_heads,
                              const void *k_cache, const void *v_cache, int32_t kv_is_fp8,
                              const float *k_scale, const float *v_scale,
                              int32_t num_pages, int32_t num_kv_heads,
                              int32_t page_size, int32_t head_dim,
                              const int32_t *page_indptr, const int32_t *page_indices, int64_t nnz,
                              const int32_t *seq_lens, const uint8_t *abort_mask,
                              double sm_scale, const int32_t *rows, int32_t nrows,
                              double *out)
{
    int32_t G = num_q_heads / num_kv_heads;
    int32_t D = head_dim;
    int32_t total = rows ? nrows : batch * num_q_heads;
    for (int32_t x = 0; x < total; ++x) {
        int32_t flat = rows ? rows[x] : x;
        int32_t r = flat / num_q_heads;
        int32_t i = flat % num_q_heads;
        int32_t h = i / G;
        int32_t T = seq_lens[r];
        int64_t npages = (int64_t)page_indptr[r + 1] - page_indptr[r];
        double *o = out + (int64_t)x * D;
        double *qd, *kd, *vd;
        int ok = 1;
        for (int32_t d = 0; d < D; ++d)
            o[d] = 0.0;
        if (abort_mask && abort_mask[r])
            continue;                                   /* aborted: zero row */
        if (page_indptr[r] < 0 || npages < 0 || page_indptr[r + 1] > nnz)
            continue;                                   /* malformed CSR row */
        if (T <= 0 || (int64_t)T > npages * page_size)
            continue;                                   /* empty, or more tokens than pages */
        for (int32_t t = 0; t < T && ok; t += page_size) {
            int32_t page = page_indices[page_indptr[r] + t / page_size];
            if (page < 0 || page >= num_pages)
                ok = 0;
        }
        if (!ok)
            continue;                                   /* bad page id: zero row */
        qd = (double *)malloc(sizeof(double) * (size_t)D);
        kd = (double *)malloc(sizeof(double) * (size_t)T * D);
        vd = (double *)malloc(sizeof(double) * (size_t)T * D);
        for (int32_t d = 0; d < D; ++d)
            qd[d] = oracle_bf16_to_double(q[((int64_t)r * num_q_heads + i) * D + d]);
        for (int32_t t = 0; t < T; ++t) {
            int64_t page = page_indices[page_indptr[r] + t / page_size];
            int64_t off = t % page_size;
            int64_t base = ((page * num_kv_heads + h) * page_size + off) * D;
            for (int32_t d = 0; d < D; ++d) {
                kd[(int64_t)t * D + d] = cache_value(k_cache, kv_is_fp8, base + d, k_scale, h);
                vd[(int64_t)t * D + d] = cache_value(v_cache, kv_is_fp8, base + d, v_scale, h);
            }
        }
        oracle_dense_attn(qd, kd, vd, T, D, sm_scale, o);
        free(qd);
        free(kd);
        free(vd);
    }
}

/* ------------------------------------------------------------------------ */
/* Reallocation: hand pages to new owners.  [GN], [CF]: a page's tag changes */
/* each time the page is reallocated, so holders of the old (page, tag) pair */
/* fail the check.  Optional scrub zeroes the page's K and V bytes first.    */
/* ------------------------------------------------------------------------ */
void oracle_kv_page_realloc(uint32_t *page_tags, int32_t num_pages,
                            const int32_t *pages, int32_t n, uint32_t *new_tags,
                            uint8_t *k_cache, uint8_t *v_cache,
                            int32_t num_kv_heads, int32_t page_size, int32_t head_dim,
                            int32_t elem_bytes)
{
    int64_t page_bytes = (int64_t)num_kv_heads * page_size * head_dim * elem_bytes;
    for (int32_t j = 0; j < n; ++j) {
        int32_t p = pages[j];
        if (p < 0 || p >= num_pages) {
            new_tags[j] = 0;               /* not a page of this pool: nothing changes */
            continue;
        }
        page_tags[p] = page_tags[p] + 1u;  /* 32-bit wrap counts as a change */
        new_tags[j] = page_tags[p];
        if (k_cache && v_cache) {
            memset(k_cache + (int64_t)p * page_bytes, 0, (size_t)page_bytes);
            memset(v_cache + (int64_t)p * page_bytes, 0, (size_t)page_bytes);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Scale calibration for a bulk (prefill) write: per KV head, the largest    */
/* |value| over all tokens, scale = fl32(amax / 448) (448 = the largest      */
/* finite e4m3 magnitude), 1 when the head is all zeros.                     */
/* ------------------------------------------------------------------------ */
void oracle_kv_calibrate_scales(const uint16_t *k, const uint16_t *v, int64_t n_tokens,
                                int32_t num_kv_heads, int32_t head_dim,
                                float *k_scale, float *v_scale)
{
    for (int32_t h = 0; h < num_kv_heads; ++h) {
        double ka = 0.0, va = 0.0;
        for (int64_t n = 0; n < n_tokens; ++n) {
            for (int32_t d = 0; d < head_dim; ++d) {
                int64_t i = (n * num_kv_heads + h) * head_dim + d;
                double a = fabs(oracle_bf16_to_double(k[i]));
                double b = fabs(oracle_bf16_to_double(v[i]));
                if (a > ka) ka = a;
                if (b > va) va = b;
            }
        }
        k_scale[h] = ka > 0.0 ? (float)(ka / 448.0) : 1.0f;
        v_scale[h] = va > 0.0 ? (float)(va / 448.0) : 1.0f;
    }
}
