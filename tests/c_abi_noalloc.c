/* c_abi_noalloc.c -- paged_decode_attn_noalloc through libfkv's C ABI alone
 * (plain C with the CUDA runtime: no Python, no torch), checked against the C
 * oracle.  Test infrastructure: built and run by test_zz_no_alloc.py.
 *
 * The no-allocation entry point serves callers that cannot hand the library
 * a workspace; its scratch is an array inside the library whose device
 * address the library looks up per CUDA context.  This program
 *   1. runs two different batches back to back on one stream (the second call
 *      reuses the scratch the first one left behind),
 *   2. resets the device (cudaDeviceReset ends this process's context, so
 *      the library's device code is loaded again in a new one and the array
 *      may sit elsewhere), then
 *   3. runs the first batch again in the new context,
 * and requires every output row to be within the attention tolerance of the
 * oracle (an element fails only if it is off by more than 2e-3 absolute and
 * 1e-2 relative), aborted rows zero, and the sticky device error word clear.
 * The program allocates its own inputs and outputs; only the library call
 * under test goes without a workspace. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "fkv.h"

/* the oracle (oracle/fkv_oracle.c, linked into this program) */
void oracle_kv_append_fp8(const uint16_t *k_new, const uint16_t *v_new, const int64_t *slot_mapping,
                          int32_t n_tokens, const float *k_scale, const float *v_scale, uint8_t *k_cache,
                          uint8_t *v_cache, int32_t num_pages, int32_t num_kv_heads, int32_t page_size,
                          int32_t head_dim);
void oracle_paged_decode_attn(const uint16_t *q, int32_t batch, int32_t num_q_heads, const void *k_cache,
                              const void *v_cache, int32_t kv_is_fp8, const float *k_scale, const float *v_scale,
                              int32_t num_pages, int32_t num_kv_heads, int32_t page_size, int32_t head_dim,
                              const int32_t *page_indptr, const int32_t *page_indices, int64_t nnz,
                              const int32_t *seq_lens, const uint8_t *abort_mask, double sm_scale,
                              const int32_t *rows, int32_t nrows, double *out);
void oracle_kv_calibrate_scales(const uint16_t *k, const uint16_t *v, int64_t n_tokens, int32_t num_kv_heads,
                                int32_t head_dim, float *k_scale, float *v_scale);

enum { D = 128, MAX_B = 8 };

static uint64_t g_state;

static uint64_t next_u64(void) { /* splitmix64 */
    uint64_t z = (g_state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static double uniform01(void) { return (double)(next_u64() >> 11) * (1.0 / 9007199254740992.0); }

static float normal(void) { /* Box-Muller */
    double u1 = uniform01(), u2 = uniform01();
    if (u1 < 1e-300) u1 = 1e-300;
    return (float)(sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2));
}

static uint16_t to_bf16(float f) { /* round to nearest, ties to even */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

static double bf16_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* One batch on the host: FP8 caches encoded by the oracle, pages shuffled over
 * a pool with spare pages, and the oracle's attention rows. */
struct batch {
    int32_t B, hq, hkv, S, P, nnz;
    int32_t seq[MAX_B], indptr[MAX_B + 1], *indices;
    uint8_t abort_mask[MAX_B];
    uint16_t *q;
    uint8_t *kc, *vc;
    float ks[16], vs[16];
    size_t pool;
    double *want;
};

static void make_batch(struct batch *b, uint64_t seed, int32_t B, int32_t hq, int32_t hkv, int32_t S,
                       const int32_t *seq, const uint8_t *abort_mask) {
    g_state = seed;
    b->B = B;
    b->hq = hq;
    b->hkv = hkv;
    b->S = S;
    b->indptr[0] = 0;
    for (int r = 0; r < B; ++r) {
        b->seq[r] = seq[r];
        b->abort_mask[r] = abort_mask[r];
        b->indptr[r + 1] = b->indptr[r] + (seq[r] + S - 1) / S;
    }
    b->nnz = b->indptr[B];
    b->P = b->nnz + 7;
    int32_t *perm = malloc(sizeof(int32_t) * b->P);
    for (int i = 0; i < b->P; ++i) perm[i] = i;
    for (int i = b->P - 1; i > 0; --i) {
        int j = (int)(next_u64() % (uint64_t)(i + 1));
        int32_t t = perm[i];
        perm[i] = perm[j];
        perm[j] = t;
    }
    b->indices = perm; /* the first nnz entries are the page table */
    int32_t ntok = 0;
    for (int r = 0; r < B; ++r) ntok += seq[r];
    int64_t *slots = malloc(sizeof(int64_t) * ntok);
    uint16_t *k = malloc(2u * ntok * hkv * D), *v = malloc(2u * ntok * hkv * D);
    int32_t n = 0;
    for (int r = 0; r < B; ++r)
        for (int t = 0; t < seq[r]; ++t, ++n) slots[n] = (int64_t)b->indices[b->indptr[r] + t / S] * S + t % S;
    for (int64_t i = 0; i < (int64_t)ntok * hkv * D; ++i) {
        k[i] = to_bf16(normal());
        v[i] = to_bf16(normal());
    }
    b->q = malloc(2u * B * hq * D);
    for (int i = 0; i < B * hq * D; ++i) b->q[i] = to_bf16(normal());
    b->pool = (size_t)b->P * hkv * S * D;
    b->kc = calloc(b->pool, 1);
    b->vc = calloc(b->pool, 1);
    oracle_kv_calibrate_scales(k, v, ntok, hkv, D, b->ks, b->vs);
    oracle_kv_append_fp8(k, v, slots, ntok, b->ks, b->vs, b->kc, b->vc, b->P, hkv, S, D);
    b->want = malloc(sizeof(double) * B * hq * D);
    oracle_paged_decode_attn(b->q, B, hq, b->kc, b->vc, 1, b->ks, b->vs, b->P, hkv, S, D, b->indptr, b->indices,
                             b->nnz, b->seq, b->abort_mask, 1.0 / sqrt((double)D), NULL, B * hq, b->want);
    free(slots);
    free(k);
    free(v);
}

/* Device copies of one batch's inputs and its output. */
struct dev_batch {
    void *q, *out;
    uint8_t *kc, *vc, *mask;
    float *ks, *vs;
    int32_t *indptr, *indices, *seq;
};

#define CK(x)                                                                                \
    do {                                                                                     \
        cudaError_t e_ = (x);                                                                \
        if (e_ != cudaSuccess) {                                                             \
            fprintf(stderr, "%s failed: %s\n", #x, cudaGetErrorString(e_));                 \
            return 2;                                                                        \
        }                                                                                    \
    } while (0)

static int upload(const struct batch *b, struct dev_batch *d) {
    const size_t qbytes = 2u * b->B * b->hq * D;
    CK(cudaMalloc(&d->q, qbytes));
    CK(cudaMalloc(&d->out, qbytes));
    CK(cudaMalloc((void **)&d->kc, b->pool));
    CK(cudaMalloc((void **)&d->vc, b->pool));
    CK(cudaMalloc((void **)&d->mask, b->B));
    CK(cudaMalloc((void **)&d->ks, sizeof(float) * b->hkv));
    CK(cudaMalloc((void **)&d->vs, sizeof(float) * b->hkv));
    CK(cudaMalloc((void **)&d->indptr, sizeof(int32_t) * (b->B + 1)));
    CK(cudaMalloc((void **)&d->indices, sizeof(int32_t) * b->nnz));
    CK(cudaMalloc((void **)&d->seq, sizeof(int32_t) * b->B));
    CK(cudaMemcpy(d->q, b->q, qbytes, cudaMemcpyHostToDevice));
    CK(cudaMemset(d->out, 0xFF, qbytes)); /* NaN bf16: a row the call does not write fails the check */
    CK(cudaMemcpy(d->kc, b->kc, b->pool, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d->vc, b->vc, b->pool, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d->mask, b->abort_mask, b->B, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d->ks, b->ks, sizeof(float) * b->hkv, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d->vs, b->vs, sizeof(float) * b->hkv, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d->indptr, b->indptr, sizeof(int32_t) * (b->B + 1), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d->indices, b->indices, sizeof(int32_t) * b->nnz, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d->seq, b->seq, sizeof(int32_t) * b->B, cudaMemcpyHostToDevice));
    return 0;
}

static fkv_status attend(const struct batch *b, const struct dev_batch *d) {
    return paged_decode_attn_noalloc(d->q, b->B, b->hq, d->kc, d->vc, FKV_KV_FP8_E4M3, d->ks, d->vs, b->P, b->hkv,
                                     b->S, D, d->indptr, d->indices, b->nnz, d->seq, d->mask,
                                     1.0f / sqrtf((float)D), d->out, NULL);
}

/* 0 when every element of the device output is within the tolerance of the
 * oracle and aborted rows are zero. */
static int check(const char *what, const struct batch *b, const struct dev_batch *d) {
    const int n = b->B * b->hq * D;
    uint16_t *got = malloc(2u * n);
    CK(cudaMemcpy(got, d->out, 2u * n, cudaMemcpyDeviceToHost));
    double max_err = 0.0;
    int bad = 0;
    for (int i = 0; i < n; ++i) {
        const double g = bf16_value(got[i]), o = b->want[i], e = fabs(g - o);
        if (isnan(e) || e > max_err) max_err = e;
        if (!(e <= 2e-3) && !(e <= 1e-2 * fabs(o))) ++bad;
        if (b->abort_mask[i / (b->hq * D)] && g != 0.0) ++bad;
    }
    free(got);
    if (bad) {
        fprintf(stderr, "%s: %d of %d elements outside the tolerance (max abs err %g)\n", what, bad, n, max_err);
        return 1;
    }
    printf("%s: %d elements within tolerance, max abs err %.3g\n", what, n, max_err);
    return 0;
}

static void release(struct dev_batch *d) {
    cudaFree(d->q);
    cudaFree(d->out);
    cudaFree(d->kc);
    cudaFree(d->vc);
    cudaFree(d->mask);
    cudaFree(d->ks);
    cudaFree(d->vs);
    cudaFree(d->indptr);
    cudaFree(d->indices);
    cudaFree(d->seq);
}

#define FK(x)                                                                                \
    do {                                                                                     \
        fkv_status s_ = (x);                                                                 \
        if (s_ != FKV_OK) {                                                                  \
            fprintf(stderr, "%s failed: %s\n", #x, fkv_status_string(s_));                   \
            return 3;                                                                        \
        }                                                                                    \
    } while (0)

int main(void) {
    /* A: 8 query heads per KV head, 64-token pages, one request long enough
     * to be split over many warps and merged.  B: 4 query heads per KV head,
     * 16-token pages, one aborted request. */
    const int32_t seq_a[4] = {3000, 1, 700, 129};
    const uint8_t ab_a[4] = {0, 0, 0, 0};
    const int32_t seq_b[5] = {65, 2048, 17, 400, 33};
    const uint8_t ab_b[5] = {0, 0, 1, 0, 0};
    struct batch a, b;
    make_batch(&a, 7001, 4, 16, 2, 64, seq_a, ab_a);
    make_batch(&b, 7002, 5, 16, 4, 16, seq_b, ab_b);

    struct dev_batch da, db;
    int rc;
    if ((rc = upload(&a, &da)) || (rc = upload(&b, &db))) return rc;
    /* two calls in a row on one stream: the second reuses the scratch */
    FK(attend(&a, &da));
    FK(attend(&b, &db));
    CK(cudaDeviceSynchronize());
    int fails = check("call 1 (batch A)", &a, &da) + check("call 2 (batch B)", &b, &db);
    uint32_t dev_err = 0;
    FK(fkv_device_error(&dev_err, 1));
    if (dev_err) {
        fprintf(stderr, "device error word %#x before the reset\n", dev_err);
        ++fails;
    }
    release(&da);
    release(&db);

    /* a new context: the library must look the scratch address up again */
    CK(cudaDeviceReset());
    if ((rc = upload(&a, &da))) return rc;
    FK(attend(&a, &da));
    CK(cudaDeviceSynchronize());
    fails += check("call 3 (batch A, after cudaDeviceReset)", &a, &da);
    FK(fkv_device_error(&dev_err, 1));
    if (dev_err) {
        fprintf(stderr, "device error word %#x after the reset\n", dev_err);
        ++fails;
    }
    release(&da);
    if (fails) return 1;
    printf("c abi noalloc ok\n");
    return 0;
}
