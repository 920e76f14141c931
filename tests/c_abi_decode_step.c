/* c_abi_decode_step.c -- one decode step through libfkv's C ABI alone (plain
 * C with the CUDA runtime: no Python, no torch), checked against the C
 * oracle.  Test infrastructure: built and run by test_gpu_c_abi.py.
 *
 * A small batch (3 requests, 8 query / 2 KV heads, 16-token pages scattered
 * over a pool with spare pages) is drawn from a fixed-seed generator.  On the
 * device: per-head scales of the context (kv_calibrate_scales), the whole
 * context written as e4m3 (kv_append_fp8), the integrity check with one stale
 * tag (kv_page_tag_check), then attention (paged_decode_attn); and the same
 * append and check once more as one launch (kv_append_fp8_tag_check) into a
 * second pair of pools.  The scales, every pool byte of both pairs and both
 * abort masks must equal the oracle's bit for bit; the
 * attention rows must be within the tolerance (an element fails only if it is
 * off by more than 2e-3 absolute and 1e-2 relative), the aborted row zero. */
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
void oracle_kv_page_tag_check(const uint32_t *page_tags, int32_t num_pages, const int32_t *page_indptr,
                              const int32_t *page_indices, const uint32_t *expected_tags, int32_t batch,
                              int64_t nnz, uint8_t *abort_mask);
void oracle_paged_decode_attn(const uint16_t *q, int32_t batch, int32_t num_q_heads, const void *k_cache,
                              const void *v_cache, int32_t kv_is_fp8, const float *k_scale, const float *v_scale,
                              int32_t num_pages, int32_t num_kv_heads, int32_t page_size, int32_t head_dim,
                              const int32_t *page_indptr, const int32_t *page_indices, int64_t nnz,
                              const int32_t *seq_lens, const uint8_t *abort_mask, double sm_scale,
                              const int32_t *rows, int32_t nrows, double *out);
void oracle_kv_calibrate_scales(const uint16_t *k, const uint16_t *v, int64_t n_tokens, int32_t num_kv_heads,
                                int32_t head_dim, float *k_scale, float *v_scale);

static uint64_t g_state = 20261202u;

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

#define CK(x)                                                                                \
    do {                                                                                     \
        cudaError_t e_ = (x);                                                                \
        if (e_ != cudaSuccess) {                                                             \
            fprintf(stderr, "%s failed: %s\n", #x, cudaGetErrorString(e_));                 \
            return 2;                                                                        \
        }                                                                                    \
    } while (0)
#define FK(x)                                                                                \
    do {                                                                                     \
        fkv_status s_ = (x);                                                                 \
        if (s_ != FKV_OK) {                                                                  \
            fprintf(stderr, "%s failed: %s\n", #x, fkv_status_string(s_));                   \
            return 3;                                                                        \
        }                                                                                    \
    } while (0)

int main(void) {
    enum { B = 3, HQ = 8, HKV = 2, S = 16, D = 128, SPARE = 5 };
    const int32_t seq[B] = {50, 17, 33};
    int32_t indptr[B + 1];
    indptr[0] = 0;
    for (int r = 0; r < B; ++r) indptr[r + 1] = indptr[r] + (seq[r] + S - 1) / S;
    const int32_t nnz = indptr[B], P = nnz + SPARE;
    int32_t perm[64];
    for (int i = 0; i < P; ++i) perm[i] = i;
    for (int i = P - 1; i > 0; --i) { /* physical pages in a shuffled order */
        int j = (int)(next_u64() % (uint64_t)(i + 1));
        int32_t t = perm[i];
        perm[i] = perm[j];
        perm[j] = t;
    }
    int32_t indices[64];
    for (int i = 0; i < nnz; ++i) indices[i] = perm[i];

    int32_t ntok = 0;
    for (int r = 0; r < B; ++r) ntok += seq[r];
    int64_t *slots = malloc(sizeof(int64_t) * ntok);
    uint16_t *k = malloc(2u * ntok * HKV * D), *v = malloc(2u * ntok * HKV * D);
    uint16_t *q = malloc(2u * B * HQ * D);
    int32_t n = 0;
    for (int r = 0; r < B; ++r)
        for (int t = 0; t < seq[r]; ++t, ++n) slots[n] = (int64_t)indices[indptr[r] + t / S] * S + t % S;
    for (int32_t i = 0; i < ntok * HKV * D; ++i) {
        k[i] = to_bf16(normal());
        v[i] = to_bf16(normal());
    }
    for (int i = 0; i < B * HQ * D; ++i) q[i] = to_bf16(normal());
    uint32_t tags[64], expected[64];
    for (int p = 0; p < P; ++p) tags[p] = (uint32_t)next_u64();
    for (int i = 0; i < nnz; ++i) expected[i] = tags[indices[i]];
    tags[indices[indptr[1] + 1]] += 1u; /* request 1's second page was reallocated: it must abort */

    /* device side, through the C ABI only */
    void *dk, *dv, *dq, *dout, *dws;
    int64_t *dslots;
    float *dks, *dvs;
    uint8_t *dkc, *dvc, *dmask;
    int32_t *dindptr, *dindices, *dseq;
    uint32_t *dtags, *dexp;
    const size_t pool = (size_t)P * HKV * S * D;
    CK(cudaMalloc(&dk, 2u * ntok * HKV * D));
    CK(cudaMalloc(&dv, 2u * ntok * HKV * D));
    CK(cudaMalloc(&dq, 2u * B * HQ * D));
    CK(cudaMalloc(&dout, 2u * B * HQ * D));
    CK(cudaMalloc((void **)&dslots, sizeof(int64_t) * ntok));
    CK(cudaMalloc((void **)&dks, sizeof(float) * HKV));
    CK(cudaMalloc((void **)&dvs, sizeof(float) * HKV));
    CK(cudaMalloc((void **)&dkc, pool));
    CK(cudaMalloc((void **)&dvc, pool));
    CK(cudaMalloc((void **)&dmask, B));
    CK(cudaMalloc((void **)&dindptr, sizeof(indptr)));
    CK(cudaMalloc((void **)&dindices, sizeof(int32_t) * nnz));
    CK(cudaMalloc((void **)&dseq, sizeof(seq)));
    CK(cudaMalloc((void **)&dtags, sizeof(uint32_t) * P));
    CK(cudaMalloc((void **)&dexp, sizeof(uint32_t) * nnz));
    CK(cudaMemcpy(dk, k, 2u * ntok * HKV * D, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dv, v, 2u * ntok * HKV * D, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dq, q, 2u * B * HQ * D, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dslots, slots, sizeof(int64_t) * ntok, cudaMemcpyHostToDevice));
    CK(cudaMemset(dkc, 0, pool));
    CK(cudaMemset(dvc, 0, pool));
    CK(cudaMemcpy(dindptr, indptr, sizeof(indptr), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dindices, indices, sizeof(int32_t) * nnz, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dseq, seq, sizeof(seq), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dtags, tags, sizeof(uint32_t) * P, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dexp, expected, sizeof(uint32_t) * nnz, cudaMemcpyHostToDevice));

    const size_t ws_bytes = paged_decode_attn_workspace_size(B, HQ, HKV, D, FKV_KV_FP8_E4M3);
    if (ws_bytes == 0) {
        fprintf(stderr, "workspace size query failed\n");
        return 3;
    }
    CK(cudaMalloc(&dws, ws_bytes));
    const float sm_scale = 1.0f / sqrtf((float)D);
    FK(kv_calibrate_scales(dk, dv, ntok, HKV, D, dks, dvs, NULL));
    FK(kv_append_fp8(dk, dv, dslots, ntok, dks, dvs, dkc, dvc, P, HKV, S, D, NULL));
    FK(kv_page_tag_check(dtags, P, dindptr, dindices, dexp, B, nnz, dmask, NULL));
    /* the same append and check in one launch, into a second pair of pools and a second mask */
    uint8_t *dkc2, *dvc2, *dmask2;
    CK(cudaMalloc((void **)&dkc2, pool));
    CK(cudaMalloc((void **)&dvc2, pool));
    CK(cudaMalloc((void **)&dmask2, B));
    CK(cudaMemset(dkc2, 0, pool));
    CK(cudaMemset(dvc2, 0, pool));
    FK(kv_append_fp8_tag_check(dk, dv, dslots, ntok, dks, dvs, dkc2, dvc2, P, HKV, S, D, dtags, dindptr, dindices,
                               dexp, B, nnz, dmask2, NULL));
    FK(paged_decode_attn(dq, B, HQ, dkc, dvc, FKV_KV_FP8_E4M3, dks, dvs, P, HKV, S, D, dindptr, dindices, nnz,
                         dseq, dmask, sm_scale, dout, dws, ws_bytes, NULL));
    CK(cudaDeviceSynchronize());
    uint32_t dev_err = 0;
    FK(fkv_device_error(&dev_err, 1));

    float gks[HKV], gvs[HKV];
    uint8_t *gkc = malloc(pool), *gvc = malloc(pool), gmask[B];
    uint16_t *gout = malloc(2u * B * HQ * D);
    CK(cudaMemcpy(gks, dks, sizeof gks, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gvs, dvs, sizeof gvs, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gkc, dkc, pool, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gvc, dvc, pool, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gmask, dmask, B, cudaMemcpyDeviceToHost));
    uint8_t *gkc2 = malloc(pool), *gvc2 = malloc(pool), gmask2[B];
    CK(cudaMemcpy(gkc2, dkc2, pool, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gvc2, dvc2, pool, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gmask2, dmask2, B, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gout, dout, 2u * B * HQ * D, cudaMemcpyDeviceToHost));

    /* the oracle */
    float oks[HKV], ovs[HKV];
    uint8_t *okc = calloc(pool, 1), *ovc = calloc(pool, 1), omask[B];
    double *oout = malloc(sizeof(double) * B * HQ * D);
    oracle_kv_calibrate_scales(k, v, ntok, HKV, D, oks, ovs);
    oracle_kv_append_fp8(k, v, slots, ntok, oks, ovs, okc, ovc, P, HKV, S, D);
    oracle_kv_page_tag_check(tags, P, indptr, indices, expected, B, nnz, omask);
    oracle_paged_decode_attn(q, B, HQ, okc, ovc, 1, oks, ovs, P, HKV, S, D, indptr, indices, nnz, seq, omask,
                             1.0 / sqrt((double)D), NULL, B * HQ, oout);

    int fails = 0;
    if (memcmp(gks, oks, sizeof gks) || memcmp(gvs, ovs, sizeof gvs)) {
        fprintf(stderr, "scales differ from the oracle\n");
        ++fails;
    }
    if (memcmp(gkc, okc, pool) || memcmp(gvc, ovc, pool)) {
        fprintf(stderr, "pool bytes differ from the oracle\n");
        ++fails;
    }
    if (memcmp(gkc2, okc, pool) || memcmp(gvc2, ovc, pool) || memcmp(gmask2, omask, B)) {
        fprintf(stderr, "the append-and-check launch differs from the oracle\n");
        ++fails;
    }
    if (memcmp(gmask, omask, B) || omask[1] != 1 || omask[0] != 0 || omask[2] != 0) {
        fprintf(stderr, "abort mask %d%d%d (oracle %d%d%d)\n", gmask[0], gmask[1], gmask[2], omask[0], omask[1],
                omask[2]);
        ++fails;
    }
    double max_err = 0.0;
    int bad = 0;
    for (int i = 0; i < B * HQ * D; ++i) {
        const double g = bf16_value(gout[i]), o = oout[i], e = fabs(g - o);
        if (e > max_err) max_err = e;
        if (e > 2e-3 && e > 1e-2 * fabs(o)) ++bad;
        if (i / (HQ * D) == 1 && g != 0.0) ++bad; /* the aborted request's row is zero */
    }
    if (bad) {
        fprintf(stderr, "%d attention elements outside the tolerance (max abs err %g)\n", bad, max_err);
        ++fails;
    }
    if (dev_err) {
        fprintf(stderr, "device error word %#x\n", dev_err);
        ++fails;
    }
    if (fails) return 1;
    printf("c abi decode step ok: %d tokens, scales and %zu pool bytes bit-exact, mask %d%d%d, max abs err %.3g\n",
           ntok, 2 * pool, gmask[0], gmask[1], gmask[2], max_err);
    return 0;
}
