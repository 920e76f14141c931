// kv_append.cu -- quantize-on-write of new tokens into the paged KV pools.
//
// Cloudflare post ("Smaller, faster, safer: running Kimi and GLM at scale", as
// extracted on the "Cloudflare Workers AI Optimizes Large Model Serving ..."
// page): the KV cache is stored as 8-bit floating point (FP8, e4m3) instead of
// BF16, which halves its size.  One fp32 scale per KV head (per layer) maps
// bf16 values into e4m3's range.
//
// Each thread handles 8 consecutive elements of one (token, kv head, K|V)
// row: a 16-byte bf16 load, eight IEEE fp32 divisions, four
// round-to-nearest-even saturating conversions, one 8-byte store.  Two warps'
// worth of threads cover K and V of one (token, head); the pool layout is
// [page][head][slot][128].  The work is tiny per decode step (one token per
// request) and plain bandwidth for a bulk prefill write.
#include "fkv_common.cuh"

namespace fkv {

constexpr int kHeadDim = 128;
constexpr int kChunks = kHeadDim / 8;     // 16-byte bf16 chunks per row

__global__ void __launch_bounds__(256)
kv_append_fp8_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                     const int64_t *__restrict__ slots, int64_t n_tokens,
                     const float *__restrict__ k_scale, const float *__restrict__ v_scale,
                     uint8_t *__restrict__ k_cache, uint8_t *__restrict__ v_cache,
                     int32_t num_pages, int32_t num_kv_heads, int32_t page_size, uint32_t *err) {
    grid_dep_wait();        // earlier readers of the pool (attention) have finished
    grid_dep_launch();
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t per_token = static_cast<int64_t>(num_kv_heads) * 2 * kChunks;
    const int64_t n = gid / per_token;
    if (n >= n_tokens) return;
    const int rem = static_cast<int>(gid - n * per_token);
    const int h = rem / (2 * kChunks);
    const bool is_v = (rem / kChunks) & 1;
    const int chunk = rem % kChunks;
    const int64_t slot = __ldg(slots + n);
    if (slot < 0) return;                          // padding token
    const int64_t page = slot / page_size;
    const int64_t off = slot - page * page_size;
    if (page >= num_pages) {                       // outside the pool: skip, record
        if (rem == 0) atomicOr(err, FKV_DEVERR_APPEND_SLOT);
        return;
    }
    const int64_t row = n * num_kv_heads + h;
    const uint4 raw = __ldg((is_v ? v_new : k_new) + row * kChunks + chunk);
    const float scale = __ldg((is_v ? v_scale : k_scale) + h);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t packed[2];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        float x[4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint32_t u = w[2 * p + j];
            x[2 * j] = __uint_as_float(u << 16);              // bf16 -> fp32, exact
            x[2 * j + 1] = __uint_as_float(u & 0xFFFF0000u);
        }
        // one IEEE round-to-nearest division each, then one RNE to e4m3
        const uint16_t c01 = f32x2_to_e4m3x2(__fdiv_rn(x[1], scale), __fdiv_rn(x[0], scale));
        const uint16_t c23 = f32x2_to_e4m3x2(__fdiv_rn(x[3], scale), __fdiv_rn(x[2], scale));
        packed[p] = static_cast<uint32_t>(c01) | (static_cast<uint32_t>(c23) << 16);
    }
    uint8_t *dst = (is_v ? v_cache : k_cache) +
                   ((page * num_kv_heads + h) * page_size + off) * kHeadDim + chunk * 8;
    *reinterpret_cast<uint2 *>(dst) = make_uint2(packed[0], packed[1]);
}

__global__ void __launch_bounds__(256)
kv_append_bf16_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                      const int64_t *__restrict__ slots, int64_t n_tokens,
                      uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                      int32_t num_pages, int32_t num_kv_heads, int32_t page_size, uint32_t *err) {
    grid_dep_wait();        // earlier readers of the pool (attention) have finished
    grid_dep_launch();
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t per_token = static_cast<int64_t>(num_kv_heads) * 2 * kChunks;
    const int64_t n = gid / per_token;
    if (n >= n_tokens) return;
    const int rem = static_cast<int>(gid - n * per_token);
    const int h = rem / (2 * kChunks);
    const bool is_v = (rem / kChunks) & 1;
    const int chunk = rem % kChunks;
    const int64_t slot = __ldg(slots + n);
    if (slot < 0) return;
    const int64_t page = slot / page_size;
    const int64_t off = slot - page * page_size;
    if (page >= num_pages) {
        if (rem == 0) atomicOr(err, FKV_DEVERR_APPEND_SLOT);
        return;
    }
    const int64_t row = n * num_kv_heads + h;
    const uint4 raw = __ldg((is_v ? v_new : k_new) + row * kChunks + chunk);
    (is_v ? v_cache : k_cache)[((page * num_kv_heads + h) * page_size + off) * kChunks + chunk] = raw;
}

static fkv_status check_append_args(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                                    int32_t n_tokens, const void *k_cache, const void *v_cache,
                                    int32_t num_pages, int32_t num_kv_heads, int32_t page_size,
                                    int32_t head_dim) {
    if (n_tokens < 0 || num_pages <= 0 || num_kv_heads <= 0 || page_size <= 0) return FKV_ERR_INVALID_ARG;
    if (head_dim != kHeadDim) return FKV_ERR_UNSUPPORTED;
    if (n_tokens == 0) return FKV_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return FKV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return FKV_ERR_INVALID_ARG;
    return FKV_OK;
}

}  // namespace fkv

using namespace fkv;

extern "C" fkv_status kv_append_fp8(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                                    int32_t n_tokens, const float *k_scale, const float *v_scale,
                                    uint8_t *k_cache, uint8_t *v_cache, int32_t num_pages,
                                    int32_t num_kv_heads, int32_t page_size, int32_t head_dim,
                                    void *stream) {
    fkv_status st = check_append_args(k_new, v_new, slot_mapping, n_tokens, k_cache, v_cache, num_pages,
                                      num_kv_heads, page_size, head_dim);
    if (st != FKV_OK || n_tokens == 0) return st;
    if (!k_scale || !v_scale) return FKV_ERR_INVALID_ARG;
    uint32_t *err = device_error_word();
    if (!err) return FKV_ERR_CUDA;
    const int64_t threads = static_cast<int64_t>(n_tokens) * num_kv_heads * 2 * kChunks;
    const int64_t blocks = (threads + 255) / 256;
    if (blocks > 0x7FFFFFFFLL) return FKV_ERR_INVALID_ARG;
    const cudaError_t e = launch_pdl(kv_append_fp8_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                                     static_cast<cudaStream_t>(stream), static_cast<const uint4 *>(k_new),
                                     static_cast<const uint4 *>(v_new), slot_mapping, static_cast<int64_t>(n_tokens),
                                     k_scale, v_scale, k_cache, v_cache, num_pages, num_kv_heads, page_size, err);
    return e == cudaSuccess ? FKV_OK : FKV_ERR_CUDA;
}

extern "C" fkv_status kv_append_bf16(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                                     int32_t n_tokens, void *k_cache, void *v_cache, int32_t num_pages,
                                     int32_t num_kv_heads, int32_t page_size, int32_t head_dim,
                                     void *stream) {
    fkv_status st = check_append_args(k_new, v_new, slot_mapping, n_tokens, k_cache, v_cache, num_pages,
                                      num_kv_heads, page_size, head_dim);
    if (st != FKV_OK || n_tokens == 0) return st;
    uint32_t *err = device_error_word();
    if (!err) return FKV_ERR_CUDA;
    const int64_t threads = static_cast<int64_t>(n_tokens) * num_kv_heads * 2 * kChunks;
    const int64_t blocks = (threads + 255) / 256;
    if (blocks > 0x7FFFFFFFLL) return FKV_ERR_INVALID_ARG;
    const cudaError_t e = launch_pdl(kv_append_bf16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                                     static_cast<cudaStream_t>(stream), static_cast<const uint4 *>(k_new),
                                     static_cast<const uint4 *>(v_new), slot_mapping, static_cast<int64_t>(n_tokens),
                                     static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), num_pages,
                                     num_kv_heads, page_size, err);
    return e == cudaSuccess ? FKV_OK : FKV_ERR_CUDA;
}
