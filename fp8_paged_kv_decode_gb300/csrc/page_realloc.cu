// page_realloc.cu -- hand physical pages to new owners on the device.
//
// "Kimi and GLM Reasoning Slimming: Hands-On Test", section "Giving Every
// Physical Cache Page a 'Generation Number'", and the Cloudflare post's
// integrity-checking section: a page's tag changes each time the page is
// reallocated, so a request still holding the old (page, tag) pair fails the
// integrity check.  The same page mentions clearing GPU memory as a further
// defence; the optional scrub zeroes the page's K and V bytes.
//
// One CTA per (listed page, 16 KB chunk of the page): the chunk-0 CTA of each
// page bumps its tag and records the new tag for the new owner; every CTA of
// a page zeroes its chunk of K and V when a scrub is asked for.
#include "fkv_common.cuh"

namespace fkv {

constexpr int kScrubThreads = 256;
constexpr int kScrubChunk = kScrubThreads * 4 * 16;    // bytes of K (and of V) zeroed per CTA

__global__ void __launch_bounds__(kScrubThreads)
kv_page_realloc_kernel(uint32_t *__restrict__ page_tags, int32_t num_pages, const int32_t *__restrict__ pages,
                       uint32_t *__restrict__ new_tags, uint8_t *__restrict__ k_cache,
                       uint8_t *__restrict__ v_cache, int64_t page_bytes, uint32_t *err) {
    grid_dep_wait();          // earlier kernels (attention reading these pages) have finished
    grid_dep_launch();
    const int j = blockIdx.x;
    const int32_t p = __ldg(pages + j);
    const bool in_pool = p >= 0 && p < num_pages;
    if (blockIdx.y == 0 && threadIdx.x == 0) {
        if (in_pool) {
            new_tags[j] = atomicAdd(page_tags + p, 1u) + 1u;      // wraps modulo 2^32
        } else {
            new_tags[j] = 0u;
            atomicOr(err, FKV_DEVERR_REALLOC_PAGE);
        }
    }
    if (!in_pool || k_cache == nullptr) return;
    const int64_t c0 = static_cast<int64_t>(blockIdx.y) * kScrubChunk;
    uint4 *kp = reinterpret_cast<uint4 *>(k_cache + static_cast<int64_t>(p) * page_bytes + c0);
    uint4 *vp = reinterpret_cast<uint4 *>(v_cache + static_cast<int64_t>(p) * page_bytes + c0);
    const int64_t n16 = min(static_cast<int64_t>(kScrubChunk), page_bytes - c0) / 16;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int64_t i = threadIdx.x; i < n16; i += kScrubThreads) {
        kp[i] = z;
        vp[i] = z;
    }
}

}  // namespace fkv

using namespace fkv;

extern "C" fkv_status kv_page_realloc(uint32_t *page_tags, int32_t num_pages, const int32_t *pages, int32_t n,
                                      uint32_t *new_tags, void *k_cache, void *v_cache, int32_t kv_dtype,
                                      int32_t num_kv_heads, int32_t page_size, int32_t head_dim, void *stream) {
    if (n < 0 || num_pages < 0) return FKV_ERR_INVALID_ARG;
    if (n == 0) return FKV_OK;
    if (!page_tags || !pages || !new_tags) return FKV_ERR_INVALID_ARG;
    if ((k_cache == nullptr) != (v_cache == nullptr)) return FKV_ERR_INVALID_ARG;
    int64_t page_bytes = 0;
    unsigned chunks = 1;
    if (k_cache) {
        if (kv_dtype != FKV_KV_FP8_E4M3 && kv_dtype != FKV_KV_BF16) return FKV_ERR_INVALID_ARG;
        if (num_kv_heads <= 0 || page_size <= 0) return FKV_ERR_INVALID_ARG;
        if (head_dim != 128) return FKV_ERR_UNSUPPORTED;
        if (!aligned16(k_cache) || !aligned16(v_cache)) return FKV_ERR_INVALID_ARG;
        page_bytes = static_cast<int64_t>(num_kv_heads) * page_size * head_dim * (kv_dtype == FKV_KV_BF16 ? 2 : 1);
        const int64_t c = (page_bytes + kScrubChunk - 1) / kScrubChunk;
        if (c > 65535) return FKV_ERR_UNSUPPORTED;
        chunks = static_cast<unsigned>(c);
    }
    uint32_t *err = device_error_word();
    if (!err) return FKV_ERR_CUDA;
    const cudaError_t e = launch_pdl(kv_page_realloc_kernel, dim3(static_cast<unsigned>(n), chunks),
                                     dim3(kScrubThreads), 0, static_cast<cudaStream_t>(stream), page_tags, num_pages,
                                     pages, new_tags, static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache),
                                     page_bytes, err);
    return e == cudaSuccess ? FKV_OK : FKV_ERR_CUDA;
}
