// tag_check.cu -- the batched KV-page integrity check.
//
// "Kimi and GLM Reasoning Slimming: Hands-On Test", section "Giving Every
// Physical Cache Page a 'Generation Number'", and the Cloudflare post's
// integrity-checking section: every physical page carries a tag that changes
// when the page is reallocated; each request records the pages and tags it
// expects; before decode reads the cache the two are compared and a request
// with any mismatch is aborted (fail closed).  The post runs the validation
// as a separate batch pass, not fused into the attention kernel; this file is
// that pass.
//
// One CTA per request (tag_check_row.cuh); the abort mask stays on the
// device for the attention call.
#include "tag_check_row.cuh"

namespace fkv {

constexpr int kCheckThreads = 128;

__global__ void __launch_bounds__(kCheckThreads)
kv_page_tag_check_kernel(const uint32_t *__restrict__ page_tags, int32_t num_pages,
                         const int32_t *__restrict__ page_indptr, const int32_t *__restrict__ page_indices,
                         const uint32_t *__restrict__ expected_tags, int64_t nnz,
                         uint8_t *__restrict__ abort_mask) {
    grid_dep_wait();        // tags and tables written by earlier kernels are visible
    grid_dep_launch();
    const int r = blockIdx.x;
    const int bad = tag_check_row<kCheckThreads>(page_tags, num_pages, page_indptr, page_indices, expected_tags,
                                                 nnz, r);
    if (threadIdx.x == 0) abort_mask[r] = bad ? 1 : 0;
}

}  // namespace fkv

using namespace fkv;

extern "C" fkv_status kv_page_tag_check(const uint32_t *page_tags, int32_t num_pages,
                                        const int32_t *page_indptr, const int32_t *page_indices,
                                        const uint32_t *expected_tags, int32_t batch, int64_t nnz,
                                        uint8_t *abort_mask, void *stream) {
    if (batch < 0 || nnz < 0 || num_pages < 0) return FKV_ERR_INVALID_ARG;
    if (batch == 0) return FKV_OK;
    if (!page_indptr || !abort_mask) return FKV_ERR_INVALID_ARG;
    if (nnz > 0 && (!page_indices || !expected_tags)) return FKV_ERR_INVALID_ARG;
    if (num_pages > 0 && !page_tags) return FKV_ERR_INVALID_ARG;
    const cudaError_t e = launch_pdl(kv_page_tag_check_kernel, dim3(batch), dim3(kCheckThreads), 0,
                                     static_cast<cudaStream_t>(stream), page_tags, num_pages, page_indptr,
                                     page_indices, expected_tags, nnz, abort_mask);
    return e == cudaSuccess ? FKV_OK : FKV_ERR_CUDA;
}
