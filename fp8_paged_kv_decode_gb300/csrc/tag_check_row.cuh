// tag_check_row.cuh -- one request's row of the per-page generation-tag check.
//
// "Kimi and GLM Reasoning Slimming: Hands-On Test", section "Giving Every
// Physical Cache Page a 'Generation Number'": for each page a request expects,
// the live tag of the page is compared with the tag the request recorded; any
// difference (or a page that does not exist) aborts the request.  Shared by
// the stand-alone check kernel and by the append kernel that runs the check
// in the same launch, so both compute the same mask by construction.
#pragma once

#include "fkv_common.cuh"

namespace fkv {

// Called by all kThreads threads of a block for request r; returns the
// request's verdict (nonzero: abort) in every thread.  The threads stride
// over the request's CSR row with four independent gathers in flight each
// (the tag array is small and stays in L2) and the block ORs the verdicts.
template <int kThreads>
__device__ __forceinline__ int tag_check_row(const uint32_t *__restrict__ page_tags, int32_t num_pages,
                                             const int32_t *__restrict__ page_indptr,
                                             const int32_t *__restrict__ page_indices,
                                             const uint32_t *__restrict__ expected_tags, int64_t nnz, int r) {
    const int64_t begin = __ldg(page_indptr + r);
    const int64_t end = __ldg(page_indptr + r + 1);
    int bad = 0;
    if (begin < 0 || end < begin || end > nnz) {
        bad = 1;                                            // malformed row: fail closed
    } else {
        int64_t j = begin + threadIdx.x;
        for (; j + 3 * kThreads < end; j += 4 * kThreads) {
            int32_t p[4];
            uint32_t e[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                p[u] = __ldg(page_indices + j + u * kThreads);
                e[u] = __ldg(expected_tags + j + u * kThreads);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (p[u] < 0 || p[u] >= num_pages) bad = 1;        // no such page
                else bad |= __ldg(page_tags + p[u]) != e[u];     // stale or mismatched
            }
        }
        for (; j < end; j += kThreads) {
            const int32_t p = __ldg(page_indices + j);
            const uint32_t e = __ldg(expected_tags + j);
            if (p < 0 || p >= num_pages) bad = 1;
            else bad |= __ldg(page_tags + p) != e;
        }
    }
    return __syncthreads_or(bad);
}

}  // namespace fkv
