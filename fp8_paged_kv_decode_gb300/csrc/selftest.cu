// selftest.cu -- the failure path of the kernels' bounded waits, run on purpose.
//
// Every wait in the library's kernels is on an mbarrier that a copy (or the
// other warp of a CTA) completes, and gives up after a time limit: the
// kernel then records FKV_DEVERR_TIMEOUT in the device error word and ends
// normally, so the context stays usable.  fkv_selftest_wait runs the two wait
// helpers those kernels use -- the spinning one of the computing warps and
// the sleeping one of a producer warp -- on an mbarrier that nothing
// completes, so the path can be seen working on the GPU without a fault: the
// waits end after limit_ns, the error bit is set, later calls still work.
// With `complete`, the block completes the barrier first and both waits must
// return at once.
#include "fkv_common.cuh"

namespace fkv {

constexpr uint64_t kSelftestMaxNs = 10000000000ull;   // at most 10 s of waiting

__global__ void __launch_bounds__(64) selftest_wait_kernel(uint64_t limit_ns, int complete, uint32_t *err,
                                                           uint32_t *result) {
    __shared__ __align__(8) uint64_t bar_word;
    const uint32_t bar = smem_u32(&bar_word);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (complete && threadIdx.x == 0) mbar_arrive(bar);     // phase 0 completes
    __syncthreads();
    const bool ok = threadIdx.x < 32 ? mbar_wait_bounded(bar, 0, limit_ns)
                                     : mbar_wait_bounded_sleep(bar, 0, limit_ns);
    if ((threadIdx.x & 31) == 0) {
        if (!ok) atomicOr(err, FKV_DEVERR_TIMEOUT);
        if (result) result[threadIdx.x >> 5] = ok ? 1u : 0u;
    }
}

}  // namespace fkv

using namespace fkv;

extern "C" fkv_status fkv_selftest_wait(uint64_t limit_ns, int32_t complete, uint32_t *result, void *stream) {
    if (limit_ns > kSelftestMaxNs) return FKV_ERR_INVALID_ARG;
    uint32_t *err = device_error_word();
    if (!err) return FKV_ERR_CUDA;
    selftest_wait_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, complete ? 1 : 0, err, result);
    return cudaGetLastError() == cudaSuccess ? FKV_OK : FKV_ERR_CUDA;
}
