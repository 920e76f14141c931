// kv_calibrate.cu -- per-KV-head FP8 scales for a bulk (prefill) write.
//
// The Cloudflare post keeps prefill in BF16 and stores the cache that decode
// reads as FP8 e4m3 ("Smaller, faster, safer: running Kimi and GLM at scale",
// extracted on the "Cloudflare Workers AI Optimizes Large Model Serving ..."
// page).  Handing a prompt's K/V to the FP8 cache needs one scale per KV head;
// this computes scale = fl32(amax / 448) from the prompt itself (448 is the
// largest finite e4m3 magnitude; an all-zero head gets 1), after which
// kv_append_fp8 writes the whole prompt.
//
// Pass 1: each CTA reduces |x| of one (KV head, K or V) over a strided set of
// tokens, 16 lanes per 128-element row.  The maximum is kept as the bf16
// magnitude bits: for non-negative values the integer order of the bits is
// the numeric order, so warp shuffles and one integer atomicMax per CTA
// (into the output array, cleared first) suffice.  Pass 2 turns each maximum
// into its scale with one IEEE division, in place.
#include <algorithm>

#include "fkv_common.cuh"

namespace fkv {

constexpr int kCalThreads = 256;
constexpr int kCalRows = kCalThreads / 16;    // token rows per CTA per iteration

constexpr int kCalUnroll = 4;                 // rows whose loads each thread keeps in flight
constexpr int kCalBlocksPerSM = 8;            // resident CTAs per SM the kernel is compiled for

__global__ void __launch_bounds__(kCalThreads, kCalBlocksPerSM)
kv_amax_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v, int64_t n_tokens, int32_t num_kv_heads,
               uint32_t *__restrict__ k_amax, uint32_t *__restrict__ v_amax) {
    grid_dep_wait();
    grid_dep_launch();
    __shared__ uint32_t s_max[kCalThreads / 32];
    const int h = blockIdx.y;
    const bool is_v = blockIdx.z != 0;
    const uint4 *src = is_v ? v : k;
    const int lane16 = threadIdx.x & 15;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kCalRows;
    uint32_t mx = 0;
    for (int64_t n0 = static_cast<int64_t>(blockIdx.x) * kCalRows + (threadIdx.x >> 4); n0 < n_tokens;
         n0 += kCalUnroll * stride) {
        uint4 x[kCalUnroll];
#pragma unroll
        for (int u = 0; u < kCalUnroll; ++u) {       // every load issued before any is used
            const int64_t n = n0 + u * stride;
            x[u] = n < n_tokens ? __ldg(src + (n * num_kv_heads + h) * 16 + lane16) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kCalUnroll; ++u) {
            const uint32_t w[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) mx = max(mx, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t m = 0;
        for (int i = 0; i < kCalThreads / 32; ++i) m = max(m, s_max[i]);
        atomicMax((is_v ? v_amax : k_amax) + h, m << 16);        // bf16 bits -> fp32 bits
    }
}

__global__ void kv_scale_finalize_kernel(float *__restrict__ k_scale, float *__restrict__ v_scale,
                                         int32_t num_kv_heads) {
    grid_dep_wait();
    grid_dep_launch();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= 2 * num_kv_heads) return;
    float *s = i < num_kv_heads ? k_scale + i : v_scale + (i - num_kv_heads);
    const float amax = *s;                                      // holds the maximum's bits
    *s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
}

}  // namespace fkv

using namespace fkv;

extern "C" fkv_status kv_calibrate_scales(const void *k, const void *v, int64_t n_tokens, int32_t num_kv_heads,
                                          int32_t head_dim, float *k_scale, float *v_scale, void *stream) {
    if (n_tokens < 0 || num_kv_heads <= 0 || num_kv_heads > 65535) return FKV_ERR_INVALID_ARG;
    if (head_dim != 128) return FKV_ERR_UNSUPPORTED;
    if (!k_scale || !v_scale) return FKV_ERR_INVALID_ARG;
    if (n_tokens > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return FKV_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(k_scale, 0, sizeof(float) * num_kv_heads, st) != cudaSuccess ||
        cudaMemsetAsync(v_scale, 0, sizeof(float) * num_kv_heads, st) != cudaSuccess)
        return FKV_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    if (n_tokens > 0) {
        const int sms = device_sm_count();
        int64_t gx = (n_tokens + kCalRows - 1) / kCalRows;
        // one wave: kCalBlocksPerSM CTAs per SM over all (KV head, K|V) pairs
        const int64_t target =
            std::max<int64_t>(1, static_cast<int64_t>(sms > 0 ? sms : 1) * kCalBlocksPerSM / (2 * num_kv_heads));
        gx = std::min(gx, target);
        e = launch_pdl(kv_amax_kernel, dim3(static_cast<unsigned>(gx), num_kv_heads, 2), dim3(kCalThreads), 0, st,
                       static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), n_tokens, num_kv_heads,
                       reinterpret_cast<uint32_t *>(k_scale), reinterpret_cast<uint32_t *>(v_scale));
        if (e != cudaSuccess) return FKV_ERR_CUDA;
    }
    e = launch_pdl(kv_scale_finalize_kernel, dim3((2 * num_kv_heads + 127) / 128), dim3(128), 0, st, k_scale,
                   v_scale, num_kv_heads);
    return e == cudaSuccess ? FKV_OK : FKV_ERR_CUDA;
}
