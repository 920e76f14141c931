// fkv_api.cu -- library-wide host helpers: status strings, the sticky device
// error word, cached device properties.
#include <mutex>
#include <string>

#include "fkv_common.cuh"

namespace fkv {

// Sticky error word: kernels OR FKV_DEVERR_* bits into it instead of trapping.
__device__ uint32_t g_device_error;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t *g_err_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}
}  // namespace

uint32_t *device_error_word() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<uint32_t *>(p);
    }
    return g_err_ptr[dev];
}

int device_sm_count() {
    const int dev = current_device();
    if (dev < 0) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace fkv

extern "C" const char *fkv_status_string(fkv_status s) {
    switch (s) {
        case FKV_OK: return "ok";
        case FKV_ERR_INVALID_ARG: return "invalid argument";
        case FKV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case FKV_ERR_CUDA: return "CUDA runtime error";
        case FKV_ERR_SCRATCH_LIMIT: return "shape needs more scratch than the no-allocation entry point holds";
    }
    return "unknown status";
}

extern "C" fkv_status fkv_device_error(uint32_t *flags, int32_t clear) {
    if (!flags) return FKV_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return FKV_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, fkv::g_device_error, sizeof v) != cudaSuccess) return FKV_ERR_CUDA;
    if (clear) {
        const uint32_t zero = 0;
        if (cudaMemcpyToSymbol(fkv::g_device_error, &zero, sizeof zero) != cudaSuccess) return FKV_ERR_CUDA;
    }
    *flags = v;
    return FKV_OK;
}

extern "C" int32_t fkv_kernels_per_call(const char *entry_point) {
    if (!entry_point) return -1;
    const std::string e(entry_point);
    if (e == "kv_append_fp8" || e == "kv_append_bf16" || e == "kv_page_tag_check" || e == "kv_page_realloc")
        return 1;
    if (e == "paged_decode_attn" || e == "paged_decode_attn_noalloc") return 2;   // plan, split attention
    if (e == "kv_calibrate_scales") return 2;                                     // amax, finalize
    return -1;
}
