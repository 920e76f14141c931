// fkv_api.cu -- library-wide host helpers: status strings, the sticky device
// error word, cached device properties.
#include <cudaTypedefs.h>

#include <mutex>
#include <string>

#include "fkv_common.cuh"

namespace fkv {

// Sticky error word: kernels OR FKV_DEVERR_* bits into it instead of trapping.
__device__ uint32_t g_device_error;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
CachedSymbol g_err_word[kMaxDevices];
int g_sm_count[kMaxDevices] = {};

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

PFN_cuCtxGetCurrent_v4000 g_ctx_get_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_get_id = nullptr;
std::once_flag g_ctx_fns_once;
}  // namespace

unsigned long long current_context_id() {
    std::call_once(g_ctx_fns_once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    });
    if (!g_ctx_get_current || !g_ctx_get_id) return 0;
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

uint32_t *device_error_word() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    CachedSymbol &c = g_err_word[dev];
    const unsigned long long ctx = current_context_id();
    if (ctx != 0 && ctx == c.ctx_id && c.ptr) return static_cast<uint32_t *>(c.ptr);
    // First use in this context, or a new context: look the address up again.
    // cudaGetSymbolAddress makes the primary context current if nothing had,
    // so the id is read after it (0: not cached, looked up on every call).
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess || !p) return nullptr;
    c.ptr = p;
    c.ctx_id = current_context_id();
    return static_cast<uint32_t *>(p);
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
    if (e == "kv_append_fp8" || e == "kv_append_bf16" || e == "kv_page_tag_check" || e == "kv_page_realloc" ||
        e == "kv_append_fp8_tag_check" || e == "kv_append_bf16_tag_check")
        return 1;
    if (e == "paged_decode_attn" || e == "paged_decode_attn_noalloc") return 2;   // plan, split attention
    if (e == "kv_calibrate_scales") return 2;                                     // amax, finalize
    return -1;
}
