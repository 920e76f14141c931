// decode_attn_noalloc.cu -- paged_decode_attn for callers that cannot allocate.
//
// Some callers of this library have no way to obtain device memory of their
// own: a plugin inside a host runtime that owns every device allocation and
// hands the plugin only its input and output buffers, or a latency-critical
// serving loop that forbids cudaMalloc on its hot path because the call can
// synchronise the device and stall every other stream.  Such callers cannot
// provide the scratch workspace that paged_decode_attn needs.
//
// paged_decode_attn_noalloc runs the same computation with its scratch in a
// fixed array compiled into this library instead.  It allocates nothing: no
// cudaMalloc, no cudaFree, no allocating library routine.  The array below
// exists once per GPU that loads the library and stays reserved until the
// process exits.
#include <mutex>

#include "fkv_common.cuh"

namespace fkv {
namespace {

constexpr size_t kScratchBytes = FKV_NOALLOC_SCRATCH_BYTES;

// Device scratch shared by every call on a device.  In host code this name is
// only a stand-in for the device symbol, never a device address: the address
// comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
CachedSymbol g_scratch[kMaxDevices];

// Device address of the scratch array on the current device.  It is looked
// up (cudaGetSymbolAddress, with the device current) the first time this
// entry point runs in a context and kept with that context's id; when the
// context changes -- cudaDeviceReset, or a primary context released and
// created again, after which the library's device code is loaded anew and
// the array may sit elsewhere -- the old address is dropped and looked up
// again.
void *scratch_for_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    CachedSymbol &c = g_scratch[dev];
    const unsigned long long ctx = current_context_id();
    if (ctx != 0 && ctx == c.ctx_id && c.ptr) return c.ptr;
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
    c.ptr = ptr;
    // Read after the lookup, which makes the primary context current if
    // nothing had; an id of 0 is never matched, so the address is then
    // looked up on every call.
    c.ctx_id = current_context_id();
    return ptr;
}

}  // namespace
}  // namespace fkv

extern "C" fkv_status paged_decode_attn_noalloc(const void *q, int32_t batch, int32_t num_q_heads,
                                                const void *k_cache, const void *v_cache, int32_t kv_dtype,
                                                const float *k_scale, const float *v_scale, int32_t num_pages,
                                                int32_t num_kv_heads, int32_t page_size, int32_t head_dim,
                                                const int32_t *page_indptr, const int32_t *page_indices,
                                                int64_t nnz, const int32_t *seq_lens, const uint8_t *abort_mask,
                                                float sm_scale, void *out, void *stream) {
    if (batch > 0) {
        const size_t need =
            paged_decode_attn_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, kv_dtype);
        if (need > fkv::kScratchBytes) return FKV_ERR_SCRATCH_LIMIT;
    }
    void *scratch = fkv::scratch_for_current_device();
    if (!scratch) return FKV_ERR_CUDA;
    // The existing call does the rest; its plan kernel clears the arrival
    // counters at the start of every call, so nothing left in the scratch by
    // an earlier call is read.
    return paged_decode_attn(q, batch, num_q_heads, k_cache, v_cache, kv_dtype, k_scale, v_scale, num_pages,
                             num_kv_heads, page_size, head_dim, page_indptr, page_indices, nnz, seq_lens,
                             abort_mask, sm_scale, out, scratch, fkv::kScratchBytes, stream);
}
