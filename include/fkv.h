/*
 * fkv.h -- C ABI of libfkv: FP8 paged-KV decode attention for sm_103a (GB300).
 *
 * The operations follow the description of Cloudflare's serving work in
 * "Cloudflare Workers AI Optimizes Large Model Serving with KV Cache
 * Quantization, Weight Compression, and Integrity Checks" (the extracted text
 * of the post "Smaller, faster, safer: running Kimi and GLM at scale") and
 * "Kimi and GLM Reasoning Slimming: Hands-On Test", section "Giving Every
 * Physical Cache Page a 'Generation Number'":
 *   - the KV cache is stored as FP8 e4m3 instead of BF16, halving its size;
 *   - the FP8 attention kernel converts cache values as it reads them;
 *   - every physical page has a tag that changes when it is reallocated; each
 *     request records the (page, tag) pairs it expects; a separate batch check
 *     (not fused into attention) runs before decode reads the cache, and a
 *     mismatching request is aborted (fail closed); deployments that do not
 *     enable the check pay nothing.
 *
 * Conventions for every call
 *   - All array arguments are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or retains them.  `stream` is a cudaStream_t
 *     passed as void* (NULL = the legacy default stream).
 *   - Calls are asynchronous on `stream`: no host synchronisation, no
 *     device-to-host copy.  Host-side argument checks return
 *     FKV_ERR_INVALID_ARG / FKV_ERR_UNSUPPORTED synchronously and launch
 *     nothing; a failed launch returns FKV_ERR_CUDA.
 *   - Data-dependent problems found on the device never trap: they are
 *     recorded in a sticky per-device error word (see fkv_device_error) and
 *     the affected output is handled as documented per call.
 *   - head_dim must be 128.  Cache, q and out must be 16-byte aligned.
 *
 * Layouts
 *   KV pool (one per K and one per V, per layer):
 *       [num_pages][num_kv_heads][page_size][head_dim]
 *     one (page, head) tile is page_size * head_dim contiguous elements;
 *     elements are e4m3 codes (1 byte) or bf16 (2 bytes).
 *   Page table (CSR): page_indptr int32[batch + 1], page_indices int32[nnz];
 *     token t of request r lives in page page_indices[page_indptr[r] + t /
 *     page_size] at offset t % page_size.
 *   Queries / outputs: bf16 [batch][num_q_heads][head_dim]; query head i
 *     attends with KV head i / (num_q_heads / num_kv_heads).
 */
#ifndef FKV_H_
#define FKV_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FKV_API __attribute__((visibility("default")))
#else
#define FKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FKV_OK = 0,
    FKV_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misalignment, small workspace */
    FKV_ERR_UNSUPPORTED = 2,   /* valid but not implemented (head_dim != 128, a group size that does not split into groups of <= 8, ...) */
    FKV_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    FKV_ERR_SCRATCH_LIMIT = 4  /* paged_decode_attn_noalloc: the shape needs more scratch than
                                  FKV_NOALLOC_SCRATCH_BYTES */
} fkv_status;

typedef enum {
    FKV_KV_FP8_E4M3 = 0,
    FKV_KV_BF16 = 1
} fkv_kv_dtype;

/* Bits of the sticky device error word. */
#define FKV_DEVERR_APPEND_SLOT   0x1u  /* kv_append_*: slot beyond the pool, token skipped */
#define FKV_DEVERR_ATTN_PAGE     0x2u  /* paged_decode_attn: page id outside [0, num_pages), row zeroed */
#define FKV_DEVERR_TIMEOUT       0x4u  /* a bounded wait on a copy gave up; the call's output is not valid */
#define FKV_DEVERR_REALLOC_PAGE  0x8u  /* kv_page_realloc: a listed id is outside [0, num_pages), skipped */

FKV_API const char *fkv_status_string(fkv_status s);

/*
 * kv_append_fp8 -- quantize new tokens' K and V to e4m3 and write them into
 * their page slots.  (Cloudflare post: the cache is stored as FP8 e4m3 instead
 * of BF16.)  For every token n with slot = slot_mapping[n] >= 0, KV head h and
 * element d:
 *     code = e4m3_rne_satfinite( fl32( fl32(x) / scale[h] ) )
 * i.e. an IEEE round-to-nearest fp32 division followed by one
 * round-to-nearest-even to e4m3; |values| > 448 and +-Inf saturate to +-448,
 * NaN stays NaN.  The code goes to cache[slot / page_size][h][slot %
 * page_size][d].
 *
 *   k_new, v_new   bf16 [n_tokens][num_kv_heads][head_dim]
 *   slot_mapping   int64 [n_tokens]; < 0 means "padding, skip"
 *   k_scale, v_scale  fp32 [num_kv_heads], positive and finite (this layer)
 *   k_cache, v_cache  uint8 pools (layout above)
 * A slot whose page is >= num_pages is skipped and sets FKV_DEVERR_APPEND_SLOT.
 * Bytes outside the written slots are never touched.  n_tokens == 0 is a no-op.
 */
FKV_API fkv_status kv_append_fp8(const void *k_new, const void *v_new,
                         const int64_t *slot_mapping, int32_t n_tokens,
                         const float *k_scale, const float *v_scale,
                         uint8_t *k_cache, uint8_t *v_cache,
                         int32_t num_pages, int32_t num_kv_heads,
                         int32_t page_size, int32_t head_dim, void *stream);

/*
 * kv_append_bf16 -- the BF16-cache counterpart of kv_append_fp8 (the
 * comparison baseline the Cloudflare post measures against): the same
 * placement, values stored unchanged.
 */
FKV_API fkv_status kv_append_bf16(const void *k_new, const void *v_new,
                          const int64_t *slot_mapping, int32_t n_tokens,
                          void *k_cache, void *v_cache,
                          int32_t num_pages, int32_t num_kv_heads,
                          int32_t page_size, int32_t head_dim, void *stream);

/*
 * kv_calibrate_scales -- the per-KV-head scales for writing a whole prompt
 * into the FP8 cache (Cloudflare post: prefill keeps BF16, the cache decode
 * reads is FP8 e4m3).  For each KV head h, separately for K and for V:
 *     amax = max |x| over all n_tokens tokens and head_dim elements of head h
 *     scale[h] = fl32(amax / 448)  (IEEE division; 448 = largest e4m3 value),
 *                1 when amax is 0 (including n_tokens == 0)
 * then kv_append_fp8 with these scales quantizes the prompt (bulk write).
 *
 *   k, v      bf16 [n_tokens][num_kv_heads][head_dim], finite values
 *             (a NaN or Inf input gives a NaN or Inf scale)
 *   k_scale, v_scale  fp32 [num_kv_heads] outputs (also used as the
 *             reduction's scratch; nothing else is written)
 * Launches two kernels and two memsets on `stream`.
 */
FKV_API fkv_status kv_calibrate_scales(const void *k, const void *v, int64_t n_tokens,
                                       int32_t num_kv_heads, int32_t head_dim,
                                       float *k_scale, float *v_scale, void *stream);

/*
 * kv_page_tag_check -- the separate batched integrity pass ("Kimi and GLM
 * Reasoning Slimming: Hands-On Test", section "Giving Every Physical Cache
 * Page a 'Generation Number'"; Cloudflare post, integrity checking).  For each
 * request r:
 *     abort_mask[r] = 1  if its CSR row is malformed (indptr[r] < 0,
 *                        indptr[r+1] < indptr[r] or indptr[r+1] > nnz), or
 *                        for any j in [indptr[r], indptr[r+1]):
 *                        page_indices[j] outside [0, num_pages) or
 *                        page_tags[page_indices[j]] != expected_tags[j]
 *     abort_mask[r] = 0  otherwise.
 *
 *   page_tags      uint32 [num_pages]  live generation tags
 *   page_indptr    int32 [batch + 1], page_indices int32 [nnz]
 *   expected_tags  uint32 [nnz]  parallel to page_indices
 *   abort_mask     uint8 [batch]  output, stays on the device; pass it to
 *                  paged_decode_attn.  Not calling this function and passing
 *                  abort_mask = NULL there is the no-tracker path.
 * batch == 0 is a no-op.
 */
FKV_API fkv_status kv_page_tag_check(const uint32_t *page_tags, int32_t num_pages,
                             const int32_t *page_indptr, const int32_t *page_indices,
                             const uint32_t *expected_tags, int32_t batch, int64_t nnz,
                             uint8_t *abort_mask, void *stream);

/*
 * kv_append_fp8_tag_check -- kv_append_fp8 and kv_page_tag_check of one
 * decode step in a single launch.  (Cloudflare post, integrity checking: the
 * check runs as a separate batch pass before decode reads the cache, not
 * inside the attention kernel; this call keeps it a pass of its own and only
 * shares the append's launch.)
 *
 * Equivalent to kv_append_fp8(k_new ... head_dim) followed by
 * kv_page_tag_check(page_tags, num_pages, page_indptr, page_indices,
 * expected_tags, batch, nnz, abort_mask) on the same stream: the same cache
 * bytes, the same mask, the same argument checks and error codes.  The two
 * parts touch disjoint memory (the append writes only cache bytes, the check
 * reads tags and tables and writes only abort_mask), so the kernel runs them
 * side by side; the caller must not pass buffers that overlap across the two
 * parts.  page_tags has num_pages entries (the pool the append writes into).
 * n_tokens == 0 runs the check alone, batch == 0 the append alone.
 */
FKV_API fkv_status kv_append_fp8_tag_check(const void *k_new, const void *v_new,
                                   const int64_t *slot_mapping, int32_t n_tokens,
                                   const float *k_scale, const float *v_scale,
                                   uint8_t *k_cache, uint8_t *v_cache,
                                   int32_t num_pages, int32_t num_kv_heads,
                                   int32_t page_size, int32_t head_dim,
                                   const uint32_t *page_tags, const int32_t *page_indptr,
                                   const int32_t *page_indices, const uint32_t *expected_tags,
                                   int32_t batch, int64_t nnz, uint8_t *abort_mask, void *stream);

/*
 * kv_append_bf16_tag_check -- the same one-launch prologue for a BF16 cache:
 * kv_append_bf16 followed by kv_page_tag_check, with the same arguments,
 * results, argument checks and rules as kv_append_fp8_tag_check (no scales).
 */
FKV_API fkv_status kv_append_bf16_tag_check(const void *k_new, const void *v_new,
                                    const int64_t *slot_mapping, int32_t n_tokens,
                                    void *k_cache, void *v_cache,
                                    int32_t num_pages, int32_t num_kv_heads,
                                    int32_t page_size, int32_t head_dim,
                                    const uint32_t *page_tags, const int32_t *page_indptr,
                                    const int32_t *page_indices, const uint32_t *expected_tags,
                                    int32_t batch, int64_t nnz, uint8_t *abort_mask, void *stream);

/*
 * kv_page_realloc -- hand pages to new owners on the device ("Kimi and GLM
 * Reasoning Slimming: Hands-On Test", section "Giving Every Physical Cache
 * Page a 'Generation Number'": a page's tag changes each time it is
 * reallocated, so holders of the old (page, tag) pair fail the check; the
 * same page names clearing GPU memory as a further defence).  For each j:
 *     p = pages[j]; page_tags[p] += 1 (modulo 2^32); new_tags[j] = page_tags[p]
 * and, when k_cache / v_cache are given, every byte of page p in both pools
 * is zeroed (all KV heads).  new_tags[j] is the tag the new owner records as
 * its expected tag.
 *
 *   page_tags   uint32 [num_pages], updated in place
 *   pages       int32 [n]; list each page at most once per call (a repeated
 *               page still ends with its tag bumped once per listing, but
 *               which listing receives which new tag is unspecified)
 *   new_tags    uint32 [n] output; 0 for an id outside [0, num_pages), which
 *               is skipped and sets FKV_DEVERR_REALLOC_PAGE
 *   k_cache, v_cache  both NULL (no scrub) or the pools of this layer, of
 *               dtype kv_dtype with num_kv_heads, page_size, head_dim = 128
 * n == 0 is a no-op.
 */
FKV_API fkv_status kv_page_realloc(uint32_t *page_tags, int32_t num_pages,
                                   const int32_t *pages, int32_t n, uint32_t *new_tags,
                                   void *k_cache, void *v_cache, int32_t kv_dtype,
                                   int32_t num_kv_heads, int32_t page_size, int32_t head_dim,
                                   void *stream);

/*
 * paged_decode_attn_workspace_size -- bytes of device workspace that
 * paged_decode_attn needs for this shape on the current device (it depends on
 * the device's SM count).  Returns 0 for unsupported shapes.
 */
FKV_API size_t paged_decode_attn_workspace_size(int32_t batch, int32_t num_q_heads,
                                        int32_t num_kv_heads, int32_t head_dim,
                                        int32_t kv_dtype);

/*
 * paged_decode_attn -- decode-phase attention over the paged cache, values
 * converted from the cache format as they are read (Cloudflare post: the FP8
 * attention kernel converts values as it reads them).  For each request r and
 * query head i (kv head h = i / G):
 *     out[r][i] = sum_t softmax_t( sm_scale * q[r][i] . k_t ) v_t
 * over the request's seq_lens[r] tokens, with k_t = code * k_scale[h] and
 * v_t = code * v_scale[h] for FP8 (the bf16 values for BF16).
 *
 *   q              bf16 [batch][num_q_heads][head_dim]
 *   k_cache, v_cache  pools (layout above) of dtype kv_dtype (fkv_kv_dtype)
 *   k_scale, v_scale  fp32 [num_kv_heads] for FP8; ignored (may be NULL) for BF16
 *   page_indptr, page_indices  the CSR page table; nnz = length of page_indices
 *   seq_lens       int32 [batch]  tokens to attend per request
 *   abort_mask     uint8 [batch] from kv_page_tag_check, or NULL (no tracker)
 *   sm_scale       softmax scale, usually 1/sqrt(head_dim)
 *   out            bf16 [batch][num_q_heads][head_dim]
 *   workspace      device scratch of at least
 *                  paged_decode_attn_workspace_size(...) bytes, 256-byte
 *                  aligned; no initialisation needed; must not be shared by
 *                  calls that overlap on the GPU.
 * Fail closed: a request that is aborted, has a malformed CSR row (indptr[r]
 * < 0, indptr[r+1] < indptr[r] or indptr[r+1] > nnz), has seq_lens[r] <= 0,
 * has more tokens than its pages hold, or whose pages include an id outside
 * [0, num_pages), gets an all-zero output row, and no other row is affected.
 * The pages of the first four kinds are not read.  An id outside the pool is
 * never dereferenced: that tile is copied from page 0 instead, and the row is
 * written as zeros whatever those bytes hold (FKV_DEVERR_ATTN_PAGE is set).
 * Deterministic: the same call gives the same bytes every time (the split
 * over warps depends only on the live requests, and the merge of a split
 * (request, KV head) does not depend on which warp performs it or when).
 * Supported: head_dim 128, page_size in {16, 32, 64, 128}, group size
 * G = num_q_heads / num_kv_heads in 1..8, or above 8 when G splits into R
 * equal groups of at most 8 with R a power of two up to 8 (10, 12, 16, 24,
 * 32, 64, ...): each group is then served as a virtual KV head that reads
 * the KV head's pages again, so such a call reads R times the K/V bytes.
 * Other G return FKV_ERR_UNSUPPORTED.
 */
FKV_API fkv_status paged_decode_attn(const void *q, int32_t batch, int32_t num_q_heads,
                             const void *k_cache, const void *v_cache, int32_t kv_dtype,
                             const float *k_scale, const float *v_scale,
                             int32_t num_pages, int32_t num_kv_heads,
                             int32_t page_size, int32_t head_dim,
                             const int32_t *page_indptr, const int32_t *page_indices,
                             int64_t nnz, const int32_t *seq_lens, const uint8_t *abort_mask,
                             float sm_scale, void *out,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * paged_decode_attn_noalloc -- paged_decode_attn for callers that cannot
 * allocate device memory.  (The pages describe no such entry point; it has no
 * counterpart there.)
 *
 * Who needs it: code that has no allocator of its own -- a plugin inside a
 * host runtime that owns all device memory and passes the plugin only its
 * input and output buffers -- and serving loops that forbid cudaMalloc on the
 * hot path because it can synchronise the device and stall other streams.
 * Neither can hand paged_decode_attn its workspace.
 *
 * What it does: exactly paged_decode_attn (same arguments, same results,
 * same fail-closed rules) minus the workspace arguments.  Its scratch is one
 * fixed device array of FKV_NOALLOC_SCRATCH_BYTES compiled into the library;
 * every GPU that loads the library reserves that array until the process
 * exits.  The call itself allocates nothing (no cudaMalloc, no cudaFree, no
 * allocating library routine).
 *
 * Limits and rules:
 *   - A shape whose workspace (paged_decode_attn_workspace_size) exceeds
 *     FKV_NOALLOC_SCRATCH_BYTES is rejected with FKV_ERR_SCRATCH_LIMIT before
 *     anything is launched.  With 8 query heads per KV head, 16 MiB covers
 *     roughly batch * num_kv_heads up to 3000 on a 152-SM GB300.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.  The address is kept together with the id
 *     of the CUDA context it was found in.  When the context changes --
 *     cudaDeviceReset, or the primary context released and created again,
 *     which loads the library's device code anew -- the kept address is
 *     dropped and the next call looks it up again (so that call, too, is a
 *     first call and belongs outside stream capture).
 *   - All calls on a device share the one array and it keeps whatever the
 *     last call left in it (each call clears what it needs cleared).  Calls
 *     that overlap on the GPU -- on different streams, or from different host
 *     threads without ordering -- race on it and give wrong results; order
 *     them on one stream or serialise them.
 */
#define FKV_NOALLOC_SCRATCH_BYTES (16u << 20)
FKV_API fkv_status paged_decode_attn_noalloc(const void *q, int32_t batch, int32_t num_q_heads,
                                     const void *k_cache, const void *v_cache, int32_t kv_dtype,
                                     const float *k_scale, const float *v_scale,
                                     int32_t num_pages, int32_t num_kv_heads,
                                     int32_t page_size, int32_t head_dim,
                                     const int32_t *page_indptr, const int32_t *page_indices,
                                     int64_t nnz, const int32_t *seq_lens, const uint8_t *abort_mask,
                                     float sm_scale, void *out, void *stream);

/*
 * fkv_device_error -- read (and optionally clear) the sticky device error word
 * of the current device.  Synchronises the device.  *flags receives the OR of
 * FKV_DEVERR_* bits recorded since the last clear.
 */
FKV_API fkv_status fkv_device_error(uint32_t *flags, int32_t clear);

/* Number of kernels one call launches (for launch accounting). */
FKV_API int32_t fkv_kernels_per_call(const char *entry_point);

/*
 * fkv_selftest_wait -- run the failure path of the kernels' bounded waits
 * (diagnostic; the pages have no counterpart).  Every wait in the library's
 * kernels is on an mbarrier that a copy or another warp completes, and gives
 * up after a time limit, recording FKV_DEVERR_TIMEOUT instead of hanging.
 * This launches one block whose two warps run those two wait helpers (the
 * spinning and the sleeping one) on an mbarrier that nothing completes: each
 * gives up after limit_ns nanoseconds, sets FKV_DEVERR_TIMEOUT and the kernel
 * ends normally.  With complete != 0 the block completes the barrier first
 * and both waits return at once (no error bit).  result: NULL, or a device
 * uint32[2] receiving 1 (the wait saw the barrier complete) or 0 (it gave
 * up) per warp.  limit_ns above 10 s returns FKV_ERR_INVALID_ARG.
 * Asynchronous on `stream`; read the outcome with fkv_device_error.
 */
FKV_API fkv_status fkv_selftest_wait(uint64_t limit_ns, int32_t complete, uint32_t *result, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FKV_H_ */
