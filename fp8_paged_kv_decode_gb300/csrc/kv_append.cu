// kv_append.cu -- quantize-on-write of new tokens into the paged KV pools.
//
// Cloudflare post ("Smaller, faster, safer: running Kimi and GLM at scale", as
// extracted on the "Cloudflare Workers AI Optimizes Large Model Serving ..."
// page): the KV cache is stored as 8-bit floating point (FP8, e4m3) instead of
// BF16, which halves its size.  One fp32 scale per KV head (per layer) maps
// bf16 values into e4m3's range.
//
// Grid: x over groups of 16 tokens, y over KV heads, so no thread divides a
// 64-bit index.  16 threads serve one (token, head): 8 for its K row and 8
// for its V row, 16 elements each (two 16-byte bf16 loads, one 16-byte e4m3
// store).  The pool layout is [page][head][slot][128].  Per decode step the
// work is tiny (one token per request); for a bulk prefill write it is plain
// bandwidth, provided the arithmetic per element stays small -- hence the
// division below.
#include "tag_check_row.cuh"

namespace fkv {

constexpr int kHeadDim = 128;
constexpr int kElemsPerThread = 16;
constexpr int kThreadsPerRow = kHeadDim / kElemsPerThread;   // 8
constexpr int kThreadsPerToken = 2 * kThreadsPerRow;         // K and V: 16
constexpr int kBlock = 256;
constexpr int kTokensPerBlock = kBlock / kThreadsPerToken;   // 16

// Resident blocks per SM the FP8 kernel is compiled for: each thread keeps
// 32 bytes of loads in flight, so residency sets the bytes in flight per SM.
#ifndef FKV_APPEND_MIN_BLOCKS
#define FKV_APPEND_MIN_BLOCKS 8
#endif

// Division by the per-head scale, exactly as IEEE round-to-nearest fp32
// division, from its correctly rounded reciprocal y = RN(1/b) and one
// remainder correction (the correction step of Markstein's division,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", 1990):
//     q0 = RN(a*y),  r = RN(a - b*q0) (one fma),  q = RN(q0 + r*y) (one fma).
// The theorem's precondition (q0 within one ulp of a/b) does not hold for
// every operand pair, so the claim rests on an exhaustive check instead: for
// every bf16 significand of a and every fp32 significand of b, q equals the
// correctly rounded quotient.  Powers of two carry over exactly while every
// intermediate stays clear of underflow and overflow, which holds for
// 2^-30 <= b <= 2^30 and 2^-64 <= |a| <= 2^64 (q0, q within 2^+-94, r zero or
// at least 2^-111).  Below 2^-64, |a/b| < 2^-34 and both this and the exact
// quotient give a zero code; such inputs only need a finite, correctly signed
// result, which the sequence gives.  Anything else (a huge or non-finite a,
// a scale out of range) takes __fdiv_rn.  The sequence runs on |a|; the
// caller puts the sign back on the e4m3 code (sign-magnitude, and rounding
// to nearest even is symmetric), so -0 and tiny negatives keep their sign.
// The three steps run on two lanes at once with the packed two-lane fp32
// instructions (mul.rn.f32x2, fma.rn.f32x2), each lane rounding exactly as
// the scalar instruction does: 1.4 % faster on a bulk write than the scalar
// sequence.  word holds two bf16 elements (low half = lower element); they
// are widened to fp32 with their sign bits cleared.  nb = (-b, -b), yy = (y, y);
// the result is the two e4m3 codes of |word|, the lower element in the low byte.
__device__ __forceinline__ uint16_t div2_abs_to_e4m3x2(uint32_t word, uint64_t nb, uint64_t yy) {
    const uint32_t wm = word & 0x7FFF7FFFu;
    uint64_t m, q0, r, q;
    asm("mov.b64 %0, {%1, %2};" : "=l"(m) : "r"(wm << 16), "r"(wm & 0xFFFF0000u));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q0) : "l"(m), "l"(yy));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(q0), "l"(nb), "l"(m));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(r), "l"(yy), "l"(q0));
    uint32_t lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(q));
    return f32x2_to_e4m3x2(__uint_as_float(hi), __uint_as_float(lo));
}

// Lane-wise maximum of two pairs of unsigned 16-bit values.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ bool recip_scale_ok(float b) {
    return b >= 0x1p-30f && b <= 0x1p30f;     // false for NaN too
}

// Token of this thread in the block's 16-token group bx, or -1 past the end
// (no memory access: the row loads do not wait for the slot).
__device__ __forceinline__ int64_t token_of(int64_t n_tokens, unsigned bx) {
    const int64_t n = static_cast<int64_t>(bx) * kTokensPerBlock + (threadIdx.x / kThreadsPerToken);
    return n < n_tokens ? n : -1;
}

// Element offset of the (slot, KV head by) row in the pool, or -1: nothing
// to write (a padding slot, or one outside the pool, which is recorded).
__device__ __forceinline__ int64_t slot_offset(int64_t slot, int32_t num_pages, int32_t num_kv_heads,
                                               int32_t page_size, int32_t page_shift, uint32_t *err, unsigned by) {
    if (slot < 0) return -1;                                      // padding token
    const int64_t page = page_shift >= 0 ? (slot >> page_shift) : slot / page_size;
    const int64_t off = slot - page * page_size;
    if (page >= num_pages) {                                      // outside the pool: skip, record
        if ((threadIdx.x % kThreadsPerToken) == 0) atomicOr(err, FKV_DEVERR_APPEND_SLOT);
        return -1;
    }
    return ((page * num_kv_heads + by) * page_size + off) * kHeadDim;
}

// The e4m3 codes of one thread's 16 bf16 elements (two uint4 of the row, in
// order) divided by the scale b, as one uint4 (code k in byte k).
__device__ __forceinline__ uint4 encode16(const uint4 r0, const uint4 r1, float b) {
    const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    uint32_t big = 0;                                          // largest |x| bit patterns, per half
#pragma unroll
    for (int j = 0; j < 8; ++j) big = max_u16x2(big, w[j] & 0x7FFF7FFFu);
    // word j holds elements 2j (low half) and 2j+1; packed word p holds codes 4p .. 4p+3
    uint32_t packed[4];
    if (recip_scale_ok(b) && (big >> 16) <= 0x5F80u && (big & 0xFFFFu) <= 0x5F80u) {   // |x| <= 2^64
        const float y = __frcp_rn(b);
        uint64_t nb, yy;
        asm("mov.b64 %0, {%1, %1};" : "=l"(nb) : "r"(__float_as_uint(-b)));
        asm("mov.b64 %0, {%1, %1};" : "=l"(yy) : "r"(__float_as_uint(y)));
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint32_t u0 = w[2 * p], u1 = w[2 * p + 1];
            const uint16_t lo = div2_abs_to_e4m3x2(u0, nb, yy);
            const uint16_t hi = div2_abs_to_e4m3x2(u1, nb, yy);
            // the four elements' sign bits: bit 7 of each bf16's high byte
            const uint32_t sgn = prmt(u0, u1, 0x7531u) & 0x80808080u;
            packed[p] = (static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16)) | sgn;
        }
    } else {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint32_t u0 = w[2 * p], u1 = w[2 * p + 1];
            const uint16_t lo = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(u0 & 0xFFFF0000u), b),
                                                __fdiv_rn(__uint_as_float(u0 << 16), b));
            const uint16_t hi = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(u1 & 0xFFFF0000u), b),
                                                __fdiv_rn(__uint_as_float(u1 << 16), b));
            packed[p] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
        }
    }
    return make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

// One thread's share of the FP8 append in block (bx, by).
__device__ __forceinline__ void append_fp8_part(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                                const int64_t *__restrict__ slots, int64_t n_tokens,
                                                const float *__restrict__ k_scale, const float *__restrict__ v_scale,
                                                uint8_t *__restrict__ k_cache, uint8_t *__restrict__ v_cache,
                                                int32_t num_pages, int32_t num_kv_heads, int32_t page_size,
                                                int32_t page_shift, uint32_t *err, unsigned bx, unsigned by) {
    const int64_t n = token_of(n_tokens, bx);
    if (n < 0) return;
    const int h = by;
    const int sub = threadIdx.x % kThreadsPerToken;
    const bool is_v = sub >= kThreadsPerRow;
    const int chunk = sub % kThreadsPerRow;
    // 16 bf16 = two uint4 per thread; row (n, h) starts at uint4 index (n*Hkv + h) * 16
    const uint4 *src = (is_v ? v_new : k_new) + (n * num_kv_heads + h) * (kHeadDim / 8) + chunk * 2;
    // the row, its scale and its slot are independent loads, all in flight at
    // once (1.4 % faster on a bulk write than loading the row after the slot
    // has come back; placing the slot's use after the quotient instead, at
    // the store, measured 0.7 % slower than that).  Streaming hints on both
    // sides (the bf16 input is read once, the codes are not read back by this
    // kernel): 4.8 % faster on a bulk write than plain loads and stores, while
    // either hint alone is not
    const uint4 r0 = __ldcs(src), r1 = __ldcs(src + 1);
    const float b = __ldg((is_v ? v_scale : k_scale) + h);
    const int64_t slot = __ldg(slots + n);
    const int64_t dst_off = slot_offset(slot, num_pages, num_kv_heads, page_size, page_shift, err, by);
    if (dst_off < 0) return;
    uint8_t *dst = (is_v ? v_cache : k_cache) + dst_off + chunk * kElemsPerThread;
    __stcs(reinterpret_cast<uint4 *>(dst), encode16(r0, r1, b));
}

__global__ void __launch_bounds__(kBlock, FKV_APPEND_MIN_BLOCKS)
kv_append_fp8_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                     const int64_t *__restrict__ slots, int64_t n_tokens,
                     const float *__restrict__ k_scale, const float *__restrict__ v_scale,
                     uint8_t *__restrict__ k_cache, uint8_t *__restrict__ v_cache,
                     int32_t num_pages, int32_t num_kv_heads, int32_t page_size, int32_t page_shift,
                     uint32_t *err) {
    grid_dep_wait();        // earlier readers of the pool (attention) have finished
    grid_dep_launch();
    append_fp8_part(k_new, v_new, slots, n_tokens, k_scale, v_scale, k_cache, v_cache, num_pages, num_kv_heads,
                    page_size, page_shift, err, blockIdx.x, blockIdx.y);
}

// The decode step's append and the integrity check in one launch.  The two
// touch disjoint memory -- the append writes cache bytes only, the check
// reads tags and page tables and writes the abort mask -- so running them
// side by side gives exactly the bytes and the mask of kv_append_fp8
// followed by kv_page_tag_check, and the check still runs as its own pass
// before attention, outside the attention kernel.  Blocks [0, batch) check
// one request each; the rest are the append's (16-token group, KV head)
// blocks in x-major order.
__global__ void __launch_bounds__(kBlock, FKV_APPEND_MIN_BLOCKS)
kv_append_fp8_tag_check_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                               const int64_t *__restrict__ slots, int64_t n_tokens,
                               const float *__restrict__ k_scale, const float *__restrict__ v_scale,
                               uint8_t *__restrict__ k_cache, uint8_t *__restrict__ v_cache,
                               int32_t num_pages, int32_t num_kv_heads, int32_t page_size, int32_t page_shift,
                               uint32_t *err, unsigned append_blocks_x,
                               const uint32_t *__restrict__ page_tags, const int32_t *__restrict__ page_indptr,
                               const int32_t *__restrict__ page_indices, const uint32_t *__restrict__ expected_tags,
                               int32_t batch, int64_t nnz, uint8_t *__restrict__ abort_mask) {
    grid_dep_wait();        // earlier kernels' tags, tables and pool readers are done
    grid_dep_launch();
    const unsigned b = blockIdx.x;
    if (b < static_cast<unsigned>(batch)) {
        const int bad = tag_check_row<kBlock>(page_tags, num_pages, page_indptr, page_indices, expected_tags, nnz,
                                              static_cast<int>(b));
        if (threadIdx.x == 0) abort_mask[b] = bad ? 1 : 0;
        return;
    }
    const unsigned a = b - static_cast<unsigned>(batch);
    append_fp8_part(k_new, v_new, slots, n_tokens, k_scale, v_scale, k_cache, v_cache, num_pages, num_kv_heads,
                    page_size, page_shift, err, a % append_blocks_x, a / append_blocks_x);
}

// One thread's share of the BF16 append in block (bx, by): the row copied
// unchanged.
__device__ __forceinline__ void append_bf16_part(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                                 const int64_t *__restrict__ slots, int64_t n_tokens,
                                                 uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                                 int32_t num_pages, int32_t num_kv_heads, int32_t page_size,
                                                 int32_t page_shift, uint32_t *err, unsigned bx, unsigned by) {
    const int64_t n = token_of(n_tokens, bx);
    if (n < 0) return;
    const int h = by;
    const int sub = threadIdx.x % kThreadsPerToken;
    const bool is_v = sub >= kThreadsPerRow;
    const int chunk = sub % kThreadsPerRow;
    const uint4 *src = (is_v ? v_new : k_new) + (n * num_kv_heads + h) * (kHeadDim / 8) + chunk * 2;
    const uint4 r0 = __ldg(src), r1 = __ldg(src + 1);          // in flight with the slot's load
    const int64_t slot = __ldg(slots + n);
    const int64_t dst_off = slot_offset(slot, num_pages, num_kv_heads, page_size, page_shift, err, by);
    if (dst_off < 0) return;
    uint4 *dst = (is_v ? v_cache : k_cache) + dst_off / 8 + chunk * 2;
    dst[0] = r0;
    dst[1] = r1;
}

__global__ void __launch_bounds__(kBlock)
kv_append_bf16_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                      const int64_t *__restrict__ slots, int64_t n_tokens,
                      uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                      int32_t num_pages, int32_t num_kv_heads, int32_t page_size, int32_t page_shift,
                      uint32_t *err) {
    grid_dep_wait();        // earlier readers of the pool (attention) have finished
    grid_dep_launch();
    append_bf16_part(k_new, v_new, slots, n_tokens, k_cache, v_cache, num_pages, num_kv_heads, page_size,
                     page_shift, err, blockIdx.x, blockIdx.y);
}

// The BF16 cache's step prologue in one launch, laid out like
// kv_append_fp8_tag_check_kernel: check blocks first, then the append's.
__global__ void __launch_bounds__(kBlock)
kv_append_bf16_tag_check_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                const int64_t *__restrict__ slots, int64_t n_tokens,
                                uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                int32_t num_pages, int32_t num_kv_heads, int32_t page_size, int32_t page_shift,
                                uint32_t *err, unsigned append_blocks_x,
                                const uint32_t *__restrict__ page_tags, const int32_t *__restrict__ page_indptr,
                                const int32_t *__restrict__ page_indices,
                                const uint32_t *__restrict__ expected_tags, int32_t batch, int64_t nnz,
                                uint8_t *__restrict__ abort_mask) {
    grid_dep_wait();        // earlier kernels' tags, tables and pool readers are done
    grid_dep_launch();
    const unsigned b = blockIdx.x;
    if (b < static_cast<unsigned>(batch)) {
        const int bad = tag_check_row<kBlock>(page_tags, num_pages, page_indptr, page_indices, expected_tags, nnz,
                                              static_cast<int>(b));
        if (threadIdx.x == 0) abort_mask[b] = bad ? 1 : 0;
        return;
    }
    const unsigned a = b - static_cast<unsigned>(batch);
    append_bf16_part(k_new, v_new, slots, n_tokens, k_cache, v_cache, num_pages, num_kv_heads, page_size,
                     page_shift, err, a % append_blocks_x, a / append_blocks_x);
}

static fkv_status check_append_args(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                                    int32_t n_tokens, const void *k_cache, const void *v_cache,
                                    int32_t num_pages, int32_t num_kv_heads, int32_t page_size,
                                    int32_t head_dim) {
    if (n_tokens < 0 || num_pages <= 0 || num_kv_heads <= 0 || page_size <= 0) return FKV_ERR_INVALID_ARG;
    if (head_dim != kHeadDim) return FKV_ERR_UNSUPPORTED;
    if (num_kv_heads > 65535) return FKV_ERR_UNSUPPORTED;         // grid y
    if (n_tokens == 0) return FKV_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return FKV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return FKV_ERR_INVALID_ARG;
    return FKV_OK;
}

// log2(page_size) when it is a power of two, else -1 (the kernel divides).
static int32_t page_shift_of(int32_t page_size) {
    if (page_size & (page_size - 1)) return -1;
    int32_t s = 0;
    while ((1 << s) < page_size) ++s;
    return s;
}

static dim3 append_grid(int32_t n_tokens, int32_t num_kv_heads) {
    return dim3(static_cast<unsigned>((n_tokens + kTokensPerBlock - 1) / kTokensPerBlock),
                static_cast<unsigned>(num_kv_heads));
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
    const cudaError_t e = launch_pdl(kv_append_fp8_kernel, append_grid(n_tokens, num_kv_heads), dim3(kBlock), 0,
                                     static_cast<cudaStream_t>(stream), static_cast<const uint4 *>(k_new),
                                     static_cast<const uint4 *>(v_new), slot_mapping, static_cast<int64_t>(n_tokens),
                                     k_scale, v_scale, k_cache, v_cache, num_pages, num_kv_heads, page_size,
                                     page_shift_of(page_size), err);
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
    const cudaError_t e = launch_pdl(kv_append_bf16_kernel, append_grid(n_tokens, num_kv_heads), dim3(kBlock), 0,
                                     static_cast<cudaStream_t>(stream), static_cast<const uint4 *>(k_new),
                                     static_cast<const uint4 *>(v_new), slot_mapping, static_cast<int64_t>(n_tokens),
                                     static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), num_pages,
                                     num_kv_heads, page_size, page_shift_of(page_size), err);
    return e == cudaSuccess ? FKV_OK : FKV_ERR_CUDA;
}

// Argument checks of the one-launch append-and-check calls: those of the
// append, then those of kv_page_tag_check; the grid's block count.
static fkv_status check_combined_args(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                                      int32_t n_tokens, const void *k_cache, const void *v_cache,
                                      int32_t num_pages, int32_t num_kv_heads, int32_t page_size,
                                      int32_t head_dim, const uint32_t *page_tags, const int32_t *page_indptr,
                                      const int32_t *page_indices, const uint32_t *expected_tags, int32_t batch,
                                      int64_t nnz, uint8_t *abort_mask, int64_t &append_blocks_x,
                                      int64_t &blocks) {
    const fkv_status st = check_append_args(k_new, v_new, slot_mapping, n_tokens, k_cache, v_cache, num_pages,
                                            num_kv_heads, page_size, head_dim);
    if (st != FKV_OK) return st;
    if (batch < 0 || nnz < 0) return FKV_ERR_INVALID_ARG;
    if (batch > 0) {
        if (!page_indptr || !abort_mask || !page_tags) return FKV_ERR_INVALID_ARG;
        if (nnz > 0 && (!page_indices || !expected_tags)) return FKV_ERR_INVALID_ARG;
    }
    append_blocks_x = (static_cast<int64_t>(n_tokens) + kTokensPerBlock - 1) / kTokensPerBlock;
    blocks = append_blocks_x * num_kv_heads + batch;
    if (blocks > 0x7FFFFFFF) return FKV_ERR_UNSUPPORTED;
    return FKV_OK;
}

extern "C" fkv_status kv_append_fp8_tag_check(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                                              int32_t n_tokens, const float *k_scale, const float *v_scale,
                                              uint8_t *k_cache, uint8_t *v_cache, int32_t num_pages,
                                              int32_t num_kv_heads, int32_t page_size, int32_t head_dim,
                                              const uint32_t *page_tags, const int32_t *page_indptr,
                                              const int32_t *page_indices, const uint32_t *expected_tags,
                                              int32_t batch, int64_t nnz, uint8_t *abort_mask, void *stream) {
    int64_t gx = 0, blocks = 0;
    const fkv_status st = check_combined_args(k_new, v_new, slot_mapping, n_tokens, k_cache, v_cache, num_pages,
                                              num_kv_heads, page_size, head_dim, page_tags, page_indptr,
                                              page_indices, expected_tags, batch, nnz, abort_mask, gx, blocks);
    if (st != FKV_OK) return st;
    if (n_tokens > 0 && (!k_scale || !v_scale)) return FKV_ERR_INVALID_ARG;
    if (blocks == 0) return FKV_OK;
    uint32_t *err = device_error_word();
    if (!err) return FKV_ERR_CUDA;
    const cudaError_t e = launch_pdl(kv_append_fp8_tag_check_kernel, dim3(static_cast<unsigned>(blocks)),
                                     dim3(kBlock), 0, static_cast<cudaStream_t>(stream),
                                     static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new),
                                     slot_mapping, static_cast<int64_t>(n_tokens), k_scale, v_scale, k_cache,
                                     v_cache, num_pages, num_kv_heads, page_size, page_shift_of(page_size), err,
                                     static_cast<unsigned>(gx > 0 ? gx : 1), page_tags, page_indptr, page_indices,
                                     expected_tags, batch, nnz, abort_mask);
    return e == cudaSuccess ? FKV_OK : FKV_ERR_CUDA;
}

extern "C" fkv_status kv_append_bf16_tag_check(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                                               int32_t n_tokens, void *k_cache, void *v_cache, int32_t num_pages,
                                               int32_t num_kv_heads, int32_t page_size, int32_t head_dim,
                                               const uint32_t *page_tags, const int32_t *page_indptr,
                                               const int32_t *page_indices, const uint32_t *expected_tags,
                                               int32_t batch, int64_t nnz, uint8_t *abort_mask, void *stream) {
    int64_t gx = 0, blocks = 0;
    const fkv_status st = check_combined_args(k_new, v_new, slot_mapping, n_tokens, k_cache, v_cache, num_pages,
                                              num_kv_heads, page_size, head_dim, page_tags, page_indptr,
                                              page_indices, expected_tags, batch, nnz, abort_mask, gx, blocks);
    if (st != FKV_OK) return st;
    if (blocks == 0) return FKV_OK;
    uint32_t *err = device_error_word();
    if (!err) return FKV_ERR_CUDA;
    const cudaError_t e = launch_pdl(kv_append_bf16_tag_check_kernel, dim3(static_cast<unsigned>(blocks)),
                                     dim3(kBlock), 0, static_cast<cudaStream_t>(stream),
                                     static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new),
                                     slot_mapping, static_cast<int64_t>(n_tokens), static_cast<uint4 *>(k_cache),
                                     static_cast<uint4 *>(v_cache), num_pages, num_kv_heads, page_size,
                                     page_shift_of(page_size), err, static_cast<unsigned>(gx > 0 ? gx : 1),
                                     page_tags, page_indptr, page_indices, expected_tags, batch, nnz, abort_mask);
    return e == cudaSuccess ? FKV_OK : FKV_ERR_CUDA;
}
