// decode_attn.cu -- paged decode attention over an FP8 e4m3 (or BF16) cache.
//
// What is computed: for each request r and query head i (KV head h = i / G)
//     out[r][i] = sum_t softmax_t(sm_scale * q[r][i] . k_t) v_t
// over the request's tokens, gathered through its CSR page table, with K/V
// converted from the cache format as they are read.  The Cloudflare post
// ("Smaller, faster, safer: running Kimi and GLM at scale", extracted on the
// "Cloudflare Workers AI Optimizes Large Model Serving ..." page) stores the
// cache as FP8 e4m3 instead of BF16 and notes the FP8 attention kernel has to
// convert values as it reads them; requests aborted by the separate integrity
// check are not read (fail closed).
//
// GB300 design (two launches, chained with programmatic dependent launch):
//  1. plan (one CTA): tiles per request from seq_lens / abort mask / page
//     table; prefix over requests; the first request of each computing warp;
//     zeroed arrival counters.  A "tile" is kTile tokens of one
//     (request, KV head) unit.
//  2. attention (persistent, one computing warp per CTA, grid = SMs x
//     resident CTAs): the concatenation of all units' tiles is cut into equal
//     contiguous ranges, one per computing warp (split-KV with even load
//     across the lognormal context mix); a small batch instead gives each
//     unit whole warps of its own (the kernel instance for batches of up to
//     64 requests, whose warps test the live requests' tiles and fall back
//     to the even split).  For batches of up to 128
//     requests each warp finds its own range from the inputs and starts its
//     copies before the plan kernel has finished.  Each warp streams its tiles
//     through a private ring of shared-memory stages filled by 128B-swizzled
//     TMA tensor copies (one box per page: the K and V tiles of a (page, head)
//     are contiguous in HBM); when a tile spans several small pages a second,
//     producer warp issues the copies.  QK^T and PV run on the tensor cores as
//     m16n8k16 MMAs with tokens on M and the G <= 8 query heads of the KV head
//     on N; e4m3 codes become f16 exactly in registers (the per-head scales
//     fold into the logit factor and the output); softmax is online in fp32
//     with warp shuffles.  A warp that covers a whole unit writes the bf16
//     output directly; otherwise it writes an unnormalised fp32 partial
//     (o, m, l), and the last of the unit's warps to arrive (an atomic
//     counter, no waiting) merges the partials with a log-sum-exp rescale
//     (two levels for units split over many warps), fetching them with 1-D
//     bulk copies into its idle stage ring at the end of its range.  The
//     merge's arithmetic is fixed (merge_parts_smem), so the bytes of a row
//     do not depend on which warp merges it or when.  Rows of requests with
//     no tiles (aborted, empty, malformed) are zero-filled by the warps, one
//     request each.
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "fkv_common.cuh"

// Tokens per pipeline stage and ring depth of each KV dtype.
#ifndef FKV_FP8_TILE
#define FKV_FP8_TILE 64
#endif
#ifndef FKV_FP8_STAGES
#define FKV_FP8_STAGES 3
#endif
#ifndef FKV_BF16_TILE
#define FKV_BF16_TILE 64
#endif
#ifndef FKV_BF16_STAGES
#define FKV_BF16_STAGES 2
#endif
// How the producer warp waits for a stage to be released.
#ifndef FKV_PRODUCER_WAIT
#define FKV_PRODUCER_WAIT mbar_wait_bounded_sleep
#endif
// L2 hint of the K/V tile copies (streamed once unless pages are shared).
#ifndef FKV_KV_EVICT_FIRST
#define FKV_KV_EVICT_FIRST 1
#endif

namespace fkv {

constexpr int kD = 128;
constexpr int kMaxGroup = 8;             // query heads of one unit (MMA N)
constexpr int kMaxSplit = 8;             // virtual KV heads per KV head (group sizes up to 64)
constexpr int kPlanThreads = 1024;
constexpr int kPlanSmemPrefix = 4096;    // requests whose prefix the plan searches in smem
constexpr uint64_t kWaitLimitNs = 2000000000ull;     // a copy that has not landed in 2 s has failed
constexpr uint64_t kDrainLimitNs = 200000000ull;
constexpr uint32_t kFull = 0xffffffffu;
#ifndef FKV_MERGE_CHUNK
#define FKV_MERGE_CHUNK 9
#endif
// Small batches may give each (request, KV head) unit whole warps (1) instead
// of an even split of the batch's tiles (0); ranges then hold at least
// FKV_ALIGNED_MIN_TILES tiles.
#ifndef FKV_ALIGNED_SCHEDULE
#define FKV_ALIGNED_SCHEDULE 1
#endif
#ifndef FKV_ALIGNED_MIN_TILES
#define FKV_ALIGNED_MIN_TILES 2
#endif
#ifndef FKV_MIN_TILES_PER_WARP
#define FKV_MIN_TILES_PER_WARP 12
#endif
constexpr int kNone = 0, kFinalDue = 1, kChunkDue = 2;   // merge duties of a warp
constexpr int kChunk = FKV_MERGE_CHUNK;  // parts merged per first-level merge of a long unit
constexpr int kMinTilesPerWarp = FKV_MIN_TILES_PER_WARP;   // small batches use fewer, longer warp ranges
constexpr int kMinAlignedTiles = FKV_ALIGNED_MIN_TILES;
// Batches of up to this many requests are scheduled by the attention warps
// from the inputs (at most 1024: one 32-request chunk per lane).  Past ~128
// every warp reading all the requests' rows costs more than waiting for the
// plan kernel's table (at 1024 requests of 256 tokens: 133 vs 122 us).
#ifndef FKV_LOCAL_PLAN_MAX
#define FKV_LOCAL_PLAN_MAX 128
#endif
// At the end of its range a warp holding the first part of a unit of at most
// three parts, whose other parts have all arrived, merges from its registers
// (1) instead of publishing its part and arriving (0).
#ifndef FKV_TRY_LAST
#define FKV_TRY_LAST 1
#endif
constexpr int kLocalPlanMax = FKV_LOCAL_PLAN_MAX;
static_assert(kLocalPlanMax <= 1024, "one 32-request chunk per lane");
// Attention CTA: one warp that both issues copies and computes, or (kWS) a
// producer warp that issues copies and a consumer warp that computes.
__host__ __device__ constexpr int attn_threads(bool ws) { return ws ? 64 : 32; }      // batches up to this size: each warp finds its own range

template <bool kFp8>
struct Cfg;
template <>
struct Cfg<true> {
    static constexpr int kTile = FKV_FP8_TILE;
    static constexpr int kStages = FKV_FP8_STAGES;
    static constexpr int kHalves = 1;           // 128-byte-wide column blocks per token row
};
template <>
struct Cfg<false> {
    static constexpr int kTile = FKV_BF16_TILE;
    static constexpr int kStages = FKV_BF16_STAGES;
    static constexpr int kHalves = 2;
};

template <bool kFp8>
struct Layout {
    static constexpr int kTile = Cfg<kFp8>::kTile;
    static constexpr int kStages = Cfg<kFp8>::kStages;
    static constexpr int kHalves = Cfg<kFp8>::kHalves;
    static constexpr int kHalfBytes = kTile * 128;              // one column block of a K (or V) tile
    static constexpr int kTileBytes = kHalves * kHalfBytes;     // a K (or V) tile
    static constexpr int kStageBytes = 2 * kTileBytes;          // K then V
    // stage buffers, then per stage a full and an empty mbarrier, the merge
    // mbarrier, and per stage a bad-page flag
    static constexpr int kSmem = 1024 + kStages * kStageBytes + 20 * kStages + 8;
    static_assert(kTile == 32 || kTile == 64, "tile of 32 or 64 tokens");
    static_assert(kHalfBytes % 1024 == 0, "stage buffers stay 1024-byte aligned for the 128B swizzle");
};

struct AttnParams {
    const __nv_bfloat16 *q;
    const float *k_scale;
    const float *v_scale;
    const int32_t *indptr;
    const int32_t *indices;
    const int32_t *seq_lens;
    const uint8_t *abort_mask; // nullptr: no request aborted
    int64_t nnz;               // entries of page_indices
    const int64_t *prefix;     // [B+1] tile prefix over requests (tiles x Hkv)
    const int32_t *warp_req;   // [NW + 1] request holding each warp's first tile; [NW] = warps with work
    float *part_o;             // [slots][G][D]   slots = B*Hkv + NW
    float2 *part_ml;           // [slots][GP] (m in log2 units, l; l < 0 marks an invalid unit)
    int32_t *counters;         // [B*Hkv] arrivals per split unit (or per chunk of it)
    int32_t *chunk_counters;   // [slots] arrivals per first-level chunk, indexed by its first slot
    __nv_bfloat16 *out;
    uint32_t *err;
    // Hkv, G: units per request and query heads per unit.  With more than
    // kMaxGroup query heads per KV head each KV head is served as 2^hshift
    // virtual heads of G query heads (consecutive query rows) that read the
    // same pages: unit head h reads KV head h >> hshift.
    int B, Hq, Hkv, G, GP, P, S, NW;   // GP = G rounded up to even: 16-byte statistics rows
    int hshift;
    float sm_scale_log2;
};

// ---------------------------------------------------------------------------
// 1. plan
// ---------------------------------------------------------------------------
// Tiles of request r over all its KV heads; 0 if it is aborted, empty or has a
// malformed page-table row (indptr out of order or past nnz, or fewer pages
// than its length needs).  The plan kernel and the attention warps' own
// schedule both count with this, so their prefixes agree exactly.  Loads go
// to L2 (the inputs may have been written by the kernels just before).
struct RequestInfo {
    int64_t tiles;        // over all KV heads
    int32_t seq_len, row; // length and first page-table entry
};

__device__ __forceinline__ RequestInfo request_info(const int32_t *seq_lens, const int32_t *indptr,
                                                   const uint8_t *abort_mask, int64_t nnz, int r, int Hkv, int S,
                                                   int tile) {
    const int32_t sl = __ldcg(seq_lens + r);
    const int32_t b = __ldcg(indptr + r), e = __ldcg(indptr + r + 1);
    const bool alive = abort_mask == nullptr || __ldcg(abort_mask + r) == 0;
    RequestInfo ri{0, sl, b};
    if (alive && sl > 0 && b >= 0 && e >= b && e <= nnz && static_cast<int64_t>(e - b) * S >= sl)
        ri.tiles = ((static_cast<int64_t>(sl) + tile - 1) / tile) * Hkv;
    return ri;
}

__device__ __forceinline__ int64_t request_tiles(const int32_t *seq_lens, const int32_t *indptr,
                                                 const uint8_t *abort_mask, int64_t nnz, int r, int Hkv, int S,
                                                 int tile) {
    return request_info(seq_lens, indptr, abort_mask, nnz, r, Hkv, S, tile).tiles;
}

// Warps that get work: every one streams at least kMinTilesPerWarp tiles, so a
// small batch is not split into ranges too short to pay for their start-up
// and merge (large batches use all NW).
__device__ __forceinline__ int working_warps(int64_t T, int NW) {
    const int64_t nw64 = (T + kMinTilesPerWarp - 1) / kMinTilesPerWarp;
    return static_cast<int>(nw64 < 1 ? 1 : (nw64 > NW ? NW : nw64));
}

__global__ void __launch_bounds__(kPlanThreads)
attn_plan_kernel(const int32_t *__restrict__ seq_lens, const int32_t *__restrict__ indptr,
                 const uint8_t *__restrict__ abort_mask, int64_t nnz, int B, int Hkv, int S, int tile, int NW,
                 int64_t *__restrict__ prefix, int32_t *__restrict__ warp_req, int32_t *__restrict__ counters) {
    grid_dep_wait();                   // the abort mask of the integrity check is complete
    grid_dep_launch();                 // let the attention grid start its prologue
    __shared__ int64_t s_warp_tot[kPlanThreads / 32];
    __shared__ int64_t s_prefix[kPlanSmemPrefix + 1];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    // arrival counters: one per unit, then one per partial slot (chunks)
    for (int64_t u = tid; u < 2 * static_cast<int64_t>(B) * Hkv + NW; u += kPlanThreads) counters[u] = 0;
    int64_t carry = 0;
    for (int base = 0; base < B; base += kPlanThreads) {
        const int r = base + tid;
        const int64_t cnt = r < B ? request_tiles(seq_lens, indptr, abort_mask, nnz, r, Hkv, S, tile) : 0;
        int64_t x = cnt;                                   // inclusive warp scan
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_warp_tot[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int64_t v = s_warp_tot[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t y = __shfl_up_sync(kFull, v, o);
                if (lane >= o) v += y;
            }
            s_warp_tot[lane] = v;                           // inclusive over warps
        }
        __syncthreads();
        const int64_t excl = carry + (wid ? s_warp_tot[wid - 1] : 0) + x - cnt;
        if (r < B) {
            prefix[r] = excl;
            if (r < kPlanSmemPrefix) s_prefix[r] = excl;
        }
        carry += s_warp_tot[31];
        __syncthreads();
    }
    if (tid == 0) {
        prefix[B] = carry;
        if (B <= kPlanSmemPrefix) s_prefix[B] = carry;
    }
    __syncthreads();
    const int64_t T = carry;
    const bool in_smem = B <= kPlanSmemPrefix;
    const int nw = working_warps(T, NW);
    if (tid == 0) warp_req[NW] = nw;
    for (int w = tid; w < nw; w += kPlanThreads) {
        const int64_t lo = static_cast<int64_t>(w) * T / nw;
        int res = B;
        if (lo < T) {
            int a = 0, z = B;                              // invariant: prefix[a] <= lo < prefix[z]
            while (z - a > 1) {
                const int mid = (a + z) >> 1;
                const int64_t pm = in_smem ? s_prefix[mid] : prefix[mid];
                if (pm <= lo) a = mid; else z = mid;
            }
            res = a;
        }
        warp_req[w] = res;
    }
}

// ---------------------------------------------------------------------------
// 2. split attention with fused merge
// ---------------------------------------------------------------------------
struct Cursor {
    int r, h, tt, nt;
};

__device__ __forceinline__ void cursor_init(Cursor &c, const AttnParams &p, int64_t x, int r) {
    while (r < p.B - 1 && p.prefix[r + 1] <= x) ++r;
    const int64_t base = p.prefix[r];
    const int nt = static_cast<int>((p.prefix[r + 1] - base) / p.Hkv);
    const int64_t rel = x - base;
    c.r = r;
    c.nt = nt;
    c.h = static_cast<int>(rel / nt);
    c.tt = static_cast<int>(rel - static_cast<int64_t>(c.h) * nt);
}

__device__ __forceinline__ void cursor_next(Cursor &c, const AttnParams &p) {
    if (++c.tt < c.nt) return;
    c.tt = 0;
    if (++c.h < p.Hkv) return;
    c.h = 0;
    int r = c.r + 1;
    while (r < p.B && p.prefix[r + 1] == p.prefix[r]) ++r;      // requests with no tiles
    c.r = r;
    c.nt = r < p.B ? static_cast<int>((p.prefix[r + 1] - p.prefix[r]) / p.Hkv) : 0;
}

// cursor at tile x of request r, whose tiles start at `base` (nt per KV head)
__device__ __forceinline__ void cursor_at(Cursor &c, int r, int64_t base, int nt, int64_t x) {
    const int64_t rel = x - base;
    c.r = r;
    c.nt = nt;
    c.h = static_cast<int>(rel / nt);
    c.tt = static_cast<int>(rel - static_cast<int64_t>(c.h) * nt);
}

// Total tiles of a batch of up to 1024 requests, computed by one warp from
// the inputs (the same sum the plan kernel forms), reading the requests 32 at
// a time with several chunks' loads in flight; lane c keeps in `mine` the
// tiles of chunk c (requests 32c .. 32c + 31).
__device__ __forceinline__ int64_t batch_tiles(const AttnParams &p, int tile, int64_t &mine) {
    const int lane = threadIdx.x & 31;
    const int nch = (p.B + 31) / 32;
    int64_t sum = 0;
    mine = 0;
#pragma unroll 4
    for (int c = 0; c < nch; ++c) {
        const int r = 32 * c + lane;
        int64_t t = r < p.B ? request_tiles(p.seq_lens, p.indptr, p.abort_mask, p.nnz, r, p.Hkv, p.S, tile) : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(kFull, t, o);
        if (lane == c) mine = t;
        sum += t;
    }
    return sum;
}

// Where the warp's first tile lies: the request r0 holding tile x (prefix[r0]
// <= x < prefix[r0 + 1], as the plan kernel's search finds it), its first
// tile, tiles per KV head, length and first page-table entry.
struct FirstRequest {
    int r0 = -1, nt0 = 0, sl0 = 0, row0 = 0;
    int64_t base0 = 0;
};

// One step of the search: the 32 requests b .. b + 31 (this lane's is ri),
// `carry` tiles before them.  Returns the tiles of these 32 requests.
__device__ __forceinline__ int64_t scan_requests(const RequestInfo &ri, int b, int64_t carry, int64_t x, int Hkv,
                                                 FirstRequest &fr) {
    const int lane = threadIdx.x & 31;
    const int64_t cnt = ri.tiles;
    int64_t inc = cnt;                                     // inclusive scan over the 32 requests
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += y;
    }
    const int64_t excl = carry + inc - cnt;
    const unsigned hit = __ballot_sync(kFull, cnt > 0 && excl <= x && x < excl + cnt);
    if (hit) {
        const int src = __ffs(hit) - 1;
        fr.r0 = b + src;
        fr.base0 = __shfl_sync(kFull, excl, src);
        fr.nt0 = static_cast<int>(__shfl_sync(kFull, cnt, src) / Hkv);
        fr.sl0 = __shfl_sync(kFull, ri.seq_len, src);
        fr.row0 = __shfl_sync(kFull, ri.row, src);
    }
    return __shfl_sync(kFull, inc, 31);
}

// Where the parts of a split unit sit: its first warp and how many warps it
// spans.  A unit over more than kChunk warps merges in chunks of kChunk
// consecutive parts; c0 is the first part of warp w's chunk.
struct UnitGeom {
    int wf, span;
    __device__ int c0(int w) const { return ((w - wf) / kChunk) * kChunk; }
    __device__ int csz(int w) const { return min(kChunk, span - c0(w)); }
    __device__ int nch() const { return (span + kChunk - 1) / kChunk; }
};

// Schedule of a small batch (up to 64 requests, each lane holding two
// requests' rows): every unit (request, KV head) gets whole warps, k_r =
// ceil(n_r / tpw) of them for a request of n_r tiles per head, each holding an
// even share of the unit's tiles.  No range then crosses a unit boundary and
// every merge runs at a range end.  tpw is the smallest count (at least
// kMinAlignedTiles) with which the warps fit: with U live units (requests
// with tiles, times Hkv), sum over units of ceil(n_u / tpw) < T / tpw + U <=
// NW once tpw >= T / (NW - U).  It is used only when tpw is below
// kMinTilesPerWarp, where the even split of the batch's tiles would leave
// warps idle; otherwise this returns false.  Both the test and tpw depend on
// the live requests only, so an aborted request changes nothing for the
// others.  Past the test every count fits in 32 bits.  Warp w
// gets tiles [lo, hi) (empty past the last unit's warps), the request holding
// them, and its unit's warps.
template <int kTile>
__device__ __forceinline__ bool place_aligned(const RequestInfo (&rc)[2], int64_t T, int NW, int Hkv, int w,
                                              int64_t &lo, int64_t &hi, FirstRequest &fr, UnitGeom &gm) {
    const int lane = threadIdx.x & 31;
    int live = (rc[0].tiles > 0) + (rc[1].tiles > 0);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) live += __shfl_xor_sync(kFull, live, o);
    const int room = NW - live * Hkv;
    if (room <= 0 || T > static_cast<int64_t>(kMinTilesPerWarp - 1) * room) return false;
    const int tpw = max(kMinAlignedTiles, (static_cast<int>(T) + room - 1) / room);
    lo = hi = 0;
    int wcarry = 0, tcarry = 0;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int n = rc[c].tiles > 0 ? (rc[c].seq_len + kTile - 1) / kTile : 0;   // tiles per KV head
        const int k = (n + tpw - 1) / tpw;                 // warps per KV head
        const int K = k * Hkv, cnt = n * Hkv;
        int kin = K, tin = cnt;                            // inclusive scans over the 32 requests
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, kin, o), z = __shfl_up_sync(kFull, tin, o);
            if (lane >= o) {
                kin += y;
                tin += z;
            }
        }
        const int wex = wcarry + kin - K;                  // this request's first warp
        const int tex = tcarry + tin - cnt;                // and first tile
        const unsigned hit = __ballot_sync(kFull, K > 0 && wex <= w && w < wex + K);
        if (hit) {
            const int src = __ffs(hit) - 1;
            const int wr = __shfl_sync(kFull, wex, src), kk = __shfl_sync(kFull, k, src);
            const int nn = __shfl_sync(kFull, n, src), base = __shfl_sync(kFull, tex, src);
            const int rel = w - wr, h = rel / kk, j = rel - h * kk;
            const int s0 = base + h * nn;
            lo = s0 + j * nn / kk;
            hi = s0 + (j + 1) * nn / kk;
            fr.r0 = 32 * c + src;
            fr.base0 = base;
            fr.nt0 = nn;
            fr.sl0 = __shfl_sync(kFull, rc[c].seq_len, src);
            fr.row0 = __shfl_sync(kFull, rc[c].row, src);
            gm.wf = wr + h * kk;
            gm.span = kk;
        }
        wcarry += __shfl_sync(kFull, kin, 31);
        tcarry += __shfl_sync(kFull, tin, 31);
    }
    return true;
}

// The same search for up to 1024 requests: the chunk holding tile x comes
// from the per-chunk totals batch_tiles left (`mine`), then that chunk's rows
// are read again and scanned.
__device__ __forceinline__ FirstRequest find_request(const AttnParams &p, int tile, int64_t x, int64_t mine) {
    const int lane = threadIdx.x & 31;
    int64_t incl = mine;                                   // inclusive scan over the chunks
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    const unsigned hit = __ballot_sync(kFull, mine > 0 && incl - mine <= x && x < incl);
    FirstRequest fr;
    if (hit) {
        const int c = __ffs(hit) - 1;
        const int64_t carry = __shfl_sync(kFull, incl - mine, c);
        const int r = 32 * c + lane;
        RequestInfo ri{0, 0, 0};
        if (r < p.B) ri = request_info(p.seq_lens, p.indptr, p.abort_mask, p.nnz, r, p.Hkv, p.S, tile);
        scan_requests(ri, 32 * c, carry, x, p.Hkv, fr);
    }
    return fr;
}

__device__ __forceinline__ uint32_t lo16(uint32_t x) { return x & 0xFFFFu; }
__device__ __forceinline__ uint32_t hi16(uint32_t x) { return x >> 16; }

// first tile of warp w's range
__device__ __forceinline__ int64_t warp_lo(int64_t w, int64_t T, int NW) { return w * T / NW; }

// the warp w with floor(w*T/NW) <= x < floor((w+1)*T/NW)
__device__ __forceinline__ int64_t warp_of_tile(int64_t x, int64_t T, int NW) {
    const int64_t w = ((x + 1) * NW + T - 1) / T - 1;
    return w < NW - 1 ? w : NW - 1;
}

// Merge n partials stored at slots slot0, slot0 + stride, ... into either the
// final bf16 rows of unit (r, h) (scaled by vsc / L) or one fp32 partial
// written to slot `dst` (the first level of a two-level merge), for a warp
// whose stage ring is idle (the end of its range).  With `maybe_empty`
// (tiles < warps) entries of warps with an empty range, which wrote nothing,
// are skipped; entry j belongs to warp wk0 + j.  Each entry arrives in two
// bulk copies (outputs, statistics) issued by the lane that owns it, all
// completing on `bar`, so a batch of up to `cap` (<= 32) entries costs one
// memory round trip.  The statistics are reduced across lanes (one entry per
// lane); each entry's weights go to shared memory and the output pass reads
// them back as broadcasts beside the entry's rows.  Longer lists go in batches
// with a running rescale.  The caller has acquired every entry (an
// acquire-release arrival after the writers' own); the proxy fence carries
// that to the bulk copies.  Returns false if a batch's copies did not land in
// time; nothing is written then.
//
// The arithmetic of one batch is the merge's definition, which the register
// merge at a range end reproduces exactly (merge_regs): with the live entries
// packed in index order at lanes 0, 1, ..., per head
//     M = max_e m_e,   w_e = 2^(m_e - M),
//     L = the xor-butterfly sum over the 32 lanes of RN(w_e l_e) (0 past the entries),
//     acc = fma(w_{n-1}, o_{n-1}, ... fma(w_1, o_1, fma(w_0, o_0, 0))),
//     row = bf16(RN(acc RN(vsc / L))), or zeros if any entry is marked bad,
// every rounding explicit (_rn operations, nothing left to contraction), so
// a row's bytes do not depend on which warp merges it, on which of the two
// paths it takes, or on when the parts arrive.
__device__ bool merge_parts_smem(const AttnParams &p, uint32_t sbuf, int cap, uint32_t bar, uint32_t &phase, int nw,
                                 int64_t slot0, int n, int stride, bool maybe_empty, int64_t wk0, int64_t T,
                                 bool final_out, int r, int h, float vsc, int64_t dst) {
    const int lane = threadIdx.x & 31;
    const int G = p.G, GP = p.GP;
    const uint32_t obytes = static_cast<uint32_t>(G) * kD * 4;     // one entry's outputs
    const uint32_t mbytes = static_cast<uint32_t>(GP) * 8;         // one entry's statistics
    const uint32_t mbase = sbuf + static_cast<uint32_t>(cap) * obytes;
    const uint32_t wbase = mbase + static_cast<uint32_t>(cap) * mbytes;   // 8 weights per entry
    float M[kMaxGroup], L[kMaxGroup];
    float4 acc[kMaxGroup];
#pragma unroll
    for (int hd = 0; hd < kMaxGroup; ++hd) {
        M[hd] = -INFINITY;
        L[hd] = 0.f;
        acc[hd] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    bool bad = false;
    for (int b0 = 0; b0 < n; b0 += cap) {
        const int nb = min(cap, n - b0);
        const int j = b0 + lane;
        const bool live = lane < nb && !(maybe_empty && warp_lo(wk0 + j, T, nw) == warp_lo(wk0 + j + 1, T, nw));
        const uint32_t lmask = __ballot_sync(kFull, live);
        const int nv = __popc(lmask);
        if (nv == 0) continue;
        const uint32_t pos = __popc(lmask & ((1u << lane) - 1u));   // live entries are packed, in order
        if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nv) * (obytes + mbytes));
        __syncwarp();
        if (live) {
            const int64_t slot = slot0 + static_cast<int64_t>(j) * stride;
            fence_proxy_async_global();
            bulk_load(sbuf + pos * obytes, p.part_o + slot * G * kD, obytes, bar);
            bulk_load(mbase + pos * mbytes, p.part_ml + slot * GP, mbytes, bar);
        }
        if (!mbar_wait_bounded(bar, phase, kWaitLimitNs)) {
            (void)mbar_wait_bounded(bar, phase, kDrainLimitNs);   // let copies in flight land
            return false;
        }
        phase ^= 1u;
        // statistics: lane e holds entry e
        float mv[kMaxGroup], lv[kMaxGroup], wv[kMaxGroup];
#pragma unroll
        for (int hd = 0; hd < kMaxGroup; ++hd) {
            mv[hd] = -INFINITY;
            lv[hd] = 0.f;
            wv[hd] = 0.f;
            if (hd < G && lane < nv) {
                const float2 ml = ld_shared_f2(mbase + lane * mbytes + hd * 8);
                mv[hd] = ml.x;
                lv[hd] = ml.y;
                bad |= ml.y < 0.f;
            }
        }
        // all kMaxGroup heads, so the shuffle chains interleave (heads >= G
        // carry m = -inf and weight 0 throughout)
#pragma unroll
        for (int hd = 0; hd < kMaxGroup; ++hd) {
            float mb = mv[hd];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, o));
            mb = fmaxf(mb, M[hd]);
            const float f = M[hd] == -INFINITY ? 0.f : ex2(M[hd] - mb);
            wv[hd] = mv[hd] == -INFINITY ? 0.f : ex2(mv[hd] - mb);
            float sl = __fmul_rn(wv[hd], lv[hd]);
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) sl = __fadd_rn(sl, __shfl_xor_sync(kFull, sl, o));
            L[hd] = __fmaf_rn(L[hd], f, sl);
            acc[hd].x = __fmul_rn(acc[hd].x, f);
            acc[hd].y = __fmul_rn(acc[hd].y, f);
            acc[hd].z = __fmul_rn(acc[hd].z, f);
            acc[hd].w = __fmul_rn(acc[hd].w, f);
            M[hd] = mb;
        }
        if (lane < nv) {
            st_shared_f4(wbase + lane * 32, make_float4(wv[0], wv[1], wv[2], wv[3]));
            st_shared_f4(wbase + lane * 32 + 16, make_float4(wv[4], wv[5], wv[6], wv[7]));
        }
        __syncwarp();
        // outputs: 4 dims of every head per lane
        for (int e = 0; e < nv; ++e) {
            const float4 w0 = ld_shared_f4(wbase + e * 32), w1 = ld_shared_f4(wbase + e * 32 + 16);
            const float wgt[kMaxGroup] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int hd = 0; hd < kMaxGroup; ++hd) {
                if (hd < G) {
                    const float4 v = ld_shared_f4(sbuf + e * obytes + hd * (kD * 4) + lane * 16);
                    acc[hd].x = __fmaf_rn(wgt[hd], v.x, acc[hd].x);
                    acc[hd].y = __fmaf_rn(wgt[hd], v.y, acc[hd].y);
                    acc[hd].z = __fmaf_rn(wgt[hd], v.z, acc[hd].z);
                    acc[hd].w = __fmaf_rn(wgt[hd], v.w, acc[hd].w);
                }
            }
        }
        __syncwarp();                                      // the next batch reuses the buffer
    }
    bad = __any_sync(kFull, bad);
    if (final_out) {
#pragma unroll
        for (int hd = 0; hd < kMaxGroup; ++hd) {
            if (hd >= G) break;
            const float sc = __fdiv_rn(vsc, L[hd]);
            uint2 *orow =
                reinterpret_cast<uint2 *>(p.out + (static_cast<int64_t>(r) * p.Hq + h * G + hd) * kD) + lane;
            *orow = bad ? make_uint2(0u, 0u)
                        : make_uint2(pack_bf16x2(__fmul_rn(acc[hd].x, sc), __fmul_rn(acc[hd].y, sc)),
                                     pack_bf16x2(__fmul_rn(acc[hd].z, sc), __fmul_rn(acc[hd].w, sc)));
        }
    } else {
#pragma unroll
        for (int hd = 0; hd < kMaxGroup; ++hd) {
            if (hd >= G) break;
            __stcg(reinterpret_cast<float4 *>(p.part_o + (dst * G + hd) * kD) + lane, acc[hd]);
        }
#pragma unroll
        for (int hd = 0; hd < kMaxGroup; ++hd)
            if (hd < G && lane == hd) __stcg(p.part_ml + dst * GP + hd, make_float2(M[hd], bad ? -1.f : L[hd]));
    }
    return true;
}

// kAligned: the instance for batches of up to 64 requests, which gives units
// whole warps (place_aligned) when the live requests' tiles pass its test and
// uses the even split otherwise.  Larger batches use the instance without
// the option (their warps do not hold the requests' rows).
template <bool kFp8, bool kWS, bool kAligned>
__global__ void __launch_bounds__(attn_threads(kWS), 1)
paged_decode_attn_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV) {
    using Lay = Layout<kFp8>;
    constexpr int kTile = Lay::kTile;
    constexpr int NST = Lay::kStages;
    constexpr int MT = kTile / 16;                       // 16-token MMA tiles per stage
    constexpr int NACC = MT >= 4 ? 1 : 2;                // independent QK accumulator chains per M tile

    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    // Stage s completes on full[s] when its copies land.  With kWS the CTA has
    // two warps: warp 0 issues the K/V copies (the producer) and warp 1
    // computes (the consumer), which releases a stage on empty[s].  A tensor
    // copy takes ~80 ns to issue, so moving the issue off the computing warp
    // pays when a 64-token tile spans several small pages (2 to 8 copies per
    // stage); with one page per tile (2 copies) the single warp, refilling a
    // stage right after it is consumed, is ~2 % faster.
    const uint32_t full_bars = sbase + NST * Lay::kStageBytes;
    const uint32_t empty_bars = full_bars + 8 * NST;
    const uint32_t merge_bar = empty_bars + 8 * NST;      // bulk copies of a shared-memory merge
    const uint32_t bad_flags = merge_bar + 8;             // per stage: 1 = a page id outside the pool
    const int lane = threadIdx.x & 31;
    const bool producer = kWS && threadIdx.x < 32;
    const int g = lane >> 2, t = lane & 3;
    const int w = blockIdx.x;
    const int S = p.S, Hkv = p.Hkv, G = p.G;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(full_bars + 8 * s, 1);
            mbar_init(empty_bars + 8 * s, 1);
        }
        mbar_init(merge_bar, 1);
        fence_mbar_init();
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    __syncthreads();

    // Schedule.  A batch of up to kLocalPlanMax requests is scheduled here,
    // by every warp from the inputs, so the first copies go out without
    // waiting for the plan kernel; the plan kernel triggers this grid only
    // after its own grid_dep_wait, so every kernel before it in the stream
    // has completed and the inputs are final.  The plan's outputs (prefix
    // table, zeroed arrival counters) are read only after wait_plan().
    bool planned = false;
    auto wait_plan = [&]() {
        if (!planned) {
            grid_dep_wait();
            planned = true;
        }
    };
    // rows of requests with no tiles (aborted, empty, malformed) are zero
    auto zero_rows = [&]() {
        for (int r = w; r < p.B; r += p.NW) {
            if (p.prefix[r + 1] != p.prefix[r]) continue;
            uint4 *orow = reinterpret_cast<uint4 *>(p.out + static_cast<int64_t>(r) * p.Hq * kD);
            for (int c = lane; c < p.Hq * kD / 8; c += 32) orow[c] = make_uint4(0u, 0u, 0u, 0u);
        }
    };
    const bool local = p.B <= kLocalPlanMax;
    int64_t T;
    int64_t chunk_tiles = 0;       // local schedule: tiles of requests 32 lane .. 32 lane + 31
    int nw;
    bool aligned = false;          // small batch: every unit has whole warps
    int64_t lo = 0, hi = 0;
    FirstRequest afr;
    UnitGeom agm{0, 0};            // the warp's unit, under the aligned schedule
    // Up to 64 requests: one load of every request's row (two per lane) serves
    // both the total and the search for the first request.
    const bool cached = p.B <= 64;
    RequestInfo rc[2] = {{0, 0, 0}, {0, 0, 0}};
    if (cached) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
            if (32 * c + lane < p.B)
                rc[c] = request_info(p.seq_lens, p.indptr, p.abort_mask, p.nnz, 32 * c + lane, Hkv, S, kTile);
        T = rc[0].tiles + rc[1].tiles;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) T += __shfl_xor_sync(kFull, T, o);
        nw = working_warps(T, p.NW);
        if (kAligned) aligned = place_aligned<kTile>(rc, T, p.NW, Hkv, w, lo, hi, afr, agm);
    } else if (local) {
        T = batch_tiles(p, kTile, chunk_tiles);
        nw = working_warps(T, p.NW);
    } else {
        wait_plan();
        T = p.prefix[p.B];
        nw = p.warp_req[p.NW];                         // warps with work (<= NW)
    }
    if (!aligned) {
        lo = w < nw ? warp_lo(w, T, nw) : 0;
        hi = w < nw ? warp_lo(w + 1, T, nw) : 0;
    }
    if (lo >= hi) {
        if (!producer) {
            wait_plan();
            zero_rows();
        }
        grid_dep_launch();
        return;
    }
    const int64_t n_tiles = hi - lo;
    // entries one shared-memory merge round holds (the idle stage ring: outputs,
    // statistics and weights of each; one entry per lane)
    const int merge_cap = min(32, (NST * Lay::kStageBytes) / (G * kD * 4 + ((G + 1) & ~1) * 8 + 32));
    uint32_t merge_phase = 0;
#if FKV_KV_EVICT_FIRST
    const uint64_t policy = l2_policy_evict_first();
#else
    const uint64_t policy = l2_policy_evict_normal();
#endif

    // ---------------- load side ----------------
    Cursor L, C;
    int pid_r = -1, pbase = 0, pidA = -1, pidB = -1, lseq = 0, lneed = 0;
    int64_t lrow0 = 0;
    if (local) {
        FirstRequest fr = afr;                         // known already under the aligned schedule
        if (!aligned && cached) {
            const int64_t c1 = scan_requests(rc[0], 0, 0, lo, Hkv, fr);
            if (fr.r0 < 0) scan_requests(rc[1], 32, c1, lo, Hkv, fr);
        } else if (!aligned) {
            fr = find_request(p, kTile, lo, chunk_tiles);
        }
        cursor_at(L, fr.r0, fr.base0, fr.nt0, lo);
        pid_r = fr.r0;                                 // the first request's page-table row is known
        lseq = fr.sl0;
        lrow0 = fr.row0;
        lneed = (lseq + S - 1) / S;
        pbase = -1000;
    } else {
        cursor_init(L, p, lo, p.warp_req[w]);
    }
    C = L;

    auto fetch_ids = [&](int b) -> int {
        const int pos = b + lane;
        return pos < lneed ? __ldcg(p.indices + lrow0 + pos) : -1;
    };
    auto page_id = [&](int pos) -> int {
        if (pos < pbase || pos >= pbase + 64) {
            pbase = pos & ~31;
            pidA = fetch_ids(pbase);
            pidB = fetch_ids(pbase + 32);
        } else if (pos >= pbase + 32) {
            pidA = pidB;
            pbase += 32;
            pidB = fetch_ids(pbase + 32);
        }
        return __shfl_sync(kFull, pidA, pos - pbase);
    };
    auto issue = [&](int stage) {
        if (L.r != pid_r) {
            pid_r = L.r;
            lseq = __ldcg(p.seq_lens + L.r);
            lrow0 = __ldcg(p.indptr + L.r);
            lneed = (lseq + S - 1) / S;
            pbase = -1000;
        }
        const int tok0 = L.tt * kTile;
        const int npg = S < kTile ? kTile / S : 1;       // pages per tile (<= 4)
        const int rows = S < kTile ? S : kTile;
        const int pos0 = tok0 / S;
        const int rowoff = S < kTile ? 0 : tok0 % S;
        int ids[4] = {-1, -1, -1, -1};
        bool bad = false;
        uint32_t bytes = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (k >= npg || pos0 + k >= lneed) break;    // page beyond the request's last token
            int id = page_id(pos0 + k);
            if (id < 0 || id >= p.P) {                   // never dereference an id outside the pool
                bad = true;
                id = 0;
            }
            ids[k] = id;
            bytes += 2u * rows * 128u * Lay::kHalves;
        }
        if (lane == 0) {
            const uint32_t bar = full_bars + 8 * stage;
            st_shared_u32(bad_flags + 4 * stage, bad ? 1u : 0u);   // published by the arrive below
            mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (ids[k] < 0) break;
                const uint32_t dk = sbase + stage * Lay::kStageBytes + k * rows * 128;
                const uint32_t dv = dk + Lay::kTileBytes;
#pragma unroll
                for (int half = 0; half < Lay::kHalves; ++half) {
                    tma_load_4d(dk + half * Lay::kHalfBytes, &tmK, bar, half * 64, rowoff, L.h >> p.hshift, ids[k],
                                policy);
                    tma_load_4d(dv + half * Lay::kHalfBytes, &tmV, bar, half * 64, rowoff, L.h >> p.hshift, ids[k],
                                policy);
                }
            }
        }
    };

    if (!kWS) {                                        // fill the ring
        const int n_pro = n_tiles < NST ? static_cast<int>(n_tiles) : NST;
        for (int i = 0; i < n_pro; ++i) {
            issue(i);
            if (L.tt + 1 >= L.nt && L.h + 1 >= Hkv) wait_plan();   // next tile: another request (prefix table)
            cursor_next(L, p);
        }
    }
    if (producer) {
        // Stream the range: stage s is refilled once the consumer has released
        // it (tile j waits for the release of tile j - NST).
        for (int64_t j = 0; j < n_tiles; ++j) {
            const int st = static_cast<int>(j % NST);
            if (j >= NST && !FKV_PRODUCER_WAIT(empty_bars + 8 * st, static_cast<uint32_t>((j / NST - 1) & 1),
                                               kWaitLimitNs)) {
                if (lane == 0) atomicOr(p.err, FKV_DEVERR_TIMEOUT);
                break;                                 // the consumer gives up on the copies never issued
            }
            issue(st);
            if (j + 1 < n_tiles) {
                if (L.tt + 1 >= L.nt && L.h + 1 >= Hkv) wait_plan();   // next tile: another request (prefix table)
                cursor_next(L, p);
            }
        }
        grid_dep_launch();
        return;
    }
    wait_plan();
    zero_rows();

    const bool maybe_empty = !aligned && T < nw;       // warps with an empty range exist
    auto unit_geom = [&](int r, int h) {
        const int64_t base = p.prefix[r];
        const int64_t nt = (p.prefix[r + 1] - base) / Hkv;
        const int64_t s0 = base + h * nt;
        const int64_t wf = warp_of_tile(s0, T, nw);
        return UnitGeom{static_cast<int>(wf), static_cast<int>(warp_of_tile(s0 + nt - 1, T, nw) - wf + 1)};
    };
    // A merge this warp owes (kFinalDue: the single-level merge of a unit;
    // kChunkDue: the first level of a two-level merge, then the unit's
    // arrival and, if last, its second level), for unit (r, h), performed at
    // the end of the warp's range, where the stage ring is idle.
    auto merge_steps = [&](int stage, const UnitGeom &gm, int r, int h, float vsc) {
        auto merge = [&](int64_t sl0, int cnt, int stride, bool me, int64_t wk0, bool fin, int64_t d) {
            if (merge_parts_smem(p, sbase, merge_cap, merge_bar, merge_phase, nw, sl0, cnt, stride, me, wk0, T,
                                 fin, r, h, vsc, d))
                return true;
            if (lane == 0) atomicOr(p.err, FKV_DEVERR_TIMEOUT);
            return false;
        };
        const int64_t u = static_cast<int64_t>(r) * Hkv + h;
        __syncwarp();
        if (stage == kFinalDue) {
            merge(u + gm.wf, gm.span, 1, maybe_empty, gm.wf, true, 0);
            return;
        }
        const int c0 = gm.c0(w), csz = gm.csz(w);
        if (csz > 1 && !merge(u + gm.wf + c0, csz, 1, false, gm.wf + c0, false, u + gm.wf + c0)) return;
        __syncwarp();
        int last2 = 0;
        if (lane == 0) last2 = atomic_add_acq_rel_gpu(p.counters + u, 1) == gm.nch() - 1;
        if (__shfl_sync(kFull, last2, 0)) {
            __syncwarp();
            merge(u + gm.wf, gm.nch(), kChunk, false, gm.wf, true, 0);
        }
    };

    // ---------------- compute side ----------------
    uint32_t qb[8][2];
    float cfac[2] = {0.f, 0.f};
    float m[2], l[2];
    float o[8][4];
    int cseq = 0, seg_start = 0;
    bool unit_bad = false;
    float cvsc = 1.f;       // the unit's V scale
    UnitGeom cgm = agm;     // where the unit's parts sit, if it is split (span 0: not yet known)
    // a merge this warp owes from the middle of its range: at most one, since
    // only the unit it started in can end there and be split
    int def_stage = kNone, def_r = 0, def_h = 0;
    UnitGeom def_gm{0, 0};
    float def_vsc = 1.f;

    for (int64_t i = 0; i < n_tiles; ++i) {
        const int s = static_cast<int>(i % NST);
        const uint32_t parity = static_cast<uint32_t>((i / NST) & 1);

        if (i == 0 || C.tt == 0) {
            // ---- new unit (r, h): queries, logit factors, fresh softmax state ----
            cseq = __ldg(p.seq_lens + C.r);
            seg_start = C.tt;
            unit_bad = false;
            cvsc = kFp8 ? __ldg(p.v_scale + (C.h >> p.hshift)) : 1.f;
            // a unit that started in an earlier warp or ends in a later one is
            // split: find its parts now, off the merge's critical path
            // (the aligned schedule placed the warp's one unit already)
            if ((seg_start > 0 || C.nt - C.tt > n_tiles - i) && (i > 0 || cgm.span == 0))
                cgm = unit_geom(C.r, C.h);
            m[0] = m[1] = -INFINITY;
            l[0] = l[1] = 0.f;
#pragma unroll
            for (int a = 0; a < 8; ++a) o[a][0] = o[a][1] = o[a][2] = o[a][3] = 0.f;
            const int64_t qrow = static_cast<int64_t>(C.r) * p.Hq + C.h * G + g;
            const uint4 *q4 = reinterpret_cast<const uint4 *>(p.q) + qrow * (kD / 8);
            uint4 qv[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                           make_uint4(0, 0, 0, 0)};
            if (g < G) {
                if (kFp8) {            // dims 32t .. 32t+31
#pragma unroll
                    for (int k = 0; k < 4; ++k) qv[k] = __ldg(q4 + 4 * t + k);
                } else {               // dims 16t .. 16t+15 and 64+16t .. 64+16t+15
                    qv[0] = __ldg(q4 + 2 * t);
                    qv[1] = __ldg(q4 + 2 * t + 1);
                    qv[2] = __ldg(q4 + 8 + 2 * t);
                    qv[3] = __ldg(q4 + 8 + 2 * t + 1);
                }
            }
            const uint32_t qw[16] = {qv[0].x, qv[0].y, qv[0].z, qv[0].w, qv[1].x, qv[1].y, qv[1].z, qv[1].w,
                                     qv[2].x, qv[2].y, qv[2].z, qv[2].w, qv[3].x, qv[3].y, qv[3].z, qv[3].w};
            if (kFp8) {
                // bf16 -> f16 with a power-of-two row scale so the row's largest
                // magnitude lands in [2^14, 2^15): exact for every element within
                // 2^-24 of it.  The scale is undone in the logit factor.
                float amax = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    amax = fmaxf(amax, fabsf(__uint_as_float(qw[j] << 16)));
                    amax = fmaxf(amax, fabsf(__uint_as_float(qw[j] & 0xFFFF0000u)));
                }
                amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
                int e = amax > 0.f ? static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 127 : 0;
                e = max(-100, min(127, e));
                const float sc = __uint_as_float(static_cast<uint32_t>(127 + 14 - e) << 23);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t w0 = qw[2 * ks], w1 = qw[2 * ks + 1];
                    qb[ks][0] = pack_f16x2(__uint_as_float(w0 << 16) * sc, __uint_as_float(w0 & 0xFFFF0000u) * sc);
                    qb[ks][1] = pack_f16x2(__uint_as_float(w1 << 16) * sc, __uint_as_float(w1 & 0xFFFF0000u) * sc);
                }
                const float ksc = __ldg(p.k_scale + (C.h >> p.hshift)) * p.sm_scale_log2;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int ej = __shfl_sync(kFull, e, (2 * t + j) * 4);
                    cfac[j] = ksc * __uint_as_float(static_cast<uint32_t>(127 + ej - 14) << 23);
                }
            } else {
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    qb[ks][0] = qw[2 * ks];
                    qb[ks][1] = qw[2 * ks + 1];
                }
                cfac[0] = cfac[1] = p.sm_scale_log2;
            }
        }

        // ---- wait for this stage's copies ----
        if (!mbar_wait_bounded(full_bars + 8 * s, parity, kWaitLimitNs)) {
            if (lane == 0) atomicOr(p.err, FKV_DEVERR_TIMEOUT);
            // wind down: let every copy still in flight land before leaving
            // (the producer is never more than NST tiles ahead)
            const int64_t last = i + NST < n_tiles ? i + NST : n_tiles;
            for (int64_t j = i; j < last; ++j)
                (void)mbar_wait_bounded(full_bars + 8 * static_cast<int>(j % NST),
                                        static_cast<uint32_t>((j / NST) & 1), kDrainLimitNs);
            return;
        }
        if (ld_shared_u32(bad_flags + 4 * s)) {
            if (!unit_bad && lane == 0) atomicOr(p.err, FKV_DEVERR_ATTN_PAGE);
            unit_bad = true;
        }
        const uint32_t kbase = sbase + s * Lay::kStageBytes;
        const uint32_t vbase = kbase + Lay::kTileBytes;
        const int nvalid = min(kTile, cseq - C.tt * kTile);

        if (nvalid < kTile) {
            // rows past the request's last token hold stale bytes: zero V there
            // (K rows are masked out of the softmax instead)
            const int nch = (kTile - nvalid) * 8;
#pragma unroll
            for (int half = 0; half < Lay::kHalves; ++half)
                for (int c = lane; c < nch; c += 32)
                    st_shared_v4_zero(vbase + half * Lay::kHalfBytes + nvalid * 128 + c * 16);
            fence_proxy_async_smem();
            __syncwarp();
        }

        // ---- S^T = K Q^T : tokens on M (16-row tiles), heads on N ----
        float sacc[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            float acc[NACC][4];
#pragma unroll
            for (int a = 0; a < NACC; ++a) acc[a][0] = acc[a][1] = acc[a][2] = acc[a][3] = 0.f;
            const int ra = mt * 16 + g, rb = ra + 8;
            if (kFp8) {
                // this lane's 32 dims of rows ra, rb: 16-byte chunks 2t, 2t+1 (swizzled)
                const uint4 a0 = ld_shared_v4(kbase + ra * 128 + (((2 * t) ^ (ra & 7)) << 4));
                const uint4 a1 = ld_shared_v4(kbase + ra * 128 + (((2 * t + 1) ^ (ra & 7)) << 4));
                const uint4 b0 = ld_shared_v4(kbase + rb * 128 + (((2 * t) ^ (rb & 7)) << 4));
                const uint4 b1 = ld_shared_v4(kbase + rb * 128 + (((2 * t + 1) ^ (rb & 7)) << 4));
                const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    mma_f16(acc[ks % NACC], e4m3x2_to_f16x2(lo16(wa[ks])), e4m3x2_to_f16x2(lo16(wb[ks])),
                            e4m3x2_to_f16x2(hi16(wa[ks])), e4m3x2_to_f16x2(hi16(wb[ks])), qb[ks][0], qb[ks][1]);
                }
            } else {
                // dims 16t..16t+15 (half 0, chunks 2t, 2t+1) and 64+16t.. (half 1)
                uint32_t wa[16], wb[16];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int half = k >> 1, c = 2 * t + (k & 1);
                    const uint4 va = ld_shared_v4(kbase + half * Lay::kHalfBytes + ra * 128 + ((c ^ (ra & 7)) << 4));
                    const uint4 vb = ld_shared_v4(kbase + half * Lay::kHalfBytes + rb * 128 + ((c ^ (rb & 7)) << 4));
                    wa[4 * k] = va.x; wa[4 * k + 1] = va.y; wa[4 * k + 2] = va.z; wa[4 * k + 3] = va.w;
                    wb[4 * k] = vb.x; wb[4 * k + 1] = vb.y; wb[4 * k + 2] = vb.z; wb[4 * k + 3] = vb.w;
                }
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16(acc[ks % NACC], wa[2 * ks], wb[2 * ks], wa[2 * ks + 1], wb[2 * ks + 1], qb[ks][0],
                             qb[ks][1]);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) sacc[mt][c] = NACC == 2 ? acc[0][c] + acc[NACC - 1][c] : acc[0][c];
        }

        // ---- online softmax (log2 domain); columns are heads 2t, 2t+1 ----
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            if (mt * 16 + g >= nvalid) sacc[mt][0] = sacc[mt][1] = -INFINITY;
            if (mt * 16 + g + 8 >= nvalid) sacc[mt][2] = sacc[mt][3] = -INFINITY;
        }
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            mx[0] = fmaxf(mx[0], fmaxf(sacc[mt][0], sacc[mt][2]));
            mx[1] = fmaxf(mx[1], fmaxf(sacc[mt][1], sacc[mt][3]));
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            mx[j] = fmaxf(mx[j], __shfl_xor_sync(kFull, mx[j], 4));
            mx[j] = fmaxf(mx[j], __shfl_xor_sync(kFull, mx[j], 8));
            mx[j] = fmaxf(mx[j], __shfl_xor_sync(kFull, mx[j], 16));
        }
        // Each logit is scaled with one rounded multiply, the same operation
        // that forms the running maximum, so the largest logit gives exactly
        // ex2(0) = 1 and every other one at most 1.  (A fused multiply-add
        // against the rounded maximum would leave the product's rounding error,
        // up to half an ulp of the logit: harmless for ordinary logits, but
        // past ~2^33 in log2 units that error overflows ex2.)
        float alpha[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float mnew = fmaxf(m[j], __fmul_rn(mx[j], cfac[j]));
            alpha[j] = ex2(m[j] - mnew);
            m[j] = mnew;
        }
        float pr[MT][4];
        float ls[2] = {0.f, 0.f};
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                pr[mt][c] = ex2(__fmul_rn(sacc[mt][c], cfac[c & 1]) - m[c & 1]);
                ls[c & 1] += pr[mt][c];
            }
        l[0] = l[0] * alpha[0] + ls[0];
        l[1] = l[1] * alpha[1] + ls[1];
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            o[a][0] *= alpha[0];
            o[a][2] *= alpha[0];
            o[a][1] *= alpha[1];
            o[a][3] *= alpha[1];
        }
        // P^T fragments: transpose (token, head) 8x8 blocks into (head, token).
        // FP8: P in f16 (11-bit significand).  BF16: the MMA needs bf16 P, whose
        // 8-bit significand alone would cost up to 2^-9 |v| in the output, so P
        // is split into bf16 hi + lo parts and PV runs on both (16 bits).
        uint32_t pb[MT][2], pl[MT][2];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            if (kFp8) {
                pb[mt][0] = movmatrix_trans(pack_f16x2(pr[mt][0], pr[mt][1]));
                pb[mt][1] = movmatrix_trans(pack_f16x2(pr[mt][2], pr[mt][3]));
                pl[mt][0] = pl[mt][1] = 0u;
            } else {
                const uint32_t h0 = pack_bf16x2(pr[mt][0], pr[mt][1]);
                const uint32_t h1 = pack_bf16x2(pr[mt][2], pr[mt][3]);
                const uint32_t l0 = pack_bf16x2(pr[mt][0] - __uint_as_float(h0 << 16),
                                                pr[mt][1] - __uint_as_float(h0 & 0xFFFF0000u));
                const uint32_t l1 = pack_bf16x2(pr[mt][2] - __uint_as_float(h1 << 16),
                                                pr[mt][3] - __uint_as_float(h1 & 0xFFFF0000u));
                pb[mt][0] = movmatrix_trans(h0);
                pb[mt][1] = movmatrix_trans(h1);
                pl[mt][0] = movmatrix_trans(l0);
                pl[mt][1] = movmatrix_trans(l1);
            }
        }

        // ---- O^T += V^T P^T : dims on M (8 blocks of 16), tokens on K ----
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int r0 = mt * 16 + 2 * t, r1 = r0 + 1, r2 = r0 + 8, r3 = r0 + 9;
            if (kFp8) {
                // dims 16g .. 16g+15 of four token rows (16-byte chunk g, swizzled)
                const uint4 A = ld_shared_v4(vbase + r0 * 128 + ((g ^ (r0 & 7)) << 4));
                const uint4 Bv = ld_shared_v4(vbase + r1 * 128 + ((g ^ (r1 & 7)) << 4));
                const uint4 Cv = ld_shared_v4(vbase + r2 * 128 + ((g ^ (r2 & 7)) << 4));
                const uint4 Dv = ld_shared_v4(vbase + r3 * 128 + ((g ^ (r3 & 7)) << 4));
                const uint32_t a[4] = {A.x, A.y, A.z, A.w}, b[4] = {Bv.x, Bv.y, Bv.z, Bv.w};
                const uint32_t c[4] = {Cv.x, Cv.y, Cv.z, Cv.w}, d[4] = {Dv.x, Dv.y, Dv.z, Dv.w};
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    // pair the same dim of tokens (r0, r1) and (r2, r3)
                    const uint32_t ab0 = prmt(a[qq], b[qq], 0x5140), ab1 = prmt(a[qq], b[qq], 0x7362);
                    const uint32_t cd0 = prmt(c[qq], d[qq], 0x5140), cd1 = prmt(c[qq], d[qq], 0x7362);
                    mma_f16(o[2 * qq], e4m3x2_to_f16x2(lo16(ab0)), e4m3x2_to_f16x2(hi16(ab0)),
                            e4m3x2_to_f16x2(lo16(cd0)), e4m3x2_to_f16x2(hi16(cd0)), pb[mt][0], pb[mt][1]);
                    mma_f16(o[2 * qq + 1], e4m3x2_to_f16x2(lo16(ab1)), e4m3x2_to_f16x2(hi16(ab1)),
                            e4m3x2_to_f16x2(lo16(cd1)), e4m3x2_to_f16x2(hi16(cd1)), pb[mt][0], pb[mt][1]);
                }
            } else {
                // dims 8g..8g+7 (half 0, chunk g) and 64+8g.. (half 1, chunk g)
                uint32_t a[8], b[8], c[8], d[8];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const uint32_t hb = vbase + half * Lay::kHalfBytes;
                    const uint4 A = ld_shared_v4(hb + r0 * 128 + ((g ^ (r0 & 7)) << 4));
                    const uint4 Bv = ld_shared_v4(hb + r1 * 128 + ((g ^ (r1 & 7)) << 4));
                    const uint4 Cv = ld_shared_v4(hb + r2 * 128 + ((g ^ (r2 & 7)) << 4));
                    const uint4 Dv = ld_shared_v4(hb + r3 * 128 + ((g ^ (r3 & 7)) << 4));
                    a[4 * half] = A.x; a[4 * half + 1] = A.y; a[4 * half + 2] = A.z; a[4 * half + 3] = A.w;
                    b[4 * half] = Bv.x; b[4 * half + 1] = Bv.y; b[4 * half + 2] = Bv.z; b[4 * half + 3] = Bv.w;
                    c[4 * half] = Cv.x; c[4 * half + 1] = Cv.y; c[4 * half + 2] = Cv.z; c[4 * half + 3] = Cv.w;
                    d[4 * half] = Dv.x; d[4 * half + 1] = Dv.y; d[4 * half + 2] = Dv.z; d[4 * half + 3] = Dv.w;
                }
#pragma unroll
                for (int blk = 0; blk < 8; ++blk) {
                    const uint32_t A0 = prmt(a[blk], b[blk], 0x5410), A1 = prmt(a[blk], b[blk], 0x7632);
                    const uint32_t A2 = prmt(c[blk], d[blk], 0x5410), A3 = prmt(c[blk], d[blk], 0x7632);
                    mma_bf16(o[blk], A0, A1, A2, A3, pb[mt][0], pb[mt][1]);
                    mma_bf16(o[blk], A0, A1, A2, A3, pl[mt][0], pl[mt][1]);
                }
            }
        }
        __syncwarp();

        if (kWS) {
            // ---- hand the stage back to the producer ----
            if (lane == 0) mbar_arrive(empty_bars + 8 * s);
        } else if (i + NST < n_tiles) {
            // ---- refill this stage with the tile NST ahead ----
            issue(s);
            cursor_next(L, p);
        }

        // ---- end of this warp's share of the unit ----
        if (C.tt == C.nt - 1 || i == n_tiles - 1) {
            float lt[2] = {l[0], l[1]};
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                lt[j] += __shfl_xor_sync(kFull, lt[j], 4);
                lt[j] += __shfl_xor_sync(kFull, lt[j], 8);
                lt[j] += __shfl_xor_sync(kFull, lt[j], 16);
            }
            const bool whole = seg_start == 0 && C.tt == C.nt - 1;
            const int64_t u = static_cast<int64_t>(C.r) * Hkv + C.h;
            // parts of a split unit that hold tiles (warps of its span with a
            // non-empty range)
            auto unit_parts = [&](const UnitGeom &gm) {
                int n = gm.span;
                if (maybe_empty) {
                    n = 0;
                    for (int64_t x = gm.wf; x < gm.wf + gm.span; ++x) n += warp_lo(x, T, nw) != warp_lo(x + 1, T, nw);
                }
                return n;
            };
            // The unit's final merge from this warp's registers plus the other
            // parts' partials (at most two), loaded straight from L2: their
            // statistics and the first one's outputs in one round trip, the
            // second one's outputs in another.  This warp holds the unit's
            // first part, so its registers are entry 0 of merge_parts_smem's
            // definition and the other parts follow in index order; every
            // step below is that definition's, with the same roundings, so the
            // row's bytes equal those of the merge through the stage ring.
            // The caller has acquired every other part.
            auto merge_regs = [&](int64_t u) {
                const int d0 = kFp8 ? 16 * g : 8 * g, d1 = kFp8 ? 16 * g + 8 : 64 + 8 * g;
                int64_t x0 = 0, x1 = 0;                       // the other parts, in index order
                int no = 0;
                for (int64_t x = cgm.wf; x < cgm.wf + cgm.span; ++x) {
                    if (x == w || (maybe_empty && warp_lo(x, T, nw) == warp_lo(x + 1, T, nw))) continue;
                    if (no == 0) x0 = x;
                    else x1 = x;
                    ++no;
                }
                // lanes past the group's heads read a valid row and drop it
                float2 ml[2][2];
                float4 q[2][4];
                auto load_rows = [&](int k) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int hd = min(2 * t + j, G - 1);
                        const float4 *prow =
                            reinterpret_cast<const float4 *>(p.part_o + ((u + (k ? x1 : x0)) * G + hd) * kD);
                        q[j][0] = __ldcg(prow + d0 / 4);
                        q[j][1] = __ldcg(prow + d0 / 4 + 1);
                        q[j][2] = __ldcg(prow + d1 / 4);
                        q[j][3] = __ldcg(prow + d1 / 4 + 1);
                    }
                };
#pragma unroll
                for (int k = 0; k < 2; ++k)
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        ml[k][j] = k < no ? __ldcg(p.part_ml + (u + (k ? x1 : x0)) * p.GP + min(2 * t + j, G - 1))
                                          : make_float2(-INFINITY, 0.f);
                load_rows(0);
                bool bad = unit_bad;
                float v[2][16], w1[2], w2[2], Lj[2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    bad |= ml[0][j].y < 0.f || ml[1][j].y < 0.f;
                    const float mx = fmaxf(fmaxf(m[j], ml[0][j].x), ml[1][j].x);
                    const float w0 = m[j] == -INFINITY ? 0.f : ex2(m[j] - mx);
                    w1[j] = ml[0][j].x == -INFINITY ? 0.f : ex2(ml[0][j].x - mx);
                    w2[j] = ml[1][j].x == -INFINITY ? 0.f : ex2(ml[1][j].x - mx);
                    // the lanes' butterfly sum with entries at lanes 0, 1, 2 (zeros past them)
                    const float sl = __fadd_rn(__fadd_rn(__fmul_rn(w0, lt[j]), __fmul_rn(w1[j], ml[0][j].y)),
                                               __fmul_rn(w2[j], ml[1][j].y));
                    Lj[j] = __fmaf_rn(0.f, 0.f, sl);
#pragma unroll
                    for (int a = 0; a < 8; ++a) {
                        v[j][2 * a] = __fmaf_rn(w0, o[a][j], 0.f);
                        v[j][2 * a + 1] = __fmaf_rn(w0, o[a][2 + j], 0.f);
                    }
                }
                for (int k = 0; k < no; ++k) {
                    if (k == 1) load_rows(1);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float qv[16] = {q[j][0].x, q[j][0].y, q[j][0].z, q[j][0].w, q[j][1].x, q[j][1].y,
                                              q[j][1].z, q[j][1].w, q[j][2].x, q[j][2].y, q[j][2].z, q[j][2].w,
                                              q[j][3].x, q[j][3].y, q[j][3].z, q[j][3].w};
                        const float wk = k == 0 ? w1[j] : w2[j];
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[j][e] = __fmaf_rn(wk, qv[e], v[j][e]);
                    }
                }
                bad = __any_sync(kFull, bad);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int hd = 2 * t + j;
                    if (hd >= G) continue;
                    const float f = __fdiv_rn(cvsc, Lj[j]);
                    __nv_bfloat16 *orow = p.out + (static_cast<int64_t>(C.r) * p.Hq + C.h * G + hd) * kD;
                    uint4 r0v = make_uint4(0u, 0u, 0u, 0u), r1v = make_uint4(0u, 0u, 0u, 0u);
                    if (!bad) {                                // fail closed: zeros, whatever the data
                        r0v.x = pack_bf16x2(__fmul_rn(v[j][0], f), __fmul_rn(v[j][1], f));
                        r0v.y = pack_bf16x2(__fmul_rn(v[j][2], f), __fmul_rn(v[j][3], f));
                        r0v.z = pack_bf16x2(__fmul_rn(v[j][4], f), __fmul_rn(v[j][5], f));
                        r0v.w = pack_bf16x2(__fmul_rn(v[j][6], f), __fmul_rn(v[j][7], f));
                        r1v.x = pack_bf16x2(__fmul_rn(v[j][8], f), __fmul_rn(v[j][9], f));
                        r1v.y = pack_bf16x2(__fmul_rn(v[j][10], f), __fmul_rn(v[j][11], f));
                        r1v.z = pack_bf16x2(__fmul_rn(v[j][12], f), __fmul_rn(v[j][13], f));
                        r1v.w = pack_bf16x2(__fmul_rn(v[j][14], f), __fmul_rn(v[j][15], f));
                    }
                    *reinterpret_cast<uint4 *>(orow + d0) = r0v;
                    *reinterpret_cast<uint4 *>(orow + d1) = r1v;
                }
            };
            bool merged = false;
#if FKV_TRY_LAST
            if (!whole && seg_start == 0 && i == n_tiles - 1 && (maybe_empty || cgm.span <= kChunk) &&
                unit_parts(cgm) <= 3) {
                // This warp holds the unit's first part (the unit started in
                // its range and runs to the range end).  The unit's other
                // parts usually end early in their warps' ranges, so at this
                // warp's range end they may all have arrived.  Then this warp
                // is the last: it merges its registers with their partials,
                // loaded straight from global memory (one round trip for a
                // unit over two warps), and writes the row -- no partial of
                // its own, no arrival.  Otherwise it publishes and arrives as
                // below.  (Only the first part of a unit of at most three
                // parts does this: merge_regs reproduces merge_parts_smem's
                // arithmetic for that case.)
                int known = 0;
                if (lane == 0) known = ld_acquire_gpu(p.counters + u) == unit_parts(cgm) - 1;
                merged = __shfl_sync(kFull, known, 0) != 0;
                if (merged) {
                    __syncwarp();                              // lane 0's acquire covers the warp's loads
                    merge_regs(u);
                }
            }
#endif
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int hd = 2 * t + j;
                if (hd >= G || merged) continue;
                // this lane's 16 dims of head hd, in ascending order
                float v[16];
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    v[2 * a] = o[a][j];
                    v[2 * a + 1] = o[a][2 + j];
                }
                const int d0 = kFp8 ? 16 * g : 8 * g;          // first run of dims
                const int d1 = kFp8 ? 16 * g + 8 : 64 + 8 * g; // second run (8 dims each)
                if (whole) {
                    const float f = cvsc / lt[j];
                    __nv_bfloat16 *orow = p.out + (static_cast<int64_t>(C.r) * p.Hq + C.h * G + hd) * kD;
                    uint4 r0v = make_uint4(0u, 0u, 0u, 0u), r1v = make_uint4(0u, 0u, 0u, 0u);
                    if (!unit_bad) {                           // fail closed: zeros, whatever the data
                        r0v.x = pack_bf16x2(v[0] * f, v[1] * f);
                        r0v.y = pack_bf16x2(v[2] * f, v[3] * f);
                        r0v.z = pack_bf16x2(v[4] * f, v[5] * f);
                        r0v.w = pack_bf16x2(v[6] * f, v[7] * f);
                        r1v.x = pack_bf16x2(v[8] * f, v[9] * f);
                        r1v.y = pack_bf16x2(v[10] * f, v[11] * f);
                        r1v.z = pack_bf16x2(v[12] * f, v[13] * f);
                        r1v.w = pack_bf16x2(v[14] * f, v[15] * f);
                    }
                    *reinterpret_cast<uint4 *>(orow + d0) = r0v;
                    *reinterpret_cast<uint4 *>(orow + d1) = r1v;
                } else {
                    const int64_t slot = u + w;
                    float *prow = p.part_o + (slot * G + hd) * kD;
                    __stcg(reinterpret_cast<float4 *>(prow + d0), make_float4(v[0], v[1], v[2], v[3]));
                    __stcg(reinterpret_cast<float4 *>(prow + d0 + 4), make_float4(v[4], v[5], v[6], v[7]));
                    __stcg(reinterpret_cast<float4 *>(prow + d1), make_float4(v[8], v[9], v[10], v[11]));
                    __stcg(reinterpret_cast<float4 *>(prow + d1 + 4), make_float4(v[12], v[13], v[14], v[15]));
                    if (g == 0) __stcg(p.part_ml + slot * p.GP + hd, make_float2(m[j], unit_bad ? -1.f : lt[j]));
                }
            }
            if (!whole && !merged) {
                // Merge without waiting: the last of the unit's warps to arrive
                // merges.  Units split over more than kChunk warps merge in two
                // levels (chunks of kChunk consecutive parts, then the chunks),
                // so no single warp reads a long unit's partials serially.
                // Arrivals are acquire-release atomics by lane 0 after a warp
                // barrier: they publish this warp's partial and, for the last
                // arriver, make every other part visible.
                const UnitGeom &gm = cgm;
                int stage = kNone;
                __syncwarp();
                if (maybe_empty || gm.span <= kChunk) {
                    const int nparts = unit_parts(gm);
                    int last = 0;
                    if (lane == 0) last = atomic_add_acq_rel_gpu(p.counters + u, 1) == nparts - 1;
                    stage = __shfl_sync(kFull, last, 0) ? kFinalDue : kNone;
                } else {
                    // A one-part chunk (the unit's last warp, whose part ends early in
                    // its range) is already its own result: no first level.
                    const int csz = gm.csz(w);
                    int last = csz == 1;
                    if (csz > 1 && lane == 0)
                        last = atomic_add_acq_rel_gpu(p.chunk_counters + (u + gm.wf + gm.c0(w)), 1) == csz - 1;
                    stage = __shfl_sync(kFull, last, 0) ? kChunkDue : kNone;
                }
                // at the range end the stage ring is idle: merge through it
                if (stage != kNone && i < n_tiles - 1) {
                    // mid-range: the stream would stall for the merge, and a
                    // part ending just before this range's end can be the last
                    // to arrive, putting that stall on the call's critical path;
                    // owe it until the range end instead
                    def_stage = stage;
                    def_gm = gm;
                    def_r = C.r;
                    def_h = C.h;
                    def_vsc = cvsc;
                    stage = kNone;
                }
                if (stage != kNone) merge_steps(stage, gm, C.r, C.h, cvsc);
            }
        }
        cursor_next(C, p);
    }
    if (def_stage != kNone) merge_steps(def_stage, def_gm, def_r, def_h, def_vsc);
    grid_dep_launch();
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {

constexpr int kMaxDev = 64;
std::mutex g_mu;
// Resident CTAs per SM, [dev][kv_fp8][ws], with the id of the context in
// which the kernels' shared-memory limit was raised: a new context (after
// cudaDeviceReset) loads the kernels again, so the attribute is set again.
struct CtasPerSm {
    unsigned long long ctx_id;
    int n;
};
CtasPerSm g_ctas_per_sm[kMaxDev][2][2];

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

template <bool kFp8, bool kWS>
int ctas_per_sm() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    CtasPerSm &c = g_ctas_per_sm[dev][kFp8 ? 1 : 0][kWS ? 1 : 0];
    const unsigned long long ctx = current_context_id();
    if (!c.n || ctx == 0 || ctx != c.ctx_id) {
        const int smem = Layout<kFp8>::kSmem;
        if (cudaFuncSetAttribute(paged_decode_attn_kernel<kFp8, kWS, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
            cudaFuncSetAttribute(paged_decode_attn_kernel<kFp8, kWS, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return 0;
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, paged_decode_attn_kernel<kFp8, kWS, false>,
                                                          attn_threads(kWS), smem) != cudaSuccess ||
            nb <= 0)
            return 0;
        c.n = nb < 16 ? nb : 16;
        c.ctx_id = current_context_id();
    }
    return c.n;
}

// Computing warps of one launch (one per CTA).
int grid_warps(bool fp8, bool ws) {
    const int sms = device_sm_count();
    const int per = fp8 ? (ws ? ctas_per_sm<true, true>() : ctas_per_sm<true, false>())
                        : (ws ? ctas_per_sm<false, true>() : ctas_per_sm<false, false>());
    return sms * per;
}

// The two-warp CTA when a tile spans several pages (page sizes below
// FKV_WS_PAGE_LIMIT, by default the tile).
#ifndef FKV_WS_PAGE_LIMIT
#define FKV_WS_PAGE_LIMIT 64
#endif
bool use_ws(int page_size, bool fp8) {
    const int tile = fp8 ? Layout<true>::kTile : Layout<false>::kTile;
    return page_size < (FKV_WS_PAGE_LIMIT < tile ? FKV_WS_PAGE_LIMIT : tile);
}

template <bool kFp8, bool kWS>
cudaError_t launch_attn(bool aligned, dim3 grid, cudaStream_t st, const AttnParams &p, const CUtensorMap &tmK,
                        const CUtensorMap &tmV) {
    const dim3 block(attn_threads(kWS));
    return aligned ? launch_pdl(paged_decode_attn_kernel<kFp8, kWS, true>, grid, block, Layout<kFp8>::kSmem, st, p,
                                tmK, tmV)
                   : launch_pdl(paged_decode_attn_kernel<kFp8, kWS, false>, grid, block, Layout<kFp8>::kSmem, st, p,
                                tmK, tmV);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
    size_t prefix, warp_req, counters, part_ml, part_o, total;
};

// Virtual KV heads per KV head for a group of G query heads: the smallest
// power of two R with G % R == 0 and G / R <= kMaxGroup (1 up to 8 query
// heads); 0 if there is none within kMaxSplit.
int group_split(int G) {
    for (int r = 1; r <= kMaxSplit; r <<= 1)
        if (G % r == 0 && G / r <= kMaxGroup) return r;
    return 0;
}

WsLayout ws_layout(int B, int Hkv, int G, int NW) {
    WsLayout L;
    const size_t units = static_cast<size_t>(B) * Hkv;
    const size_t slots = units + NW;
    L.prefix = 0;
    L.warp_req = align256(L.prefix + sizeof(int64_t) * (static_cast<size_t>(B) + 1));
    L.counters = align256(L.warp_req + sizeof(int32_t) * (NW + 1));
    L.part_ml = align256(L.counters + sizeof(int32_t) * (units + slots));
    L.part_o = align256(L.part_ml + sizeof(float2) * slots * ((G + 1) & ~1));
    L.total = align256(L.part_o + sizeof(float) * slots * G * kD);
    return L;
}

bool make_kv_map(CUtensorMap *m, const void *base, bool fp8, int P, int Hkv, int S, int tile) {
    auto enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t es = fp8 ? 1 : 2;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(S),
                                static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(P)};
    const cuuint64_t strides[3] = {kD * es, static_cast<cuuint64_t>(S) * kD * es,
                                   static_cast<cuuint64_t>(Hkv) * S * kD * es};
    const cuuint32_t box[4] = {fp8 ? 128u : 64u, static_cast<cuuint32_t>(S < tile ? S : tile), 1u, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUresult r = enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                           const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace
}  // namespace fkv

using namespace fkv;

extern "C" size_t paged_decode_attn_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                                   int32_t head_dim, int32_t kv_dtype) {
    if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return 0;
    if (head_dim != kD || (kv_dtype != FKV_KV_FP8_E4M3 && kv_dtype != FKV_KV_BF16)) return 0;
    const int R = group_split(num_q_heads / num_kv_heads);
    if (R == 0) return 0;
    // sized for either CTA shape (the page size is not known here)
    const bool fp8 = kv_dtype == FKV_KV_FP8_E4M3;
    const int n1 = grid_warps(fp8, false), n2 = grid_warps(fp8, true);
    const int NW = n1 > n2 ? n1 : n2;
    if (n1 <= 0 || n2 <= 0) return 0;
    return ws_layout(batch, num_kv_heads * R, num_q_heads / num_kv_heads / R, NW).total;
}

extern "C" fkv_status paged_decode_attn(const void *q, int32_t batch, int32_t num_q_heads, const void *k_cache,
                                        const void *v_cache, int32_t kv_dtype, const float *k_scale,
                                        const float *v_scale, int32_t num_pages, int32_t num_kv_heads,
                                        int32_t page_size, int32_t head_dim, const int32_t *page_indptr,
                                        const int32_t *page_indices, int64_t nnz, const int32_t *seq_lens,
                                        const uint8_t *abort_mask, float sm_scale, void *out, void *workspace,
                                        size_t workspace_bytes, void *stream) {
    if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_pages <= 0 || nnz < 0) return FKV_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads) return FKV_ERR_INVALID_ARG;
    if (kv_dtype != FKV_KV_FP8_E4M3 && kv_dtype != FKV_KV_BF16) return FKV_ERR_INVALID_ARG;
    if (head_dim != kD) return FKV_ERR_UNSUPPORTED;
    if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128) return FKV_ERR_UNSUPPORTED;
    // units are (request, virtual KV head) pairs of G query heads each
    const int R = group_split(num_q_heads / num_kv_heads);
    if (R == 0) return FKV_ERR_UNSUPPORTED;
    const int Hv = num_kv_heads * R, G = num_q_heads / Hv;
    if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return FKV_ERR_INVALID_ARG;
    if (batch == 0) return FKV_OK;
    const bool fp8 = kv_dtype == FKV_KV_FP8_E4M3;
    if (!q || !k_cache || !v_cache || !page_indptr || !seq_lens || !out || !workspace) return FKV_ERR_INVALID_ARG;
    if (nnz > 0 && !page_indices) return FKV_ERR_INVALID_ARG;
    if (fp8 && (!k_scale || !v_scale)) return FKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return FKV_ERR_INVALID_ARG;
    const bool two_warp = use_ws(page_size, fp8);
    const int NW = grid_warps(fp8, two_warp);
    uint32_t *err = device_error_word();
    if (NW <= 0 || !err) return FKV_ERR_CUDA;
    const WsLayout wl = ws_layout(batch, Hv, G, NW);
    if (workspace_bytes < wl.total) return FKV_ERR_INVALID_ARG;
    const int tile = fp8 ? Layout<true>::kTile : Layout<false>::kTile;

    CUtensorMap tmK, tmV;
    if (!make_kv_map(&tmK, k_cache, fp8, num_pages, num_kv_heads, page_size, tile) ||
        !make_kv_map(&tmV, v_cache, fp8, num_pages, num_kv_heads, page_size, tile))
        return FKV_ERR_CUDA;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    AttnParams p;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.indptr = page_indptr;
    p.indices = page_indices;
    p.seq_lens = seq_lens;
    p.abort_mask = abort_mask;
    p.nnz = nnz;
    p.prefix = reinterpret_cast<const int64_t *>(ws + wl.prefix);
    p.warp_req = reinterpret_cast<const int32_t *>(ws + wl.warp_req);
    p.counters = reinterpret_cast<int32_t *>(ws + wl.counters);
    p.chunk_counters = p.counters + static_cast<int64_t>(batch) * Hv;
    p.part_ml = reinterpret_cast<float2 *>(ws + wl.part_ml);
    p.part_o = reinterpret_cast<float *>(ws + wl.part_o);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.err = err;
    p.B = batch;
    p.Hq = num_q_heads;
    p.Hkv = Hv;
    p.hshift = __builtin_ctz(static_cast<unsigned>(R));
    p.G = G;
    p.GP = (G + 1) & ~1;
    p.P = num_pages;
    p.S = page_size;
    p.NW = NW;
    p.sm_scale_log2 = sm_scale * 1.4426950408889634f;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_pdl(attn_plan_kernel, dim3(1), dim3(kPlanThreads), 0, st, seq_lens, page_indptr,
                               abort_mask, nnz, batch, Hv, page_size, tile, NW,
                               reinterpret_cast<int64_t *>(ws + wl.prefix), reinterpret_cast<int32_t *>(ws + wl.warp_req),
                               reinterpret_cast<int32_t *>(ws + wl.counters));
    if (e != cudaSuccess) return FKV_ERR_CUDA;
    // Every batch of up to 64 requests (whose rows the warps hold two per
    // lane) goes to the instance that may give units whole warps; the warps
    // decide from the live requests alone, so the schedule never depends on
    // aborted or empty requests.
    const bool aligned = FKV_ALIGNED_SCHEDULE && batch <= 64;
    const dim3 grid(NW);
    if (fp8 && two_warp)
        e = launch_attn<true, true>(aligned, grid, st, p, tmK, tmV);
    else if (fp8)
        e = launch_attn<true, false>(aligned, grid, st, p, tmK, tmV);
    else if (two_warp)
        e = launch_attn<false, true>(aligned, grid, st, p, tmK, tmV);
    else
        e = launch_attn<false, false>(aligned, grid, st, p, tmK, tmV);
    if (e != cudaSuccess) return FKV_ERR_CUDA;
    return FKV_OK;
}
