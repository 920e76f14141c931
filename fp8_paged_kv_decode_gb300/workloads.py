"""Seeded synthetic workloads shared by the tests, the smoke check and the bench.

This module only draws inputs: shapes, context lengths, page tables with
generation tags, and bf16 values.  It holds none of the method's arithmetic
(no quantisation, no attention, no tag comparison); both the CUDA path and the
CPU oracle consume what it produces.

The five workload shapes follow the problem statement of the write-ups on
Cloudflare's "Smaller, faster, safer: running Kimi and GLM at scale" (up to 64
concurrent decode requests over long contexts, an FP8-vs-BF16 comparison, and
a per-page generation tag that changes on reallocation):

  tiny_gqa4          4 req, 8 q / 2 kv heads, page 16, context U[1,300]
  uniform_gqa8_8k    32 req, 64 q / 8 kv heads, page 64, context 8192 (FP8 and BF16)
  pages_shaped_64req 64 req, 64 q / 8 kv heads, page 64, context lognormal
                     (median 16384, sigma 0.8) clipped to [512, 131072],
                     1% of K channels scaled x20
  long_ctx_131k      8 req x 131072, 32 q / 4 kv heads, page 64, Q ~ 4 N(0,1)
  integrity_256req   256 req x 4096 (+1 appended), 32 q / 8 kv heads, page 16,
                     1% of in-use pages reallocated (stale expected tags)

Context convention: ``ctx`` tokens are already in the cache; a decode step
appends one token at position ``ctx`` and attends over ``ctx + 1`` tokens.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

HEAD_DIM = 128


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    page_size: int
    ctx: str                 # "uniform:<lo>:<hi>", "fixed:<n>", "lognormal:<median>:<sigma>:<lo>:<hi>"
    q_std: float = 1.0
    k_outlier_frac: float = 0.0
    k_outlier_mult: float = 20.0
    stale_frac: float = 0.0
    pool_factor: float = 1.25
    pool_pages: int = 0      # fixed pool size (0: pool_factor x pages used)
    kv_dtypes: tuple = ("fp8",)
    head_dim: int = HEAD_DIM
    seed: int = 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


WORKLOADS = {
    "tiny_gqa4": Workload("tiny_gqa4", 4, 8, 2, 16, "uniform:1:300", pool_pages=256,
                          kv_dtypes=("fp8", "bf16"), seed=1001),
    "uniform_gqa8_8k": Workload("uniform_gqa8_8k", 32, 64, 8, 64, "fixed:8192",
                                kv_dtypes=("fp8", "bf16"), seed=1002),
    "pages_shaped_64req": Workload("pages_shaped_64req", 64, 64, 8, 64,
                                   "lognormal:16384:0.8:512:131072",
                                   k_outlier_frac=0.01, kv_dtypes=("fp8", "bf16"), seed=1003),
    "long_ctx_131k": Workload("long_ctx_131k", 8, 32, 4, 64, "fixed:131072", q_std=4.0, seed=1004),
    "integrity_256req": Workload("integrity_256req", 256, 32, 8, 16, "fixed:4096",
                                 stale_frac=0.01, seed=1005),
}


def context_lengths(wl: Workload, rng: np.random.Generator) -> np.ndarray:
    """Tokens already cached per request (before the decode step's append)."""
    kind, *a = wl.ctx.split(":")
    if kind == "uniform":
        lo, hi = int(a[0]), int(a[1])
        return rng.integers(lo, hi + 1, size=wl.batch).astype(np.int64)
    if kind == "fixed":
        return np.full(wl.batch, int(a[0]), dtype=np.int64)
    if kind == "lognormal":
        med, sig, lo, hi = float(a[0]), float(a[1]), int(a[2]), int(a[3])
        x = rng.lognormal(mean=np.log(med), sigma=sig, size=wl.batch)
        return np.clip(np.rint(x), lo, hi).astype(np.int64)
    raise ValueError(wl.ctx)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 samples to bf16 (nearest, ties to even) and return the
    16-bit patterns.  Only used to draw bf16 inputs."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns back to float32 values (exact widening)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


class PagePool:
    """Host page allocator with a 32-bit generation tag per physical page.

    Every allocation of a page changes its tag (+1 modulo 2^32), so a stale
    (page, tag) pair held by a request whose page was reallocated no longer
    matches the live tag."""

    def __init__(self, num_pages: int, rng: np.random.Generator):
        self.num_pages = int(num_pages)
        self.tags = rng.integers(0, 2 ** 32, size=self.num_pages, dtype=np.uint64).astype(np.uint32)
        self.free = [int(p) for p in rng.permutation(self.num_pages)]

    def alloc(self, n: int):
        if n > len(self.free):
            raise MemoryError("page pool exhausted")
        ids = np.array([self.free.pop() for _ in range(n)], dtype=np.int32)
        self.tags[ids] = self.tags[ids] + np.uint32(1)     # uint32 wraps
        return ids, self.tags[ids].copy()

    def release(self, ids):
        self.free.extend(int(p) for p in ids)

    def reallocate(self, ids):
        """Pages released and handed straight to a new owner: they stay in use,
        their tags move on, and the old holders' expected tags go stale."""
        ids = np.asarray(ids, dtype=np.int64)
        self.tags[ids] = self.tags[ids] + np.uint32(1)


@dataclass
class PageTable:
    indptr: np.ndarray        # int32 [B+1]
    indices: np.ndarray       # int32 [nnz]
    expected_tags: np.ndarray # uint32 [nnz]
    page_tags: np.ndarray     # uint32 [P]  live tags
    num_pages: int
    stale_pages: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))


def build_page_table(wl: Workload, tokens: np.ndarray, rng: np.random.Generator) -> PageTable:
    """Allocate ceil(tokens/S) pages per request from a shuffled pool and record
    the (page, tag) pairs each request expects; then reallocate a seeded
    ``stale_frac`` of the in-use pages so their holders' tags are stale."""
    S = wl.page_size
    npages = (np.asarray(tokens, dtype=np.int64) + S - 1) // S
    used = int(npages.sum())
    P = wl.pool_pages if wl.pool_pages else int(np.ceil(wl.pool_factor * used))
    P = max(P, used)
    pool = PagePool(P, rng)
    indptr = np.zeros(wl.batch + 1, dtype=np.int32)
    indptr[1:] = np.cumsum(npages)
    indices = np.zeros(used, dtype=np.int32)
    expected = np.zeros(used, dtype=np.uint32)
    for r in range(wl.batch):
        ids, tags = pool.alloc(int(npages[r]))
        indices[indptr[r]:indptr[r + 1]] = ids
        expected[indptr[r]:indptr[r + 1]] = tags
    stale = np.zeros(0, dtype=np.int32)
    if wl.stale_frac > 0 and used > 0:
        n_stale = int(round(wl.stale_frac * used))
        stale = np.sort(rng.choice(indices, size=n_stale, replace=False)).astype(np.int32)
        pool.reallocate(stale)
    return PageTable(indptr, indices, expected, pool.tags.copy(), P, stale)


def slot_mapping(pt: PageTable, page_size: int, req: np.ndarray, pos: np.ndarray) -> np.ndarray:
    """Flat slot (page * S + offset) of token ``pos`` of request ``req``."""
    req = np.asarray(req, dtype=np.int64)
    pos = np.asarray(pos, dtype=np.int64)
    page = pt.indices[pt.indptr[req] + pos // page_size].astype(np.int64)
    return page * page_size + pos % page_size


def prefill_slots(pt: PageTable, page_size: int, ctx: np.ndarray) -> np.ndarray:
    """Slots of every cached token, request-major (token order of the K/V source)."""
    req = np.repeat(np.arange(ctx.size), ctx)
    starts = np.concatenate([[0], np.cumsum(ctx)[:-1]])
    pos = np.arange(int(ctx.sum())) - np.repeat(starts, ctx)
    return slot_mapping(pt, page_size, req, pos)


def outlier_channels(wl: Workload, rng: np.random.Generator) -> np.ndarray:
    """Distinct (kv_head, dim) K channels scaled by ``k_outlier_mult``."""
    n = int(round(wl.k_outlier_frac * wl.num_kv_heads * wl.head_dim))
    if n == 0:
        return np.zeros((0, 2), dtype=np.int64)
    flat = rng.choice(wl.num_kv_heads * wl.head_dim, size=n, replace=False)
    return np.stack([flat // wl.head_dim, flat % wl.head_dim], axis=1)


@dataclass
class HostBatch:
    """A whole workload on the host (small shapes only)."""
    wl: Workload
    ctx: np.ndarray           # int64 [B] cached tokens before the step
    seq_lens: np.ndarray      # int32 [B] = ctx + 1 (tokens attended after the append)
    pt: PageTable
    q: np.ndarray             # uint16 bf16 [B][Hq][D]
    k_src: np.ndarray         # uint16 bf16 [Ntok][Hkv][D] cached tokens, request-major
    v_src: np.ndarray
    slots_src: np.ndarray     # int64 [Ntok]
    k_new: np.ndarray         # uint16 bf16 [B][Hkv][D] the step's new token
    v_new: np.ndarray
    slots_new: np.ndarray     # int64 [B]
    k_scale: np.ndarray       # float32 [Hkv]
    v_scale: np.ndarray


def scale_from_amax(amax: np.ndarray) -> np.ndarray:
    """Per-KV-head scale the caller calibrates once: fl32(amax / 448), 1 when
    amax is 0 (448 is the largest finite e4m3 magnitude)."""
    a = np.asarray(amax, dtype=np.float32)
    s = (a / np.float32(448.0)).astype(np.float32)
    return np.where(a > 0, s, np.float32(1.0)).astype(np.float32)


def host_batch(wl: Workload, seed: int | None = None, ctx: np.ndarray | None = None) -> HostBatch:
    rng = np.random.default_rng(wl.seed if seed is None else seed)
    if ctx is None:
        ctx = context_lengths(wl, rng)
    ctx = np.asarray(ctx, dtype=np.int64)
    seq = ctx + 1
    pt = build_page_table(wl, seq, rng)
    Hkv, D = wl.num_kv_heads, wl.head_dim
    ntok = int(ctx.sum())
    q = bf16_bits(wl.q_std * rng.standard_normal((wl.batch, wl.num_q_heads, D), dtype=np.float32))
    kf = rng.standard_normal((ntok, Hkv, D), dtype=np.float32)
    vf = rng.standard_normal((ntok, Hkv, D), dtype=np.float32)
    kn = rng.standard_normal((wl.batch, Hkv, D), dtype=np.float32)
    vn = rng.standard_normal((wl.batch, Hkv, D), dtype=np.float32)
    for h, d in outlier_channels(wl, rng):
        kf[:, h, d] *= wl.k_outlier_mult
        kn[:, h, d] *= wl.k_outlier_mult
    k_src, v_src = bf16_bits(kf), bf16_bits(vf)
    k_amax = np.abs(bits_to_f32(k_src)).max(axis=(0, 2)) if ntok else np.zeros(Hkv, np.float32)
    v_amax = np.abs(bits_to_f32(v_src)).max(axis=(0, 2)) if ntok else np.zeros(Hkv, np.float32)
    return HostBatch(
        wl=wl, ctx=ctx, seq_lens=seq.astype(np.int32), pt=pt, q=q,
        k_src=k_src, v_src=v_src, slots_src=prefill_slots(pt, wl.page_size, ctx),
        k_new=bf16_bits(kn), v_new=bf16_bits(vn),
        slots_new=slot_mapping(pt, wl.page_size, np.arange(wl.batch), ctx),
        k_scale=scale_from_amax(k_amax), v_scale=scale_from_amax(v_amax))


def shard_requests(batch: int, rank: int, world: int) -> np.ndarray:
    """Requests owned by ``rank`` when a batch is split across replicas:
    contiguous, near-equal blocks; together they cover every request once."""
    bounds = [(batch * i) // world for i in range(world + 1)]
    return np.arange(bounds[rank], bounds[rank + 1], dtype=np.int64)


# ----------------------------------------------------------------------------
# full-size workloads drawn on the GPU
# ----------------------------------------------------------------------------
@dataclass
class DeviceBatch:
    """A workload whose bulk values are drawn on the GPU with a seeded torch
    generator (host draws for shapes, lengths and the page table)."""
    wl: Workload
    ctx: np.ndarray
    seq_lens: np.ndarray
    pt: PageTable
    tok_off: np.ndarray       # int64 [B] first row of each request in k_src / v_src
    q: object                 # torch bf16 [B][Hq][D]
    k_src: object             # torch bf16 [Ntok][Hkv][D]
    v_src: object
    slots_src: object         # torch int64 [Ntok]
    k_new: object             # torch bf16 [B][Hkv][D]
    v_new: object
    slots_new: object         # torch int64 [B]
    k_scale: np.ndarray       # float32 [Hkv]
    v_scale: np.ndarray


def _randn_bf16(torch, shape, gen, device, std=1.0, outliers=None, mult=1.0, chunk_rows=1 << 18):
    """N(0, std^2) samples rounded to bf16, drawn in row chunks (bounded fp32 scratch);
    ``outliers`` (kv_head, dim) columns are multiplied by ``mult`` before rounding."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    rows = shape[0]
    for a in range(0, rows, chunk_rows):
        b = min(rows, a + chunk_rows)
        x = torch.randn((b - a,) + tuple(shape[1:]), generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        if outliers is not None:
            for h, d in outliers:
                x[:, int(h), int(d)] *= mult
        out[a:b] = x.to(torch.bfloat16)
    return out


def device_batch(wl: Workload, device, seed: int | None = None, ctx: np.ndarray | None = None) -> DeviceBatch:
    import torch
    seed = wl.seed if seed is None else seed
    rng = np.random.default_rng(seed)
    if ctx is None:
        ctx = context_lengths(wl, rng)
    ctx = np.asarray(ctx, dtype=np.int64)
    seq = ctx + 1
    pt = build_page_table(wl, seq, rng)
    outl = outlier_channels(wl, rng)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    Hkv, D = wl.num_kv_heads, wl.head_dim
    ntok = int(ctx.sum())
    q = _randn_bf16(torch, (wl.batch, wl.num_q_heads, D), gen, device, std=wl.q_std)
    k_src = _randn_bf16(torch, (ntok, Hkv, D), gen, device, outliers=outl, mult=wl.k_outlier_mult)
    v_src = _randn_bf16(torch, (ntok, Hkv, D), gen, device)
    k_new = _randn_bf16(torch, (wl.batch, Hkv, D), gen, device, outliers=outl, mult=wl.k_outlier_mult)
    v_new = _randn_bf16(torch, (wl.batch, Hkv, D), gen, device)
    if ntok:
        k_amax = k_src.abs().amax(dim=(0, 2)).float().cpu().numpy()
        v_amax = v_src.abs().amax(dim=(0, 2)).float().cpu().numpy()
    else:
        k_amax = v_amax = np.zeros(Hkv, np.float32)
    tok_off = np.concatenate([[0], np.cumsum(ctx)[:-1]]).astype(np.int64)
    return DeviceBatch(
        wl=wl, ctx=ctx, seq_lens=seq.astype(np.int32), pt=pt, tok_off=tok_off, q=q, k_src=k_src, v_src=v_src,
        slots_src=torch.from_numpy(prefill_slots(pt, wl.page_size, ctx)).to(device),
        k_new=k_new, v_new=v_new,
        slots_new=torch.from_numpy(slot_mapping(pt, wl.page_size, np.arange(wl.batch), ctx)).to(device),
        k_scale=scale_from_amax(k_amax), v_scale=scale_from_amax(v_amax))


@dataclass
class CompactRequests:
    """Selected requests of a batch, re-indexed onto a compact page pool so a
    CPU check can rebuild their cache without the whole pool: page ``j`` of the
    compact pool is original page ``orig_pages[j]``."""
    reqs: np.ndarray
    q: np.ndarray             # uint16 bf16 [n][Hq][D]
    k_tokens: np.ndarray      # uint16 bf16 [Ntok'][Hkv][D] all cached + new tokens of the requests
    v_tokens: np.ndarray
    slots: np.ndarray         # int64 [Ntok'] compact slots
    indptr: np.ndarray
    indices: np.ndarray       # compact page ids
    seq_lens: np.ndarray
    orig_pages: np.ndarray    # int64 [n_pages]
    num_pages: int


def compact_requests(db: DeviceBatch, reqs) -> CompactRequests:
    import torch
    reqs = np.asarray(reqs, dtype=np.int64)
    S = db.wl.page_size
    orig, indptr, ks, vs, slots = [], [0], [], [], []
    for r in reqs:
        pages = db.pt.indices[db.pt.indptr[r]:db.pt.indptr[r + 1]].astype(np.int64)
        base = len(orig)
        orig.extend(pages.tolist())
        indptr.append(indptr[-1] + pages.size)
        a, n = int(db.tok_off[r]), int(db.ctx[r])
        k = torch.cat([db.k_src[a:a + n], db.k_new[r:r + 1]]).view(torch.int16).cpu().numpy().view(np.uint16)
        v = torch.cat([db.v_src[a:a + n], db.v_new[r:r + 1]]).view(torch.int16).cpu().numpy().view(np.uint16)
        ks.append(k)
        vs.append(v)
        pos = np.arange(n + 1)
        slots.append((base + pos // S) * S + pos % S)
    q = db.q[torch.from_numpy(reqs).to(db.q.device)].view(torch.int16).cpu().numpy().view(np.uint16)
    n_pages = len(orig)
    return CompactRequests(
        reqs=reqs, q=q, k_tokens=np.concatenate(ks), v_tokens=np.concatenate(vs), slots=np.concatenate(slots),
        indptr=np.array(indptr, np.int32), indices=np.arange(n_pages, dtype=np.int32),
        seq_lens=db.seq_lens[reqs].astype(np.int32), orig_pages=np.array(orig, np.int64), num_pages=n_pages)


def subset_batch(db: DeviceBatch, n: int) -> DeviceBatch:
    """The first ``n`` requests of a batch, same pool and page ids."""
    if not 0 <= n <= db.wl.batch:
        raise ValueError("subset of %d requests from a batch of %d" % (n, db.wl.batch))
    pt = db.pt
    nnz = int(pt.indptr[n])
    ntok = int(db.ctx[:n].sum())
    sub_pt = PageTable(pt.indptr[:n + 1].copy(), pt.indices[:nnz].copy(), pt.expected_tags[:nnz].copy(),
                       pt.page_tags, pt.num_pages, pt.stale_pages)
    wl = Workload(**{**db.wl.__dict__, "name": "%s[:%d]" % (db.wl.name, n), "batch": n})
    return DeviceBatch(wl=wl, ctx=db.ctx[:n].copy(), seq_lens=db.seq_lens[:n].copy(), pt=sub_pt,
                       tok_off=db.tok_off[:n].copy(), q=db.q[:n], k_src=db.k_src[:ntok], v_src=db.v_src[:ntok],
                       slots_src=db.slots_src[:ntok], k_new=db.k_new[:n], v_new=db.v_new[:n],
                       slots_new=db.slots_new[:n], k_scale=db.k_scale, v_scale=db.v_scale)


def admitted(page_bytes: int, pages_per_request, budget_bytes: int) -> int:
    """How many requests, taken in order, fit a KV budget (whole pages)."""
    used, n = 0, 0
    for p in pages_per_request:
        if used + int(p) * page_bytes > budget_bytes:
            break
        used += int(p) * page_bytes
        n += 1
    return n


def share_prefix(pt: PageTable, prefix_pages: int) -> PageTable:
    """Every request with more than ``prefix_pages`` pages reads request 0's
    first ``prefix_pages`` pages (a shared prompt prefix) instead of its own;
    its expected tags for them are request 0's.  Request 0 must hold at least
    that many pages."""
    indptr = pt.indptr
    n0 = int(indptr[1] - indptr[0])
    if prefix_pages > n0:
        raise ValueError("request 0 holds fewer pages than the shared prefix")
    ind, exp = pt.indices.copy(), pt.expected_tags.copy()
    src = slice(int(indptr[0]), int(indptr[0]) + prefix_pages)
    for r in range(1, indptr.size - 1):
        a, b = int(indptr[r]), int(indptr[r + 1])
        if b - a > prefix_pages:
            ind[a:a + prefix_pages] = pt.indices[src]
            exp[a:a + prefix_pages] = pt.expected_tags[src]
    return PageTable(indptr.copy(), ind, exp, pt.page_tags, pt.num_pages, pt.stale_pages)
