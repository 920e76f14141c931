"""The oracle's calls split over host threads, for full-size parity checks.

Test infrastructure.  Each call below runs the unchanged oracle function on
disjoint pieces of the work -- tokens for the append, (request, query head)
rows for attention -- from a thread pool; the oracle's C entry points release
the interpreter lock, so the pieces run in parallel.  Splitting changes no
arithmetic: every token's codes and every row's output come from one oracle
call over exactly the inputs the single-threaded call would use.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np


def host_threads() -> int:
    return max(1, os.cpu_count() or 1)


def append_fp8(orc, k_tokens, v_tokens, slots, k_scale, v_scale, k_cache, v_cache, threads=None):
    """orc.kv_append_fp8 over token chunks (every token has its own slot, so the
    chunks write disjoint bytes)."""
    n = int(np.asarray(slots).size)
    threads = threads or host_threads()
    bounds = np.linspace(0, n, min(n, threads * 4) + 1).astype(np.int64) if n else np.zeros(1, np.int64)

    def part(i):
        a, b = int(bounds[i]), int(bounds[i + 1])
        if b > a:
            orc.kv_append_fp8(k_tokens[a:b], v_tokens[a:b], slots[a:b], k_scale, v_scale, k_cache, v_cache)

    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(part, range(bounds.size - 1)))


def append_bf16(orc, k_tokens, v_tokens, slots, k_cache, v_cache, threads=None):
    n = int(np.asarray(slots).size)
    threads = threads or host_threads()
    bounds = np.linspace(0, n, min(n, threads * 4) + 1).astype(np.int64) if n else np.zeros(1, np.int64)

    def part(i):
        a, b = int(bounds[i]), int(bounds[i + 1])
        if b > a:
            orc.kv_append_bf16(k_tokens[a:b], v_tokens[a:b], slots[a:b], k_cache, v_cache)

    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(part, range(bounds.size - 1)))


def attention_rows(orc, q, k_cache, v_cache, indptr, indices, seq_lens, sm_scale, k_scale=None, v_scale=None,
                   abort_mask=None, threads=None):
    """Every [B][Hq] row of orc.paged_decode_attn, the rows split into pieces of
    about equal token count over host threads.  Returns float64 [B][Hq][D]."""
    B, Hq, D = q.shape
    threads = threads or host_threads()
    out = np.zeros((B, Hq, D), np.float64)
    seq = np.asarray(seq_lens, np.int64)
    live = np.ones(B, bool) if abort_mask is None else (np.asarray(abort_mask) == 0)
    cost = np.repeat(np.where(live, np.maximum(seq, 0), 0), Hq) + 1     # per flat row r * Hq + i
    target = max(1, int(cost.sum()) // (threads * 8))
    pieces, start, acc = [], 0, 0
    for x in range(cost.size):
        acc += int(cost[x])
        if acc >= target:
            pieces.append((start, x + 1))
            start, acc = x + 1, 0
    if start < cost.size:
        pieces.append((start, cost.size))
    flat = out.reshape(B * Hq, D)

    def part(ab):
        a, b = ab
        rows = np.arange(a, b, dtype=np.int32)
        flat[a:b] = orc.paged_decode_attn(q, k_cache, v_cache, indptr, indices, seq_lens, sm_scale,
                                          k_scale=k_scale, v_scale=v_scale, abort_mask=abort_mask, rows=rows)

    # the largest pieces first, so the last ones to finish are short
    pieces.sort(key=lambda ab: -int(cost[ab[0]:ab[1]].sum()))
    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(part, pieces))
    return out
