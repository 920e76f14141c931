"""kv_page_tag_check on the GPU: bit-exact abort masks against the oracle."""
import json
import os

import numpy as np
import pytest

from fp8_paged_kv_decode_gb300 import workloads as W
from gpu_util import dev

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def gpu_check(tags, indptr, indices, expected):
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    B = len(indptr) - 1
    mask = torch.full((B,), 7, dtype=torch.uint8, device="cuda")
    ind = np.asarray(indices, np.int32)
    exp = np.asarray(expected, np.uint32)
    fkv.kv_page_tag_check(dev(np.asarray(tags, np.uint32).view(np.int32)), dev(np.asarray(indptr, np.int32)),
                          dev(ind if ind.size else np.zeros(1, np.int32))[:ind.size],
                          dev(exp.view(np.int32) if exp.size else np.zeros(1, np.int32))[:exp.size], mask)
    torch.cuda.synchronize()
    return mask.cpu().numpy()


def test_golden_cases(orc):
    with open(os.path.join(GOLDEN, "tag_check_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        got = gpu_check(c["page_tags"], c["page_indptr"], c["page_indices"], c["expected_tags"])
        assert got.tolist() == c["abort_mask"], c["name"]


@pytest.mark.parametrize("name", ["tiny_gqa4", "integrity_256req", "long_ctx_131k"])
def test_workload_masks_bitexact(orc, name):
    wl = W.WORKLOADS[name]
    rng = np.random.default_rng(wl.seed)
    seq = W.context_lengths(wl, rng) + 1
    pt = W.build_page_table(wl, seq, rng)
    got = gpu_check(pt.page_tags, pt.indptr, pt.indices, pt.expected_tags)
    want = orc.kv_page_tag_check(pt.page_tags, pt.indptr, pt.indices, pt.expected_tags)
    assert np.array_equal(got, want)
    if wl.stale_frac:
        assert 0 < want.sum() < wl.batch


def test_random_faults_bitexact(orc):
    """Host-injected faults: stale tags, reclaimed pages, ids outside the pool,
    duplicated pages, wrap-around, empty and malformed rows."""
    rng = np.random.default_rng(5)
    for trial in range(10):
        P, B = int(rng.integers(1, 500)), int(rng.integers(1, 300))
        tags = rng.integers(0, 2 ** 32, P, dtype=np.uint64).astype(np.uint32)
        tags[rng.integers(0, P, 3)] = 0xFFFFFFFF
        counts = rng.integers(0, 700, B)
        counts[rng.random(B) < 0.1] = 0
        indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        nnz = int(indptr[-1])
        indices = rng.integers(0, P, nnz).astype(np.int32)
        expected = tags[indices].copy()
        k = max(1, nnz // 1000)
        j = rng.integers(0, max(nnz, 1), k)
        if nnz:
            expected[j[: k // 2 + 1]] += np.uint32(1)                  # stale (wraps at 2^32)
            indices[j[k // 2:]] = rng.choice([-1, P, P + 5, -(2 ** 31)])   # outside the pool
        if B > 3:
            indptr_bad = indptr.copy()
            r = int(rng.integers(1, B))
            indptr_bad[r] = indptr_bad[r + 1] + 1 if indptr_bad[r + 1] + 1 <= nnz else indptr_bad[r]
            indptr = indptr_bad
        got = gpu_check(tags, indptr, indices, expected)
        want = orc.kv_page_tag_check(tags, indptr, indices, expected)
        assert np.array_equal(got, want), trial


def test_tag_bump_aborts_exactly_the_holders(orc):
    rng = np.random.default_rng(6)
    P, B = 128, 40
    tags = rng.integers(0, 2 ** 32, P, dtype=np.uint64).astype(np.uint32)
    counts = rng.integers(1, 20, B)
    indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    indices = rng.integers(0, P, int(indptr[-1])).astype(np.int32)
    expected = tags[indices].copy()
    assert not gpu_check(tags, indptr, indices, expected).any()
    pool = W.PagePool(P, rng)
    pool.tags = tags.copy()
    p = int(indices[5])
    pool.reallocate([p])
    got = gpu_check(pool.tags, indptr, indices, expected)
    want = np.array([p in indices[indptr[r]:indptr[r + 1]] for r in range(B)], np.uint8)
    assert np.array_equal(got, want)
