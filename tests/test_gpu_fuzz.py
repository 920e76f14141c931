"""Seeded random shapes and faults, GPU against the oracle.

Each case draws a batch size, a (query heads, KV heads) pair with group size
1..8, a page size, context lengths (including 0, 1, page and tile multiples
and their neighbours), a pool with spare pages, an abort mask from the
integrity check over partly stale tags, an occasional page id outside the
pool and an occasional malformed CSR row, then compares the abort mask bit
for bit and the attention output element-wise within the tolerance."""
import numpy as np
import pytest

from gpu_util import PagedCase, assert_close, bf16_out, dev

pytestmark = pytest.mark.gpu

N_CASES = 24


def draw(rng):
    G = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    S = int(rng.choice([16, 32, 64, 128]))
    B = int(rng.integers(1, 12))
    special = [0, 1, S - 1, S, S + 1, 63, 64, 65, 127, 128, 129]
    seq = [int(rng.choice(special)) if rng.random() < 0.4 else int(rng.integers(1, 3000)) for _ in range(B)]
    kv = "bf16" if rng.random() < 0.3 else "fp8"
    return B, G * Hkv, Hkv, S, seq, kv


@pytest.mark.parametrize("case_id", range(N_CASES))
def test_fuzz_against_oracle(orc, case_id):
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    rng = np.random.default_rng(9000 + case_id)
    B, Hq, Hkv, S, seq, kv = draw(rng)
    case = PagedCase(orc, B, Hq, Hkv, S, [max(s, 0) for s in seq], kv=kv, seed=9100 + case_id,
                     spare=int(rng.integers(0, 20)), extra_pages=int(rng.integers(0, 2)))
    seqa = case.seq.copy()
    ind = case.indices.copy()
    indptr = case.indptr.copy()
    # live tags with a few stale entries -> abort mask from the GPU check
    tags = rng.integers(0, 2 ** 32, case.P, dtype=np.uint64).astype(np.uint32)
    exp = tags[np.clip(ind, 0, case.P - 1)].copy()
    stale = rng.random(exp.size) < 0.02
    exp[stale] += np.uint32(1)
    if rng.random() < 0.3 and ind.size:
        ind[int(rng.integers(0, ind.size))] = case.P + int(rng.integers(0, 5))     # outside the pool
    if rng.random() < 0.2 and B > 1:
        r = int(rng.integers(1, B))
        indptr[r] = indptr[r + 1] + 1 if indptr[r + 1] + 1 <= ind.size else indptr[r]   # malformed row
    want_mask = orc.kv_page_tag_check(tags, indptr, ind, exp)
    mask = torch.zeros(B, dtype=torch.uint8, device="cuda")
    fkv.kv_page_tag_check(dev(tags.view(np.int32)), dev(indptr), dev(ind), dev(exp.view(np.int32)), mask)
    torch.cuda.synchronize()
    assert np.array_equal(mask.cpu().numpy(), want_mask)
    use_mask = want_mask if rng.random() < 0.7 else None
    ref = orc.paged_decode_attn(case.q, case.kc, case.vc, indptr, ind, seqa, case.sm, k_scale=case.k_scale,
                                v_scale=case.v_scale, abort_mask=use_mask)
    case.indptr = indptr
    got = bf16_out(case.gpu(abort_mask=use_mask, indices=ind))
    assert_close(got, ref, "fuzz case %d: B=%d Hq=%d Hkv=%d S=%d kv=%s seq=%s" % (case_id, B, Hq, Hkv, S, kv, seq))


N_MEDIUM = 12


@pytest.mark.parametrize("case_id", range(N_MEDIUM))
def test_fuzz_medium_batches(orc, case_id):
    """Seeded batches of 40 to 200 requests with short, ragged contexts: the
    even split scheduled from each warp's own reading of the requests' rows
    (up to 64 requests in one load, up to 128 in 32-request chunks) and from
    the plan kernel's table (beyond 128), with empty and aborted requests."""
    rng = np.random.default_rng(9500 + case_id)
    B = int(rng.integers(40, 201))
    G = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([2, 4, 8]))
    S = int(rng.choice([16, 32, 64, 128]))
    special = [0, 1, S - 1, S, S + 1, 63, 64, 65]
    seq = [int(rng.choice(special)) if rng.random() < 0.3 else int(rng.integers(1, 700)) for _ in range(B)]
    kv = "bf16" if rng.random() < 0.3 else "fp8"
    case = PagedCase(orc, B, G * Hkv, Hkv, S, seq, kv=kv, seed=9600 + case_id)
    abort = (rng.random(B) < 0.05).astype(np.uint8)
    got = bf16_out(case.gpu(abort_mask=abort))
    assert_close(got, case.oracle(orc, abort_mask=abort),
                 "medium fuzz %d: B=%d Hq=%d Hkv=%d S=%d kv=%s" % (case_id, B, G * Hkv, Hkv, S, kv))
