"""kv_append_fp8_tag_check / kv_append_bf16_tag_check on the GPU: the
decode step's append and the integrity check in one launch give the oracle's
pool bytes and abort mask bit for bit, and exactly what the two separate
calls give."""
import numpy as np
import pytest

from fp8_paged_kv_decode_gb300 import workloads as W
from gpu_util import dev

pytestmark = pytest.mark.gpu


def _tables(rng, P, B, faults=True):
    tags = rng.integers(0, 2 ** 32, P, dtype=np.uint64).astype(np.uint32)
    counts = rng.integers(0, 300, B)
    indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    nnz = int(indptr[-1])
    indices = rng.integers(0, P, nnz).astype(np.int32)
    expected = tags[indices].copy()
    if faults and nnz:
        j = rng.integers(0, nnz, max(1, nnz // 500))
        expected[j[::2]] += np.uint32(1)                         # stale tags
        indices[j[1::2]] = P + 3                                 # ids outside the pool
    return tags, indptr, indices, expected


def _run(orc, P, Hkv, S, N, B, seed, combined=True, faults=True, kv="fp8"):
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    rng = np.random.default_rng(seed)
    fp8 = kv == "fp8"
    if fp8:
        kc0 = rng.integers(0, 256, (P, Hkv, S, 128)).astype(np.uint8)
        vc0 = rng.integers(0, 256, (P, Hkv, S, 128)).astype(np.uint8)
    else:
        kc0 = W.bf16_bits(rng.standard_normal((P, Hkv, S, 128)).astype(np.float32))
        vc0 = W.bf16_bits(rng.standard_normal((P, Hkv, S, 128)).astype(np.float32))
    slots = rng.choice(P * S, size=N, replace=False).astype(np.int64) if N else np.zeros(0, np.int64)
    if N:
        slots[::13] = -1                                         # padding tokens
    kb = W.bf16_bits((rng.standard_normal((N, Hkv, 128)) * 3).astype(np.float32))
    vb = W.bf16_bits(rng.standard_normal((N, Hkv, 128)).astype(np.float32))
    ks = rng.uniform(0.002, 0.02, Hkv).astype(np.float32)
    vs = rng.uniform(0.002, 0.02, Hkv).astype(np.float32)
    tags, indptr, indices, expected = _tables(rng, P, B, faults)
    # the oracle: append, then check
    kc, vc = kc0.copy(), vc0.copy()
    if N:
        if fp8:
            orc.kv_append_fp8(kb, vb, slots, ks, vs, kc, vc)
        else:
            orc.kv_append_bf16(kb, vb, slots, kc, vc)
    want_mask = orc.kv_page_tag_check(tags, indptr, indices, expected)
    # the GPU
    cdt = None if fp8 else torch.bfloat16
    kt, vt = dev(kc0, dtype=cdt), dev(vc0, dtype=cdt)
    mask = torch.full((B,), 7, dtype=torch.uint8, device="cuda")
    new = (dev(kb, dtype=torch.bfloat16) if N else torch.zeros(0, Hkv, 128, dtype=torch.bfloat16, device="cuda"),
           dev(vb, dtype=torch.bfloat16) if N else torch.zeros(0, Hkv, 128, dtype=torch.bfloat16, device="cuda"),
           dev(slots) if N else torch.zeros(0, dtype=torch.int64, device="cuda"))
    args = new + ((dev(ks), dev(vs)) if fp8 else ()) + (kt, vt)
    ind = dev(indices if indices.size else np.zeros(1, np.int32))[:indices.size]
    exp = dev(expected.view(np.int32) if expected.size else np.zeros(1, np.int32))[:expected.size]
    tg = dev(tags.view(np.int32))
    fkv.device_error(clear=True)
    if combined:
        (fkv.kv_append_fp8_tag_check if fp8 else fkv.kv_append_bf16_tag_check)(*args, tg, dev(indptr), ind, exp,
                                                                               mask)
    else:
        (fkv.kv_append_fp8 if fp8 else fkv.kv_append_bf16)(*args)
        fkv.kv_page_tag_check(tg, dev(indptr), ind, exp, mask)
    torch.cuda.synchronize()
    host = (lambda t: t.cpu().numpy()) if fp8 else (lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16))
    return host(kt), host(vt), mask.cpu().numpy(), kc, vc, want_mask


@pytest.mark.parametrize("kv", ["fp8", "bf16"])
@pytest.mark.parametrize("P,Hkv,S,N,B", [(300, 8, 16, 256, 256), (64, 2, 64, 37, 5), (2000, 4, 32, 1000, 900),
                                         (50, 1, 128, 17, 1)])
def test_combined_equals_oracle_and_separate_calls(orc, P, Hkv, S, N, B, kv):
    import fp8_paged_kv_decode_gb300 as fkv
    seed = P + N + B
    gk, gv, gm, kc, vc, want = _run(orc, P, Hkv, S, N, B, seed, combined=True, kv=kv)
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc), "pool bytes differ from the oracle"
    assert np.array_equal(gm, want), "abort mask differs from the oracle"
    assert want.any() or B == 1
    sk, sv, sm, _, _, _ = _run(orc, P, Hkv, S, N, B, seed, combined=False, kv=kv)
    assert np.array_equal(gk, sk) and np.array_equal(gv, sv) and np.array_equal(gm, sm)
    assert fkv.device_error() == 0


@pytest.mark.parametrize("kv", ["fp8", "bf16"])
def test_check_only_and_append_only(orc, kv):
    """No tokens: the launch is the check alone.  An empty batch: the append alone."""
    gk, gv, gm, kc, vc, want = _run(orc, 100, 2, 16, 0, 40, seed=9, kv=kv)
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc) and np.array_equal(gm, want)
    gk, gv, gm, kc, vc, want = _run(orc, 100, 2, 16, 60, 0, seed=10, kv=kv)
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc) and gm.size == 0


def test_integrity_workload_step(orc):
    """The integrity workload's decode step: 256 appended tokens, 1% of pages
    stale; the mask matches the oracle and the appended slots hold the
    oracle's codes."""
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    wl = W.WORKLOADS["integrity_256req"]
    rng = np.random.default_rng(wl.seed)
    ctx = W.context_lengths(wl, rng)
    pt = W.build_page_table(wl, ctx + 1, rng)
    P, Hkv, S = pt.num_pages, wl.num_kv_heads, wl.page_size
    kb = W.bf16_bits(rng.standard_normal((wl.batch, Hkv, 128)).astype(np.float32))
    vb = W.bf16_bits(rng.standard_normal((wl.batch, Hkv, 128)).astype(np.float32))
    slots = W.slot_mapping(pt, S, np.arange(wl.batch), ctx)
    ks = np.full(Hkv, 0.01, np.float32)
    vs = np.full(Hkv, 0.008, np.float32)
    kt = torch.zeros(P, Hkv, S, 128, dtype=torch.uint8, device="cuda")
    vt = torch.zeros_like(kt)
    mask = torch.full((wl.batch,), 7, dtype=torch.uint8, device="cuda")
    fkv.kv_append_fp8_tag_check(dev(kb, dtype=torch.bfloat16), dev(vb, dtype=torch.bfloat16), dev(slots), dev(ks),
                                dev(vs), kt, vt, dev(pt.page_tags.view(np.int32)), dev(pt.indptr), dev(pt.indices),
                                dev(pt.expected_tags.view(np.int32)), mask)
    torch.cuda.synchronize()
    want = orc.kv_page_tag_check(pt.page_tags, pt.indptr, pt.indices, pt.expected_tags)
    assert np.array_equal(mask.cpu().numpy(), want) and 0 < want.sum() < wl.batch
    kc = np.zeros((P, Hkv, S, 128), np.uint8)
    vc = np.zeros_like(kc)
    orc.kv_append_fp8(kb, vb, slots, ks, vs, kc, vc)
    assert np.array_equal(kt.cpu().numpy(), kc) and np.array_equal(vt.cpu().numpy(), vc)


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_combined(orc, seed):
    """Random pool sizes, head counts, page sizes, token and request counts
    and injected faults (every fourth seed on a BF16 cache): the one-launch
    call matches the oracle and the two separate calls bit for bit.  (Zero
    tokens or zero requests: test_check_only_and_append_only.)"""
    rng = np.random.default_rng(900 + seed)
    S = int(rng.choice([16, 32, 64, 128]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    P = int(rng.integers(4, 400))
    N = int(rng.integers(0, min(P * S, 600) + 1))
    B = int(rng.integers(0, 300))
    if N == 0 and B == 0:
        B = 1
    kv = "bf16" if seed % 4 == 3 else "fp8"
    gk, gv, gm, kc, vc, want = _run(orc, P, Hkv, S, N, B, seed=1000 + seed, combined=True, faults=bool(seed % 3),
                                    kv=kv)
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc), "pool bytes differ from the oracle"
    assert np.array_equal(gm, want), "abort mask differs from the oracle"
    sk, sv, sm, _, _, _ = _run(orc, P, Hkv, S, N, B, seed=1000 + seed, combined=False, faults=bool(seed % 3),
                               kv=kv)
    assert np.array_equal(gk, sk) and np.array_equal(gv, sv) and np.array_equal(gm, sm)


def test_small_integrity_step_after_one_launch_prologue(orc):
    """The first 8 requests of the integrity workload (no stale page), step
    after step: the append-and-check launch, then attention.  In this shape a
    warp whose part of a unit ends one tile before its range end can be the
    last of the unit's parts to arrive, and then owes the unit's merge in the
    middle of its range (which it performs at its range end).  Every step's
    rows must match the oracle on the cache as it stands after that step's
    append."""
    import dataclasses
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    from gpu_util import assert_close, bf16_out
    wl = dataclasses.replace(W.WORKLOADS["integrity_256req"], stale_frac=0.0, batch=8)
    hb = W.host_batch(wl)
    P, Hkv, S, D = hb.pt.num_pages, wl.num_kv_heads, wl.page_size, wl.head_dim
    kc = np.zeros((P, Hkv, S, D), np.uint8)
    vc = np.zeros_like(kc)
    orc.kv_append_fp8(hb.k_src, hb.v_src, hb.slots_src, hb.k_scale, hb.v_scale, kc, vc)
    kt, vt = dev(kc), dev(vc)
    ks, vs = dev(hb.k_scale), dev(hb.v_scale)
    indptr, indices = dev(hb.pt.indptr), dev(hb.pt.indices)
    tags, exp = dev(hb.pt.page_tags.view(np.int32)), dev(hb.pt.expected_tags.view(np.int32))
    mask = torch.full((wl.batch,), 7, dtype=torch.uint8, device="cuda")
    q = dev(hb.q, dtype=torch.bfloat16)
    out = torch.empty(wl.batch, wl.num_q_heads, D, dtype=torch.bfloat16, device="cuda")
    ws = fkv.alloc_workspace(wl.batch, wl.num_q_heads, Hkv)
    rng = np.random.default_rng(77)
    sm = 1.0 / np.sqrt(D)
    fkv.device_error(clear=True)
    for step in range(3):
        kn = W.bf16_bits(rng.standard_normal((wl.batch, Hkv, D)).astype(np.float32))
        vn = W.bf16_bits(rng.standard_normal((wl.batch, Hkv, D)).astype(np.float32))
        fkv.kv_append_fp8_tag_check(dev(kn, dtype=torch.bfloat16), dev(vn, dtype=torch.bfloat16), dev(hb.slots_new),
                                    ks, vs, kt, vt, tags, indptr, indices, exp, mask)
        fkv.paged_decode_attn(q, kt, vt, indptr, indices, dev(hb.seq_lens), sm, out, ws, k_scale=ks, v_scale=vs,
                              abort_mask=mask)
        torch.cuda.synchronize()
        orc.kv_append_fp8(kn, vn, hb.slots_new, hb.k_scale, hb.v_scale, kc, vc)
        assert not mask.cpu().numpy().any()
        ref = orc.paged_decode_attn(hb.q, kc, vc, hb.pt.indptr, hb.pt.indices, hb.seq_lens, sm,
                                    k_scale=hb.k_scale, v_scale=hb.v_scale)
        assert_close(bf16_out(out), ref, "step %d" % step)
    assert np.array_equal(kt.cpu().numpy(), kc)
    assert fkv.device_error() == 0


@pytest.mark.parametrize("nnz", [0, 1, 255, 256, 511, 1023, 1024, 1025, 2047, 2048, 2049, 3000])
def test_small_tables_with_malformed_rows(orc, nnz):
    """Page tables of up to 8 requests whose sizes straddle multiples of the
    check blocks' strides (128 and 256 threads, four entries in flight each):
    masks of the stand-alone check and of the append-and-check launch equal
    the oracle's, with stale tags, ids outside the pool, a row whose bounds
    are reversed, and a last row that ends past the entries passed."""
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    rng = np.random.default_rng(7000 + nnz)
    P = 97
    B = int(rng.integers(1, 9))
    cuts = np.sort(rng.integers(0, nnz + 1, B - 1)) if B > 1 else np.zeros(0, np.int64)
    indptr = np.concatenate([[0], cuts, [nnz]]).astype(np.int32)
    tags = rng.integers(0, 2 ** 32, P, dtype=np.uint64).astype(np.uint32)
    indices = rng.integers(0, P, nnz).astype(np.int32)
    expected = tags[indices].copy()
    if nnz:
        j = rng.integers(0, nnz, 3)
        expected[j[0]] += np.uint32(1)                       # stale
        indices[j[1]] = P + 1                                # outside the pool
    variants = [("as drawn", indptr, indices, expected)]
    if B >= 3:
        bad = indptr.copy()
        bad[1] = bad[2] + 1                                  # row 0 ends after row 1 starts: row 1 reversed
        variants.append(("reversed row", bad, indices, expected))
    if nnz >= 2:
        variants.append(("last row past the entries", indptr, indices[:nnz - 1], expected[:nnz - 1]))
    for what, ip, ind_h, exp_h in variants:
        want = orc.kv_page_tag_check(tags, ip, ind_h, exp_h)
        tg = dev(tags.view(np.int32))
        ind = dev(ind_h if ind_h.size else np.zeros(1, np.int32))[:ind_h.size]
        exp = dev(exp_h.view(np.int32) if exp_h.size else np.zeros(1, np.int32))[:exp_h.size]
        m1 = torch.full((B,), 7, dtype=torch.uint8, device="cuda")
        m2 = torch.full((B,), 7, dtype=torch.uint8, device="cuda")
        fkv.kv_page_tag_check(tg, dev(ip), ind, exp, m1)
        kc = torch.zeros((P, 1, 16, 128), dtype=torch.uint8, device="cuda")
        none_bf = torch.zeros(0, 1, 128, dtype=torch.bfloat16, device="cuda")
        one = torch.ones(1, dtype=torch.float32, device="cuda")
        fkv.kv_append_fp8_tag_check(none_bf, none_bf, torch.zeros(0, dtype=torch.int64, device="cuda"), one, one,
                                    kc, kc.clone(), tg, dev(ip), ind, exp, m2)
        torch.cuda.synchronize()
        assert np.array_equal(m1.cpu().numpy(), want), (what, "stand-alone check")
        assert np.array_equal(m2.cpu().numpy(), want), (what, "append-and-check launch")
