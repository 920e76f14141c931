"""Pools past 4 GiB: a batch whose pages sit at the top of a 5 GiB (FP8) or
10 GiB (BF16) K and V pool, so every byte offset the kernels form for its
pages exceeds 2^32.  Attention, the append and the integrity check are
compared with the oracle on the same logical cache held in a compact pool:
the oracle's results do not depend on where the pages sit (its page
permutation pin), so the compact pool's page c stands for the big pool's
page ``big_id(c)``."""
import numpy as np
import pytest

from fp8_paged_kv_decode_gb300 import workloads as W
from gpu_util import PagedCase, assert_close, dev

pytestmark = pytest.mark.gpu

P_BIG, HKV, S = 40960, 8, 128          # FP8 page: 8 x 128 x 128 B = 128 KiB; pool 5 GiB (BF16 10 GiB)


def _big_ids(p_small):
    """Compact page c -> a page near the top of the big pool (distinct, the
    last page included, 7 pages apart)."""
    ids = P_BIG - 1 - 7 * np.arange(p_small, dtype=np.int64)
    assert ids.min() * HKV * S * 128 > 2 ** 32
    return ids


def _big_pools(small_k, small_v, ids, fp8):
    import torch
    dt = torch.uint8 if fp8 else torch.bfloat16
    kb = torch.zeros((P_BIG, HKV, S, 128), dtype=dt, device="cuda")
    vb = torch.zeros((P_BIG, HKV, S, 128), dtype=dt, device="cuda")
    t = torch.from_numpy(ids).cuda()
    kb[t] = dev(small_k, dtype=None if fp8 else torch.bfloat16)
    vb[t] = dev(small_v, dtype=None if fp8 else torch.bfloat16)
    return kb, vb, t


@pytest.mark.parametrize("kv", ["fp8", "bf16"])
def test_attention_on_pages_past_4gib(orc, kv):
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    case = PagedCase(orc, B=4, Hq=32, Hkv=HKV, S=S, seq=[1, 700, 129, 2000], kv=kv, seed=91, spare=3)
    ids = _big_ids(case.P)
    kb, vb, _ = _big_pools(case.kc, case.vc, ids, case.fp8)
    q = dev(case.q, dtype=torch.bfloat16)
    out = torch.full((case.B, case.Hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = fkv.alloc_workspace(case.B, case.Hq, HKV, fkv.KV_FP8_E4M3 if case.fp8 else fkv.KV_BF16)
    big_indices = ids[case.indices].astype(np.int32)
    fkv.device_error(clear=True)
    fkv.paged_decode_attn(q, kb, vb, dev(case.indptr), dev(big_indices), dev(case.seq), case.sm, out, ws,
                          k_scale=dev(case.k_scale) if case.fp8 else None,
                          v_scale=dev(case.v_scale) if case.fp8 else None)
    torch.cuda.synchronize()
    assert fkv.device_error() == 0
    got = out.float().cpu().numpy().astype(np.float64)
    assert_close(got, case.oracle(orc), "attention over pages past 4 GiB (%s)" % kv)


@pytest.mark.parametrize("kv", ["fp8", "bf16"])
def test_append_and_check_on_pages_past_4gib(orc, kv):
    """The step's prologue in one launch on the big pool: every byte of the
    touched pages equals the oracle's append into the compact pool, and the
    mask equals the oracle's check over the big pool's tags."""
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    rng = np.random.default_rng(93)
    fp8 = kv == "fp8"
    p_small, N, B = 12, 96, 6
    ids = _big_ids(p_small)
    if fp8:
        kc0 = rng.integers(0, 256, (p_small, HKV, S, 128)).astype(np.uint8)
        vc0 = rng.integers(0, 256, (p_small, HKV, S, 128)).astype(np.uint8)
    else:
        kc0 = W.bf16_bits(rng.standard_normal((p_small, HKV, S, 128)).astype(np.float32))
        vc0 = W.bf16_bits(rng.standard_normal((p_small, HKV, S, 128)).astype(np.float32))
    small_slots = rng.choice(p_small * S, size=N, replace=False).astype(np.int64)
    small_slots[::11] = -1                                          # padding tokens
    small_slots[0] = 0                                              # first slot of the last page
    small_slots[1] = S - 1
    live = small_slots >= 0
    big_slots = np.where(live, ids[small_slots // S] * S + small_slots % S, -1).astype(np.int64)
    kf = (rng.standard_normal((N, HKV, 128)) * np.exp2(rng.integers(-6, 6, (N, HKV, 1)))).astype(np.float32)
    vf = rng.standard_normal((N, HKV, 128)).astype(np.float32)
    kn, vn = W.bf16_bits(kf), W.bf16_bits(vf)
    ks = np.float32([0.01, 0.02, 0.05, 0.1, 0.2, 0.5, 1.0, 2.0])
    vs = np.float32([0.03] * HKV)
    kc, vc = kc0.copy(), vc0.copy()
    if fp8:
        orc.kv_append_fp8(kn, vn, small_slots, ks, vs, kc, vc)
    else:
        orc.kv_append_bf16(kn, vn, small_slots, kc, vc)

    # the check: B requests over pages at the top of the pool, two stale
    tags = rng.integers(0, 2 ** 32, P_BIG, dtype=np.uint64).astype(np.uint32)
    npg = rng.integers(1, 5, B)
    indptr = np.concatenate([[0], np.cumsum(npg)]).astype(np.int32)
    indices = ids[rng.integers(0, p_small, indptr[-1])].astype(np.int32)
    indices[-1] = P_BIG - 1
    expected = tags[indices].copy()
    expected[2] ^= 1
    expected[-1] += np.uint32(1)
    want_mask = orc.kv_page_tag_check(tags, indptr, indices, expected)
    assert want_mask.any() and not want_mask.all()

    kb, vb, t = _big_pools(kc0, vc0, ids, fp8)
    mask = torch.full((B,), 7, dtype=torch.uint8, device="cuda")
    fkv.device_error(clear=True)
    args = (dev(kn, dtype=torch.bfloat16), dev(vn, dtype=torch.bfloat16), dev(big_slots))
    tail = (dev(tags), dev(indptr), dev(indices), dev(expected), mask)
    if fp8:
        fkv.kv_append_fp8_tag_check(*args, dev(ks), dev(vs), kb, vb, *tail)
    else:
        fkv.kv_append_bf16_tag_check(*args, kb, vb, *tail)
    torch.cuda.synchronize()
    assert fkv.device_error() == 0
    assert np.array_equal(mask.cpu().numpy(), want_mask)
    gk, gv = kb[t].cpu(), vb[t].cpu()
    if not fp8:
        gk, gv = gk.view(torch.int16), gv.view(torch.int16)
    assert np.array_equal(gk.numpy().view(kc.dtype), kc)
    assert np.array_equal(gv.numpy().view(vc.dtype), vc)
