"""The five workloads at full size, through the same calls and launch
configuration the benchmark times, checked against the oracle on the whole
batch: the oracle encodes every cached token and the step's token itself from
the bf16 source values (drawn by torch's generator), and every byte of both
pools must equal the GPU's; the abort mask is compared for every request; and
every (request, query head) row of the attention output is compared element
by element within the tolerance, aborted rows exactly zero.  The oracle's work
is split over the host's threads (tokens for the encode, rows for attention);
the split changes none of its arithmetic."""
import numpy as np
import pytest

import oracle_parallel as OP
from fp8_paged_kv_decode_gb300 import workloads as W
from gpu_util import assert_close, bf16_out, dev

pytestmark = pytest.mark.gpu

CASES = [("tiny_gqa4", "fp8"), ("tiny_gqa4", "bf16"), ("uniform_gqa8_8k", "fp8"), ("uniform_gqa8_8k", "bf16"),
         ("pages_shaped_64req", "fp8"), ("pages_shaped_64req", "bf16"), ("long_ctx_131k", "fp8"),
         ("integrity_256req", "fp8")]


def run_step(db, kv):
    """Populate the cache (bulk append), then one decode step: append the new
    token, check tags, attend.  Returns device tensors."""
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    wl = db.wl
    P, Hkv, S, D = db.pt.num_pages, wl.num_kv_heads, wl.page_size, wl.head_dim
    fp8 = kv == "fp8"
    dt = torch.uint8 if fp8 else torch.bfloat16
    k_cache = torch.zeros(P, Hkv, S, D, dtype=dt, device="cuda")
    v_cache = torch.zeros(P, Hkv, S, D, dtype=dt, device="cuda")
    ks, vs = dev(db.k_scale), dev(db.v_scale)
    if fp8:
        fkv.kv_append_fp8(db.k_src, db.v_src, db.slots_src, ks, vs, k_cache, v_cache)
        fkv.kv_append_fp8(db.k_new, db.v_new, db.slots_new, ks, vs, k_cache, v_cache)
    else:
        fkv.kv_append_bf16(db.k_src, db.v_src, db.slots_src, k_cache, v_cache)
        fkv.kv_append_bf16(db.k_new, db.v_new, db.slots_new, k_cache, v_cache)
    indptr, indices = dev(db.pt.indptr), dev(db.pt.indices)
    mask = torch.empty(wl.batch, dtype=torch.uint8, device="cuda")
    fkv.kv_page_tag_check(dev(db.pt.page_tags.view(np.int32)), indptr, indices,
                          dev(db.pt.expected_tags.view(np.int32)), mask)
    out = torch.full((wl.batch, wl.num_q_heads, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = fkv.alloc_workspace(wl.batch, wl.num_q_heads, Hkv, fkv.KV_FP8_E4M3 if fp8 else fkv.KV_BF16)
    fkv.paged_decode_attn(db.q, k_cache, v_cache, indptr, indices, dev(db.seq_lens), 1.0 / np.sqrt(D), out, ws,
                          k_scale=ks if fp8 else None, v_scale=vs if fp8 else None, abort_mask=mask)
    torch.cuda.synchronize()
    return k_cache, v_cache, mask, out


def _host_u16(t):
    """bf16 device tensor -> numpy uint16 bit patterns (a copy, no arithmetic)."""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _assert_pool_equal(got, want, what):
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got.reshape(-1) != want.reshape(-1))
        idx = np.unravel_index(bad[0], want.shape)
        raise AssertionError("%s: %d of %d elements differ from the oracle; first at [page %d][head %d][slot %d]"
                             "[dim %d]: got %#x want %#x" % (what, bad.size, want.size, *idx,
                                                             int(got[idx]), int(want[idx])))


@pytest.mark.parametrize("name,kv", CASES, ids=["%s-%s" % c for c in CASES])
def test_fullsize_whole_batch_parity(orc, name, kv):
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    wl = W.WORKLOADS[name]
    fkv.device_error(clear=True)
    db = W.device_batch(wl, "cuda")
    k_cache, v_cache, mask, out = run_step(db, kv)
    fp8 = kv == "fp8"
    # the abort mask over the whole batch is bit-exact
    want_mask = orc.kv_page_tag_check(db.pt.page_tags, db.pt.indptr, db.pt.indices, db.pt.expected_tags)
    assert np.array_equal(mask.cpu().numpy(), want_mask)
    assert (want_mask.sum() > 0) == (wl.stale_frac > 0)

    # the oracle's pools: every cached token and the step's token, encoded by the oracle
    P, Hkv, S, D = db.pt.num_pages, wl.num_kv_heads, wl.page_size, wl.head_dim
    slots = np.concatenate([db.slots_src.cpu().numpy(), db.slots_new.cpu().numpy()])
    k_tok = np.concatenate([_host_u16(db.k_src), _host_u16(db.k_new)])
    v_tok = np.concatenate([_host_u16(db.v_src), _host_u16(db.v_new)])
    if fp8:
        kc = np.zeros((P, Hkv, S, D), np.uint8)
        vc = np.zeros((P, Hkv, S, D), np.uint8)
        OP.append_fp8(orc, k_tok, v_tok, slots, db.k_scale, db.v_scale, kc, vc)
    else:
        kc = np.zeros((P, Hkv, S, D), np.uint16)
        vc = np.zeros((P, Hkv, S, D), np.uint16)
        OP.append_bf16(orc, k_tok, v_tok, slots, kc, vc)
    del k_tok, v_tok
    # every byte of both pools (written slots and untouched ones) equals the oracle's
    _assert_pool_equal(k_cache.cpu().numpy() if fp8 else _host_u16(k_cache), kc, "%s %s K pool" % (name, kv))
    _assert_pool_equal(v_cache.cpu().numpy() if fp8 else _host_u16(v_cache), vc, "%s %s V pool" % (name, kv))

    # every row of the attention output
    ref = OP.attention_rows(orc, _host_u16(db.q), kc, vc, db.pt.indptr, db.pt.indices, db.seq_lens,
                            1.0 / np.sqrt(D), k_scale=db.k_scale if fp8 else None,
                            v_scale=db.v_scale if fp8 else None, abort_mask=want_mask)
    got = bf16_out(out)
    assert np.isfinite(got).all()
    assert not got[want_mask.astype(bool)].any(), "aborted rows must be exactly zero"
    assert_close(got, ref, "%s %s, all %d rows" % (name, kv, wl.batch * wl.num_q_heads))
    assert fkv.device_error() == 0


def test_logit_spread_of_long_context_workload():
    """long_ctx_131k draws q ~ 4 N(0,1) so q.k / sqrt(128) has std ~4 (peaky softmax)."""
    import torch
    wl = W.WORKLOADS["long_ctx_131k"]
    db = W.device_batch(wl, "cuda", ctx=np.full(wl.batch, 4096))
    q = db.q.float()[:, 0::wl.group]                         # one q head per KV head
    k = db.k_src[:4096].float()                              # request 0, all KV heads
    s = torch.einsum("hd,thd->th", q[0], k) / np.sqrt(wl.head_dim)
    std = float(s.std())
    assert 3.5 < std < 4.5, std
