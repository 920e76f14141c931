"""kv_page_realloc on the GPU: tags, new tags and scrubbed pools against the
oracle; reallocation followed by the integrity check aborts exactly the old
holders."""
import numpy as np
import pytest

from fp8_paged_kv_decode_gb300 import workloads as W
from gpu_util import dev

pytestmark = pytest.mark.gpu


def _gpu_realloc(tags, pages, kc=None, vc=None, bf16=False):
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    t = dev(tags.view(np.int32))
    new = torch.zeros(len(pages), dtype=torch.int32, device="cuda")
    kt = vt = None
    if kc is not None:
        kt = dev(kc, dtype=torch.bfloat16) if bf16 else dev(kc)
        vt = dev(vc, dtype=torch.bfloat16) if bf16 else dev(vc)
    fkv.kv_page_realloc(t, dev(np.asarray(pages, np.int32)), new, kt, vt)
    torch.cuda.synchronize()
    out = [t.cpu().numpy().view(np.uint32), new.cpu().numpy().view(np.uint32)]
    if kc is not None:
        conv = (lambda x: x.view(torch.int16).cpu().numpy().view(np.uint16)) if bf16 else (lambda x: x.cpu().numpy())
        out += [conv(kt), conv(vt)]
    return out


@pytest.mark.parametrize("kv", ["fp8", "bf16"])
def test_realloc_matches_oracle(orc, kv):
    import fp8_paged_kv_decode_gb300 as fkv
    rng = np.random.default_rng(41)
    P, Hkv, S = 300, 8, 64
    tags = rng.integers(0, 2 ** 32, P, dtype=np.uint64).astype(np.uint32)
    tags[:5] = 0xFFFFFFFF
    pages = rng.choice(P, 40, replace=False).astype(np.int32)
    pages[0] = 2
    dt = np.uint8 if kv == "fp8" else np.uint16
    kc = rng.integers(0, 200, (P, Hkv, S, 128)).astype(dt)
    vc = rng.integers(0, 200, (P, Hkv, S, 128)).astype(dt)
    fkv.device_error(clear=True)
    gt, gn, gk, gv = _gpu_realloc(tags.copy(), pages, kc, vc, bf16=(kv == "bf16"))
    ot, ok_, ov = tags.copy(), kc.copy(), vc.copy()
    on = orc.kv_page_realloc(ot, pages, ok_, ov)
    assert np.array_equal(gt, ot) and np.array_equal(gn, on)
    assert np.array_equal(gk, ok_) and np.array_equal(gv, ov)
    assert fkv.device_error() == 0


def test_realloc_without_scrub_and_bad_ids(orc):
    import fp8_paged_kv_decode_gb300 as fkv
    tags = np.arange(10, dtype=np.uint32)
    pages = np.array([3, 10, -4, 7], np.int32)
    fkv.device_error(clear=True)
    gt, gn = _gpu_realloc(tags.copy(), pages)
    ot = tags.copy()
    on = orc.kv_page_realloc(ot, pages)
    assert np.array_equal(gt, ot) and np.array_equal(gn, on)
    assert fkv.device_error() & fkv.DEVERR_REALLOC_PAGE


def test_realloc_then_check_aborts_old_holders(orc):
    """The device-side lifecycle: pages move to new owners on the GPU and the
    next integrity check aborts exactly the requests still holding them."""
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    wl = W.WORKLOADS["integrity_256req"]
    rng = np.random.default_rng(wl.seed)
    seq = W.context_lengths(wl, rng) + 1
    import dataclasses
    pt = W.build_page_table(dataclasses.replace(wl, stale_frac=0.0), seq, rng)
    moved = np.sort(rng.choice(pt.indices, size=round(0.01 * pt.indices.size), replace=False)).astype(np.int32)
    t = dev(pt.page_tags.view(np.int32))
    new = torch.zeros(moved.size, dtype=torch.int32, device="cuda")
    mask = torch.zeros(wl.batch, dtype=torch.uint8, device="cuda")
    fkv.kv_page_realloc(t, dev(moved), new)
    fkv.kv_page_tag_check(t, dev(pt.indptr), dev(pt.indices), dev(pt.expected_tags.view(np.int32)), mask)
    torch.cuda.synchronize()
    live = pt.page_tags.copy()
    orc.kv_page_realloc(live, moved)
    want = orc.kv_page_tag_check(live, pt.indptr, pt.indices, pt.expected_tags)
    assert np.array_equal(mask.cpu().numpy(), want)
    assert 0 < want.sum() < wl.batch
