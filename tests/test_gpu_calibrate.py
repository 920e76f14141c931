"""kv_calibrate_scales on the GPU: bit-exact scales against the oracle, and the
bulk prefill write (calibrate, then kv_append_fp8) bit-exact over a pool."""
import numpy as np
import pytest

from fp8_paged_kv_decode_gb300 import workloads as W
from gpu_util import dev

pytestmark = pytest.mark.gpu


def _gpu_scales(kb, vb):
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    Hkv = kb.shape[1]
    ks = torch.full((Hkv,), 7.0, dtype=torch.float32, device="cuda")
    vs = torch.full((Hkv,), 7.0, dtype=torch.float32, device="cuda")
    k = dev(kb, dtype=torch.bfloat16) if kb.size else torch.empty(kb.shape, dtype=torch.bfloat16, device="cuda")
    v = dev(vb, dtype=torch.bfloat16) if vb.size else torch.empty(vb.shape, dtype=torch.bfloat16, device="cuda")
    fkv.kv_calibrate_scales(k, v, ks, vs)
    torch.cuda.synchronize()
    return ks.cpu().numpy(), vs.cpu().numpy()


@pytest.mark.parametrize("n,Hkv", [(0, 8), (1, 8), (17, 8), (5000, 8), (3, 1), (70000, 1), (4099, 2), (1, 4),
                                   (9000, 4), (33, 16), (3000, 16), (500, 3), (2001, 5), (1000, 12)])
def test_scales_bitexact(orc, n, Hkv):
    """Head counts that divide the 16 rows of a block and ones that do not;
    each head's maximum sits at a different token, the last head's at the
    last token, and one head is all zeros."""
    rng = np.random.default_rng(51 + n + 1000 * Hkv)
    kf = (rng.standard_normal((n, Hkv, 128)) * np.exp2(rng.integers(-6, 6, (1, Hkv, 1)))).astype(np.float32)
    vf = rng.standard_normal((n, Hkv, 128)).astype(np.float32)
    if n:
        kf[:, Hkv // 2, :] = 0.0
        for h in range(Hkv):
            if h != Hkv // 2:
                kf[(n - 1 - 7 * h) % n, h, (5 * h) % 128] = 1.0e5 * (h + 1)
        vf[n - 1, Hkv - 1, 127] = -3.0e4
    kb, vb = W.bf16_bits(kf), W.bf16_bits(vf)
    gk, gv = _gpu_scales(kb, vb)
    ok, ov = orc.kv_calibrate_scales(kb, vb)
    assert np.array_equal(gk.view(np.uint32), ok.view(np.uint32))
    assert np.array_equal(gv.view(np.uint32), ov.view(np.uint32))


def test_bulk_prefill_write(orc):
    """Calibrate on the prompt, then write it whole: bytes match the oracle's
    own calibration and encoding over the whole pool."""
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    wl = W.WORKLOADS["tiny_gqa4"]
    hb = W.host_batch(wl)
    P, Hkv, S = hb.pt.num_pages, wl.num_kv_heads, wl.page_size
    ks = torch.empty(Hkv, dtype=torch.float32, device="cuda")
    vs = torch.empty(Hkv, dtype=torch.float32, device="cuda")
    k, v = dev(hb.k_src, dtype=torch.bfloat16), dev(hb.v_src, dtype=torch.bfloat16)
    kc = torch.zeros(P, Hkv, S, 128, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    fkv.kv_calibrate_scales(k, v, ks, vs)
    fkv.kv_append_fp8(k, v, dev(hb.slots_src), ks, vs, kc, vc)
    torch.cuda.synchronize()
    oks, ovs = orc.kv_calibrate_scales(hb.k_src, hb.v_src)
    okc = np.zeros((P, Hkv, S, 128), np.uint8)
    ovc = np.zeros_like(okc)
    orc.kv_append_fp8(hb.k_src, hb.v_src, hb.slots_src, oks, ovs, okc, ovc)
    assert np.array_equal(ks.cpu().numpy(), oks) and np.array_equal(vs.cpu().numpy(), ovs)
    assert np.array_equal(kc.cpu().numpy(), okc) and np.array_equal(vc.cpu().numpy(), ovc)


def test_full_size_scales_match_harness_calibration():
    """On the 64-request workload's 1.27 M-token prompt the device scales equal
    the harness's (torch amax, numpy division): the same definition, computed
    by different code."""
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    wl = W.WORKLOADS["pages_shaped_64req"]
    db = W.device_batch(wl, "cuda")
    Hkv = wl.num_kv_heads
    ks = torch.empty(Hkv, dtype=torch.float32, device="cuda")
    vs = torch.empty(Hkv, dtype=torch.float32, device="cuda")
    fkv.kv_calibrate_scales(db.k_src, db.v_src, ks, vs)
    torch.cuda.synchronize()
    assert np.array_equal(ks.cpu().numpy(), db.k_scale) and np.array_equal(vs.cpu().numpy(), db.v_scale)
