"""kv_append_fp8 / kv_append_bf16 on the GPU: bit-exact against the oracle over whole pools."""
import numpy as np
import pytest

from fp8_paged_kv_decode_gb300 import workloads as W
from gpu_util import dev

pytestmark = pytest.mark.gpu


def _run_fp8(orc, P, Hkv, S, kf, vf, slots, ks, vs, seed=0):
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    rng = np.random.default_rng(seed)
    kc0 = rng.integers(0, 256, (P, Hkv, S, 128)).astype(np.uint8)
    vc0 = rng.integers(0, 256, (P, Hkv, S, 128)).astype(np.uint8)
    kb, vb = W.bf16_bits(kf), W.bf16_bits(vf)
    kc, vc = kc0.copy(), vc0.copy()
    orc.kv_append_fp8(kb, vb, slots, ks, vs, kc, vc)
    kt, vt = dev(kc0), dev(vc0)
    fkv.kv_append_fp8(dev(kb, dtype=torch.bfloat16), dev(vb, dtype=torch.bfloat16), dev(np.asarray(slots, np.int64)),
                      dev(np.asarray(ks, np.float32)), dev(np.asarray(vs, np.float32)), kt, vt)
    torch.cuda.synchronize()
    return kt.cpu().numpy(), vt.cpu().numpy(), kc, vc, kc0, vc0


def test_append_fp8_bitexact_whole_pool(orc):
    import fp8_paged_kv_decode_gb300 as fkv
    rng = np.random.default_rng(1)
    P, Hkv, S, N = 64, 4, 16, 300
    slots = rng.choice(P * S, size=N, replace=False).astype(np.int64)
    slots[::17] = -1                                   # padding tokens
    kf = (rng.standard_normal((N, Hkv, 128)) * np.exp2(rng.integers(-8, 8, (N, Hkv, 1)))).astype(np.float32)
    vf = rng.standard_normal((N, Hkv, 128)).astype(np.float32)
    ks = np.float32([0.003, 0.5, 1.0, 7.0])
    vs = np.float32([0.01, 0.02, 0.03, 0.04])
    fkv.device_error(clear=True)
    gk, gv, kc, vc, kc0, _ = _run_fp8(orc, P, Hkv, S, kf, vf, slots, ks, vs)
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
    # bytes outside the written slots are untouched
    written = np.zeros(P * S, bool)
    written[slots[slots >= 0]] = True
    untouched = ~written.reshape(P, S)
    assert np.array_equal(gk.transpose(0, 2, 1, 3)[untouched], kc0.transpose(0, 2, 1, 3)[untouched])
    assert fkv.device_error() == 0


def test_append_fp8_special_values(orc):
    """Saturation, ties, subnormal codes, signed zero, +-Inf; NaN inputs give a NaN code."""
    vals = np.array([0.0, -0.0, 448.0, 449.0, 464.0, 465.0, 1e6, -1e6, np.inf, -np.inf, 2.0 ** -10, 3 * 2.0 ** -10,
                     2.0 ** -9, 15 * 2.0 ** -10, 1e-30, -1e-30, 0.5625, 0.59375, 1.0625, 240.0, 248.0, -232.0],
                    dtype=np.float32)
    x = np.resize(vals, 128).astype(np.float32)
    kf = np.stack([x, -x])[:, None, :]                 # N=2, Hkv=1
    vf = np.stack([x * 0.5, x])[:, None, :]
    gk, gv, kc, vc, _, _ = _run_fp8(orc, 2, 1, 16, kf, vf, np.array([3, 20]), np.float32([1.0]), np.float32([1.0]))
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
    # NaN: both sides must produce a NaN code (either sign)
    xn = np.full(128, np.nan, np.float32)
    gk, _, kc, _, _, _ = _run_fp8(orc, 1, 1, 16, xn[None, None, :], xn[None, None, :], np.array([0]),
                                  np.float32([1.0]), np.float32([1.0]))
    assert np.all((gk[0, 0, 0] & 0x7F) == 0x7F) and np.all((kc[0, 0, 0] & 0x7F) == 0x7F)


def test_append_fp8_division_rounding(orc):
    """Scales that make x/scale land near e4m3 midpoints: the fp32 division's
    rounding decides the code, both sides must take it identically."""
    rng = np.random.default_rng(2)
    N, Hkv = 64, 2
    kf = rng.uniform(-300, 300, (N, Hkv, 128)).astype(np.float32)
    vf = rng.uniform(-1, 1, (N, Hkv, 128)).astype(np.float32)
    ks = np.float32([1.0 / 3.0, 0.7])
    vs = np.float32([np.float32(1.0) / np.float32(448.0), 1e-3])
    gk, gv, kc, vc, _, _ = _run_fp8(orc, 8, Hkv, 16, kf, vf, np.arange(N, dtype=np.int64) + 16, ks, vs)
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)


def test_append_out_of_pool_slot_is_skipped_and_flagged(orc):
    import fp8_paged_kv_decode_gb300 as fkv
    fkv.device_error(clear=True)
    rng = np.random.default_rng(3)
    kf = rng.standard_normal((3, 1, 128)).astype(np.float32)
    gk, gv, kc, vc, kc0, _ = _run_fp8(orc, 2, 1, 16, kf, kf, np.array([5, 2 * 16 + 3, 31]), np.float32([0.1]),
                                      np.float32([0.1]))
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
    assert fkv.device_error() & fkv.DEVERR_APPEND_SLOT


def test_append_bf16_bitexact(orc):
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    rng = np.random.default_rng(4)
    P, Hkv, S, N = 16, 2, 32, 100
    slots = rng.choice(P * S, size=N, replace=False).astype(np.int64)
    kb = W.bf16_bits(rng.standard_normal((N, Hkv, 128)).astype(np.float32))
    vb = W.bf16_bits(rng.standard_normal((N, Hkv, 128)).astype(np.float32))
    kc0 = rng.integers(0, 2 ** 16, (P, Hkv, S, 128)).astype(np.uint16)
    vc0 = rng.integers(0, 2 ** 16, (P, Hkv, S, 128)).astype(np.uint16)
    kc, vc = kc0.copy(), vc0.copy()
    orc.kv_append_bf16(kb, vb, slots, kc, vc)
    kt, vt = dev(kc0, dtype=torch.bfloat16), dev(vc0, dtype=torch.bfloat16)
    fkv.kv_append_bf16(dev(kb, dtype=torch.bfloat16), dev(vb, dtype=torch.bfloat16), dev(slots), kt, vt)
    torch.cuda.synchronize()
    assert np.array_equal(kt.view(torch.int16).cpu().numpy().view(np.uint16), kc)
    assert np.array_equal(vt.view(torch.int16).cpu().numpy().view(np.uint16), vc)


def test_append_empty_is_noop():
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    kc = torch.zeros(2, 1, 16, 128, dtype=torch.uint8, device="cuda")
    e = torch.empty(0, 1, 128, dtype=torch.bfloat16, device="cuda")
    s = torch.ones(1, dtype=torch.float32, device="cuda")
    fkv.kv_append_fp8(e, e, torch.empty(0, dtype=torch.int64, device="cuda"), s, s, kc, kc)
    torch.cuda.synchronize()
    assert int(kc.sum()) == 0
