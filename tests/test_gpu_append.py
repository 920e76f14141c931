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


@pytest.mark.parametrize("P,Hkv,S,N", [(64, 4, 16, 300),
                                       # a bulk write (20 504 blocks), with a ragged last group
                                       (2600, 8, 16, 41001)])
def test_append_fp8_bitexact_whole_pool(orc, P, Hkv, S, N):
    import fp8_paged_kv_decode_gb300 as fkv
    rng = np.random.default_rng(1 + N)
    slots = rng.choice(P * S, size=N, replace=False).astype(np.int64)
    slots[::17] = -1                                   # padding tokens
    outside = N > 1000
    if outside:                                        # slots past the pool: skipped and flagged
        slots[5] = P * S + 3
        slots[-2] = 2 * P * S
    kf = (rng.standard_normal((N, Hkv, 128)) * np.exp2(rng.integers(-8, 8, (N, Hkv, 1)))).astype(np.float32)
    vf = rng.standard_normal((N, Hkv, 128)).astype(np.float32)
    ks = np.resize(np.float32([0.003, 0.5, 1.0, 7.0]), Hkv)
    vs = np.resize(np.float32([0.01, 0.02, 0.03, 0.04]), Hkv)
    fkv.device_error(clear=True)
    gk, gv, kc, vc, kc0, _ = _run_fp8(orc, P, Hkv, S, kf, vf, slots, ks, vs)
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
    # bytes outside the written slots are untouched
    written = np.zeros(P * S, bool)
    written[slots[(slots >= 0) & (slots < P * S)]] = True
    untouched = ~written.reshape(P, S)
    assert np.array_equal(gk.transpose(0, 2, 1, 3)[untouched], kc0.transpose(0, 2, 1, 3)[untouched])
    assert fkv.device_error() == (fkv.DEVERR_APPEND_SLOT if outside else 0)


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


def _midpoint_rows(orc, rng, H):
    """Per KV head one (x, scale) pair with x/scale within two fp32 ulps of a
    midpoint between neighbouring e4m3 values; the head's 128-element row holds
    +-x * 2^j, j = -10..8, so each row lands near midpoints of several binades.
    Returns rows [2][H][128] (K, V) and scales [2][H]."""
    tab = orc.e4m3_decode_table()
    c = rng.integers(0, 126, (2, H))
    m = (tab[c] + tab[c + 1]) / 2
    x = W.bits_to_f32(W.bf16_bits(rng.uniform(0.0625, 256, (2, H)).astype(np.float32)))
    b0 = (x.astype(np.float64) / m).astype(np.float32)
    nudge = np.arange(H) % 5 - 2
    b = (b0.view(np.uint32).astype(np.int64) + nudge).astype(np.uint32).view(np.float32)
    d = np.arange(128)
    rows = (x[..., None] * np.exp2((d >> 1) % 19 - 10) * np.where(d & 1, -1.0, 1.0)).astype(np.float32)
    return rows, b


def test_append_fp8_division_near_midpoints(orc):
    """The fast path's reciprocal-and-correction division decides codes exactly
    where one fp32 ulp matters: quotients a few ulps from e4m3 midpoints."""
    rng = np.random.default_rng(5)
    H = 2048
    rows, b = _midpoint_rows(orc, rng, H)
    # the cases have teeth: an uncorrected quotient RN(|x| * RN(1/b)) flips codes
    corr = (rows.astype(np.float64) / b[..., None]).astype(np.float32)
    y = (1.0 / b.astype(np.float64)).astype(np.float32)
    unc = (np.abs(rows) * y[..., None]).astype(np.float32) * np.sign(rows)
    dif = corr != unc
    assert (orc.e4m3_encode_array(corr[dif]) != orc.e4m3_encode_array(unc[dif])).sum() > 1000
    kf, vf = rows[0][None], rows[1][None]                 # N = 1 token, H heads
    gk, gv, kc, vc, _, _ = _run_fp8(orc, 1, H, 16, kf, vf, np.array([5]), b[0], b[1])
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)


def test_append_fp8_division_fallback(orc):
    """Scales outside [2^-30, 2^30] and rows holding huge or infinite values go
    through IEEE division in the kernel; the codes are the same either way."""
    rng = np.random.default_rng(6)
    H = 16
    rows, b = _midpoint_rows(orc, rng, H)
    ks = b[0].copy()
    ks[:6] = np.float32([2.0 ** -31, 2.0 ** 31, 1e-40, 2.0 ** -30, 2.0 ** 30, 3e-39])
    kf = rows[0].copy()
    kf[:6] *= np.float32(2.0 ** -40)                      # keep quotients in e4m3 range for tiny scales
    kf[1] = rows[0][1] * np.float32(2.0 ** 40)
    kf[4] = rows[0][4] * np.float32(2.0 ** 30)
    vf = rows[1].copy()
    vf[7, 3] = np.inf                                     # thread with an Inf: whole chunk on IEEE division
    vf[8, 20] = np.float32(2.0 ** 65)                     # just above the fast path's limit
    vf[9, 40] = -np.float32(2.0 ** 64)                    # at the limit: fast path
    vf[10, 50] = np.float32(1e-42)                        # subnormal input
    gk, gv, kc, vc, _, _ = _run_fp8(orc, 1, H, 16, kf[None], vf[None], np.array([9]), ks, b[1])
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)


def test_append_fp8_all_bf16_patterns(orc):
    """Every bf16 bit pattern under a spread of scales; NaN inputs give a NaN
    code (either sign), everything else is bit-exact."""
    rng = np.random.default_rng(7)
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(512, 1, 128)
    H = 8
    kb = np.repeat(pats, H, axis=1)
    vb = kb[::-1].copy()
    ks = np.float32([1.0, 1.0 / 448, 0.0137, 3.0, 2.0 ** -30, 2.0 ** 31, 7.5e-3, 1e-39])
    vs = np.float32(rng.uniform(1e-3, 10, H))
    kf, vf = W.bits_to_f32(kb), W.bits_to_f32(vb)
    slots = np.arange(512, dtype=np.int64)
    gk, gv, kc, vc, _, _ = _run_fp8(orc, 32, H, 16, kf, vf, slots, ks, vs)
    for g, o, src in ((gk, kc, kf), (gv, vc, vf)):
        nan = np.isnan(src).reshape(32, 16, H, 128).transpose(0, 2, 1, 3)
        assert np.array_equal(g[~nan], o[~nan])
        assert np.all((g[nan] & 0x7F) == 0x7F) and np.all((o[nan] & 0x7F) == 0x7F)


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
