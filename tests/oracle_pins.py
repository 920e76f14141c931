"""Pins of the CPU oracle to facts fixed outside it.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with something the E4M3 format definition, IEEE
arithmetic, a library routine, a hand-derived case or a closed form fixes.
``test_oracle_pins.py`` runs them on the real oracle; ``test_oracle_mutants.py``
runs them on oracle builds with a planted mistake and requires each mistake
to be caught by at least one pin.
"""
from __future__ import annotations

import json
import os

import numpy as np

from fp8_paged_kv_decode_gb300.workloads import bf16_bits, bits_to_f32

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------------------
# independent references
# ----------------------------------------------------------------------------
def torch_e4m3_values() -> np.ndarray:
    """All 256 E4M3 code values as decoded by torch's float8_e4m3fn (an
    implementation independent of the oracle)."""
    import torch
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def positive_values() -> np.ndarray:
    """The 127 non-negative finite E4M3 values, index == code (0x00..0x7E)."""
    return torch_e4m3_values()[:127]


def nearest_even_encode(x: np.ndarray) -> np.ndarray:
    """Brute force: for each float32, the finite E4M3 code nearest in value;
    ties go to the code with an even mantissa; |x| > 448 and +-Inf saturate
    to +-448; NaN -> 0x7F with the sign bit kept."""
    x = np.asarray(x, dtype=np.float32)
    vals = positive_values()                       # ascending, code = index
    a = np.abs(x.astype(np.float64))
    sign = np.where(np.signbit(x), 0x80, 0x00).astype(np.uint8)
    out = np.zeros(x.shape, dtype=np.uint8)
    finite = np.isfinite(a) & (a <= 448.0)
    dist = np.abs(a[finite, None] - vals[None, :])   # exact in fp64
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    n_c = cand.sum(axis=1)
    first = cand.argmax(axis=1)
    last = 126 - cand[:, ::-1].argmax(axis=1)
    pick = np.where(n_c == 1, first, np.where(first % 2 == 0, first, last))
    out[finite] = pick.astype(np.uint8)
    out[np.isfinite(a) & (a > 448.0)] = 0x7E
    out[np.isinf(a)] = 0x7E
    out[np.isnan(a)] = 0x7F
    return out | sign


def encode_probe_points(seed: int = 7, n_random: int = 20000) -> np.ndarray:
    """Float32 probes: every E4M3 value, every midpoint between neighbours and
    the float32 values one ulp either side, the saturation region, zeros, and a
    log-uniform random spread over the format's range."""
    vals = positive_values()
    mids = (vals[:-1] + vals[1:]) / 2.0
    pts = [vals, mids, np.array([448.0, 456.0, 463.99, 464.0, 464.01, 480.0, 1e4, 3e38, 2 ** -10, 2 ** -11,
                                 1e-30, 1e-45, 0.0])]
    m32 = mids.astype(np.float32)
    pts += [np.nextafter(m32, np.float32(np.inf)), np.nextafter(m32, np.float32(-np.inf))]
    rng = np.random.default_rng(seed)
    pts.append(np.exp2(rng.uniform(-14.0, 9.5, n_random)))
    p = np.concatenate([np.asarray(a, dtype=np.float64) for a in pts]).astype(np.float32)
    return np.concatenate([p, -p])


# ----------------------------------------------------------------------------
# E4M3 format
# ----------------------------------------------------------------------------
def pin_e4m3_decode_landmarks(orc):
    t = orc.e4m3_decode_table()
    assert t[0x7E] == 448.0, "largest finite E4M3 magnitude is 448"
    assert t[0x08] == 2.0 ** -6, "smallest normal is 2^-6"
    assert t[0x07] == 7 * 2.0 ** -9, "largest subnormal is 7 * 2^-9"
    assert t[0x01] == 2.0 ** -9, "smallest subnormal is 2^-9"
    assert t[0x38] == 1.0, "exponent bias 7: 0x38 is 1.0"
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF]), "S.1111.111 is NaN"
    assert t[0x80] == 0.0 and np.signbit(t[0x80]), "0x80 is -0"
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0), "positive codes decode in increasing order"
    fin = t[np.isfinite(t)]
    assert np.unique(fin).size == 253, "253 distinct finite values"
    assert np.array_equal(t[0x80:0xFF], -t[0x00:0x7F]), "sign bit mirrors"


def pin_e4m3_decode_vs_torch(orc):
    t = orc.e4m3_decode_table()
    ref = torch_e4m3_values()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(t), nan)
    assert np.array_equal(t[~nan], ref[~nan])


def pin_e4m3_encode_nearest_even(orc):
    x = encode_probe_points()
    got = orc.e4m3_encode_array(x)
    want = nearest_even_encode(x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, "encode differs from nearest-even at x=%r (got %#x want %#x)" % (
        float(x[bad[0]]), int(got[bad[0]]), int(want[bad[0]]))


def pin_e4m3_encode_specials(orc):
    assert orc.e4m3_encode(float("inf")) == 0x7E and orc.e4m3_encode(float("-inf")) == 0xFE
    assert orc.e4m3_encode(float("nan")) & 0x7F == 0x7F
    assert orc.e4m3_encode(-0.0) == 0x80 and orc.e4m3_encode(0.0) == 0x00
    assert orc.e4m3_encode(1e30) == 0x7E and orc.e4m3_encode(-1e30) == 0xFE
    # ties in the subnormal range go to the even code
    assert orc.e4m3_encode(2.0 ** -10) == 0x00          # halfway 0 .. 2^-9
    assert orc.e4m3_encode(3 * 2.0 ** -10) == 0x02      # halfway 2^-9 .. 2*2^-9
    assert orc.e4m3_encode(15 * 2.0 ** -10) == 0x08     # halfway 7*2^-9 .. 2^-6 -> even 0x08


def pin_e4m3_encode_vs_torch(orc):
    import torch
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.uniform(-448, 448, 4000), rng.standard_normal(4000) * 4,
                        rng.standard_normal(2000) * 1e-2]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = orc.e4m3_encode_array(x)
    assert np.array_equal(got, ref), "encode differs from torch float8_e4m3fn for in-range values"


def pin_e4m3_roundtrip(orc):
    t = orc.e4m3_decode_table()
    for c in range(256):
        if np.isnan(t[c]):
            continue
        assert orc.e4m3_encode(t[c]) == c, "encode(decode(%#x)) != %#x" % (c, c)


# ----------------------------------------------------------------------------
# quantise-on-append
# ----------------------------------------------------------------------------
def pin_div_rn_f32(orc):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(3000) * np.exp2(rng.integers(-20, 20, 3000))).astype(np.float32)
    s = np.abs(rng.standard_normal(3000) * np.exp2(rng.integers(-20, 20, 3000))).astype(np.float32) + np.float32(1e-30)
    x = np.concatenate([x, np.float32([1.0, 3.0, 1e-38, 7.0, 448.0])])
    s = np.concatenate([s, np.float32([3.0, 7.0, 3.0, 1e30, 0.24])])
    want = (x / s).astype(np.float32)                    # numpy: IEEE binary32 division
    got = np.array([orc.div_rn_f32(float(a), float(b)) for a, b in zip(x, s)], dtype=np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def pin_append_placement(orc):
    P, Hkv, S, D = 6, 2, 16, 128
    rng = np.random.default_rng(5)
    k_cache = np.full((P, Hkv, S, D), 0xA5, dtype=np.uint8)
    v_cache = np.full((P, Hkv, S, D), 0x5A, dtype=np.uint8)
    slots = np.array([3 * S + 7, -1, 0, 5 * S + 15, P * S + 2], dtype=np.int64)   # -1: padding; last: outside pool
    kf = (rng.standard_normal((5, Hkv, D)) * 3).astype(np.float32)
    vf = (rng.standard_normal((5, Hkv, D)) * 3).astype(np.float32)
    kb, vb = bf16_bits(kf), bf16_bits(vf)
    ks = np.array([0.02, 0.5], dtype=np.float32)
    vs = np.array([0.01, 0.25], dtype=np.float32)
    orc.kv_append_fp8(kb, vb, slots, ks, vs, k_cache, v_cache)
    k_ref = np.full_like(k_cache, 0xA5)
    v_ref = np.full_like(v_cache, 0x5A)
    for n, slot in enumerate(slots):
        if slot < 0 or slot // S >= P:
            continue
        p, off = slot // S, slot % S
        for h in range(Hkv):
            k_ref[p, h, off] = nearest_even_encode((bits_to_f32(kb[n, h]) / ks[h]).astype(np.float32))
            v_ref[p, h, off] = nearest_even_encode((bits_to_f32(vb[n, h]) / vs[h]).astype(np.float32))
    assert np.array_equal(k_cache, k_ref) and np.array_equal(v_cache, v_ref)


def pin_append_bf16_placement(orc):
    """The BF16 cache stores each new token's bf16 bits unchanged at
    [page][head][offset]: K rows in the K pool, V rows in the V pool; padding
    slots (< 0) and slots past the pool write nothing; every other byte keeps
    its fill.  Expected pools are placed by hand with numpy indexing."""
    P, Hkv, S, D = 5, 3, 32, 128
    rng = np.random.default_rng(6)
    fill_k, fill_v = np.uint16(0xA5A5), np.uint16(0x5A5A)
    k_cache = np.full((P, Hkv, S, D), fill_k, dtype=np.uint16)
    v_cache = np.full((P, Hkv, S, D), fill_v, dtype=np.uint16)
    # first and last slot of the pool, a slot in the middle, padding, past the pool
    slots = np.array([0, 2 * S + 19, -7, P * S - 1, P * S, 4 * S + 1], dtype=np.int64)
    n = slots.size
    kb = bf16_bits((rng.standard_normal((n, Hkv, D)) * 5).astype(np.float32))
    vb = bf16_bits((rng.standard_normal((n, Hkv, D)) * 5).astype(np.float32))
    orc.kv_append_bf16(kb, vb, slots, k_cache, v_cache)
    k_ref = np.full_like(k_cache, fill_k)
    v_ref = np.full_like(v_cache, fill_v)
    written = 0
    for j, slot in enumerate(slots):
        if slot < 0 or slot >= P * S:
            continue
        p, off = int(slot) // S, int(slot) % S
        k_ref[p, :, off, :] = kb[j]
        v_ref[p, :, off, :] = vb[j]
        written += 1
    assert written == 4
    assert np.array_equal(k_cache, k_ref), "K rows land at [page][head][offset] of the K pool"
    assert np.array_equal(v_cache, v_ref), "V rows land at [page][head][offset] of the V pool"
    # the bf16 bits round-trip: the cache holds exactly the input values
    assert np.array_equal(bits_to_f32(k_cache[2, 1, 19]), bits_to_f32(kb[1, 1]))


def pin_append_saturates(orc):
    P, Hkv, S, D = 1, 1, 16, 128
    k = np.zeros((P, Hkv, S, D), np.uint8)
    v = np.zeros((P, Hkv, S, D), np.uint8)
    x = np.linspace(-2000, 2000, D).astype(np.float32)[None, None, :]
    b = bf16_bits(x)
    orc.kv_append_fp8(b, b, np.array([3]), np.float32([1.0]), np.float32([1.0]), k, v)
    xs = bits_to_f32(b).ravel()
    assert np.all(k[0, 0, 3][xs > 464] == 0x7E) and np.all(k[0, 0, 3][xs < -464] == 0xFE)


# ----------------------------------------------------------------------------
# integrity check
# ----------------------------------------------------------------------------
def pin_tag_check_golden(orc):
    with open(os.path.join(GOLDEN, "tag_check_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        got = orc.kv_page_tag_check(np.array(c["page_tags"], np.uint32), np.array(c["page_indptr"], np.int32),
                                    np.array(c["page_indices"], np.int32), np.array(c["expected_tags"], np.uint32))
        assert got.tolist() == c["abort_mask"], c["name"]


def pin_tag_check_bump_property(orc):
    """Reallocating page p (tag + 1) aborts exactly the requests that list p."""
    rng = np.random.default_rng(9)
    for trial in range(20):
        P, B = 64, 12
        tags = rng.integers(0, 2 ** 32, P, dtype=np.uint64).astype(np.uint32)
        counts = rng.integers(0, 9, B)
        indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        indices = rng.integers(0, P, int(counts.sum())).astype(np.int32)
        expected = tags[indices].copy()
        assert not orc.kv_page_tag_check(tags, indptr, indices, expected).any()
        p = int(rng.integers(0, P))
        live = tags.copy()
        live[p] = live[p] + np.uint32(1)
        got = orc.kv_page_tag_check(live, indptr, indices, expected)
        want = np.array([p in indices[indptr[r]:indptr[r + 1]] for r in range(B)], dtype=np.uint8)
        assert np.array_equal(got, want), trial


def pin_tag_check_page_range(orc):
    """Ids at or past the pool size abort even when the memory after the live
    tag array happens to hold the expected value."""
    tags = np.array([7, 7, 7, 7], np.uint32)          # pool of 2 pages; entries 2, 3 lie outside it
    got = orc.kv_page_tag_check(tags, np.array([0, 1, 2, 3], np.int32), np.array([0, 2, 3], np.int32),
                                np.array([7, 7, 7], np.uint32), num_pages=2)
    assert got.tolist() == [0, 1, 1]


def pin_realloc_aborts_exactly_old_holders(orc):
    """Reallocating pages (tag + 1, [GN]/[CF]) makes every request holding one
    of them fail the check, and a request that records the new tags passes."""
    rng = np.random.default_rng(31)
    P, B = 50, 10
    tags = rng.integers(0, 2 ** 32, P, dtype=np.uint64).astype(np.uint32)
    tags[3] = 0xFFFFFFFF
    counts = rng.integers(1, 8, B)
    indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    indices = rng.integers(0, P, int(indptr[-1])).astype(np.int32)
    indices[0] = 3
    expected = tags[indices].copy()
    moved = np.array([3, int(indices[5]), 17, P + 2, -1], np.int32)
    live = tags.copy()
    new = orc.kv_page_realloc(live, moved)
    for j, p in enumerate(moved):
        if 0 <= p < P:
            bumps = 1 + int((moved[:j] == p).sum())
            assert int(new[j]) == (int(tags[p]) + bumps) & 0xFFFFFFFF, "tag moves on by one per reallocation"
        else:
            assert new[j] == 0
    assert live[3] == 0, "0xFFFFFFFF wraps to 0"
    in_pool = moved[(moved >= 0) & (moved < P)]
    untouched = np.setdiff1d(np.arange(P), in_pool)
    assert np.array_equal(live[untouched], tags[untouched])
    got = orc.kv_page_tag_check(live, indptr, indices, expected)
    want = np.array([np.isin(indices[indptr[r]:indptr[r + 1]], in_pool).any() for r in range(B)], np.uint8)
    assert np.array_equal(got, want)
    # a new owner of page 17 that records the new tag passes
    ok = orc.kv_page_tag_check(live, np.array([0, 1], np.int32), np.array([17], np.int32),
                               np.array([new[2]], np.uint32))
    assert ok.tolist() == [0]


def pin_realloc_scrub_zeroes_listed_pages(orc):
    rng = np.random.default_rng(32)
    for dt in (np.uint8, np.uint16):
        kc = rng.integers(1, 200, (6, 2, 16, 128)).astype(dt)
        vc = rng.integers(1, 200, (6, 2, 16, 128)).astype(dt)
        k0, v0 = kc.copy(), vc.copy()
        tags = np.arange(6, dtype=np.uint32)
        orc.kv_page_realloc(tags, np.array([4, 1, 9], np.int32), kc, vc)
        for p in range(6):
            if p in (1, 4):
                assert not kc[p].any() and not vc[p].any()
            else:
                assert np.array_equal(kc[p], k0[p]) and np.array_equal(vc[p], v0[p])


def pin_calibration_scales(orc):
    """fl32(amax / 448) per KV head against numpy; zero heads give 1; one
    outlier decides its head; and the resulting codes reach 448 exactly."""
    rng = np.random.default_rng(33)
    N, Hkv, D = 257, 4, 128
    kf = rng.standard_normal((N, Hkv, D)).astype(np.float32)
    vf = (rng.standard_normal((N, Hkv, D)) * 0.01).astype(np.float32)
    kf[:, 2, :] = 0.0                       # all-zero heads
    vf[:, 3, :] = 0.0
    kf[100, 1, 7] = -3.0e4                  # one outlier
    kb, vb = bf16_bits(kf), bf16_bits(vf)
    ks, vs = orc.kv_calibrate_scales(kb, vb)
    for bits, got in ((kb, ks), (vb, vs)):
        amax = np.abs(bits_to_f32(bits)).max(axis=(0, 2))
        want = np.where(amax > 0, (amax / np.float32(448.0)).astype(np.float32), np.float32(1.0))
        assert np.array_equal(got.view(np.uint32), want.astype(np.float32).view(np.uint32))
    assert ks[2] == 1.0 and vs[3] == 1.0
    assert ks[1] == np.float32(np.float32(bits_to_f32(kb[100, 1, 7:8])[0] * -1) / np.float32(448.0))
    # quantizing with the calibrated scale maps each head's largest value to the largest code
    P = 1
    kc = np.zeros((P, Hkv, 16, D), np.uint8)
    vc = np.zeros((P, Hkv, 16, D), np.uint8)
    orc.kv_append_fp8(kb[100:101], vb[100:101], np.array([0]), ks, vs, kc, vc)
    assert kc[0, 1, 0, 7] == 0xFE           # -448


def pin_tag_check_malformed(orc):
    tags = np.array([1, 2], np.uint32)
    got = orc.kv_page_tag_check(tags, np.array([0, 2, 1], np.int32), np.array([0, 1], np.int32),
                                np.array([1, 2], np.uint32))
    assert got.tolist() == [0, 1], "a CSR row that ends before it starts aborts"
    got = orc.kv_page_tag_check(tags, np.array([0, 3], np.int32), np.array([0, 1], np.int32),
                                np.array([1, 2], np.uint32))
    assert got.tolist() == [1], "a CSR row past the index list aborts"


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------
def _rand_case(rng, B, Hq, Hkv, S, ctx, P=None, fp8=True, q_std=1.0):
    D = 128
    npages = (np.asarray(ctx) + S - 1) // S
    used = int(npages.sum())
    P = P or used + 3
    perm = rng.permutation(P)[:used].astype(np.int32)
    indptr = np.concatenate([[0], np.cumsum(npages)]).astype(np.int32)
    q = bf16_bits((rng.standard_normal((B, Hq, D)) * q_std).astype(np.float32))
    if fp8:
        codes = rng.integers(0, 256, (P, Hkv, S, D)).astype(np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0x3C                   # no NaN codes in the pool
        k, v = codes, rng.permutation(codes.ravel()).reshape(codes.shape)
        ks = (rng.uniform(0.001, 0.01, Hkv)).astype(np.float32)
        vs = (rng.uniform(0.001, 0.01, Hkv)).astype(np.float32)
    else:
        k = bf16_bits(rng.standard_normal((P, Hkv, S, D)).astype(np.float32))
        v = bf16_bits(rng.standard_normal((P, Hkv, S, D)).astype(np.float32))
        ks = vs = None
    return dict(q=q, k=k, v=v, indptr=indptr, indices=perm, seq=np.asarray(ctx, np.int32), ks=ks, vs=vs)


def _dequant(c, code_vals, h):
    if c["ks"] is None:
        return bits_to_f32(c["k"]).astype(np.float64), bits_to_f32(c["v"]).astype(np.float64)
    return code_vals[c["k"]] * np.float64(c["ks"])[None, :, None, None], \
        code_vals[c["v"]] * np.float64(c["vs"])[None, :, None, None]


def _numpy_reference(c, sm_scale):
    """Dense attention per row with numpy: gather through the page table,
    softmax with np.exp, weighted sum with np.dot."""
    vals = torch_e4m3_values()
    K, V = _dequant(c, vals, None)
    B, Hq, D = c["q"].shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    S = K.shape[2]
    out = np.zeros((B, Hq, D))
    qf = bits_to_f32(c["q"]).astype(np.float64)
    for r in range(B):
        T = int(c["seq"][r])
        pages = c["indices"][c["indptr"][r]:c["indptr"][r + 1]]
        t = np.arange(T)
        for i in range(Hq):
            h = i // G
            kk = K[pages[t // S], h, t % S]
            vv = V[pages[t // S], h, t % S]
            s = kk @ qf[r, i] * sm_scale
            p = np.exp(s - s.max())
            out[r, i] = (p @ vv) / p.sum()
    return out


def pin_attn_vs_numpy_dense(orc):
    rng = np.random.default_rng(21)
    sm = 1.0 / np.sqrt(128.0)
    # (Hq, Hkv): group 4, group 16 (query head i reads KV head i // 16), group 1
    for Hq, Hkv in ((8, 2), (32, 2), (3, 3)):
        for fp8 in (True, False):
            c = _rand_case(rng, 3, Hq, Hkv, 16, [1, 37, 70], fp8=fp8)
            got = orc.paged_decode_attn(c["q"], c["k"], c["v"], c["indptr"], c["indices"], c["seq"], sm,
                                        k_scale=c["ks"], v_scale=c["vs"])
            want = _numpy_reference(c, sm)
            assert np.allclose(got, want, rtol=1e-11, atol=1e-13), "Hq=%d Hkv=%d fp8=%s" % (Hq, Hkv, fp8)


def pin_attn_single_token_returns_v(orc):
    rng = np.random.default_rng(22)
    c = _rand_case(rng, 2, 4, 4, 16, [1, 1])
    got = orc.paged_decode_attn(c["q"], c["k"], c["v"], c["indptr"], c["indices"], c["seq"], 0.1,
                                k_scale=c["ks"], v_scale=c["vs"])
    vals = torch_e4m3_values()
    for r in range(2):
        page = c["indices"][c["indptr"][r]]
        for i in range(4):
            assert np.array_equal(got[r, i], vals[c["v"][page, i, 0]] * np.float64(c["vs"][i]))


def pin_attn_identical_keys_mean_of_v(orc):
    rng = np.random.default_rng(23)
    c = _rand_case(rng, 1, 2, 1, 16, [45])
    c["k"][:] = c["k"][0, 0, 0][None, None, None, :]
    got = orc.paged_decode_attn(c["q"], c["k"], c["v"], c["indptr"], c["indices"], c["seq"], 0.3,
                                k_scale=c["ks"], v_scale=c["vs"])
    vals = torch_e4m3_values()
    pages = c["indices"][:3]
    t = np.arange(45)
    vv = vals[c["v"][pages[t // 16], 0, t % 16]] * np.float64(c["vs"][0])
    assert np.allclose(got[0, 0], vv.mean(axis=0), rtol=1e-12, atol=1e-15)
    assert np.allclose(got[0, 1], vv.mean(axis=0), rtol=1e-12, atol=1e-15)


def pin_attn_two_token_closed_form(orc):
    """Two tokens whose logits differ by a known amount: the output is the
    logistic mix of the two value rows, weight 1 / (1 + exp(-(s1 - s0)))."""
    D, S = 128, 16
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = 2.0
    k = np.zeros((1, 1, S, D), np.uint8)
    v = np.zeros((1, 1, S, D), np.uint8)
    k[0, 0, 0, 0] = 0x38      # 1.0
    k[0, 0, 1, 0] = 0x40      # 2.0
    v[0, 0, 0, :] = 0x38      # 1.0
    v[0, 0, 1, :] = 0x48      # 4.0
    sm = 0.75
    got = orc.paged_decode_attn(bf16_bits(q), k, v, np.array([0, 1], np.int32), np.array([0], np.int32),
                                np.array([2], np.int32), sm, k_scale=np.float32([1.0]), v_scale=np.float32([0.5]))
    w1 = 1.0 / (1.0 + np.exp(-(2.0 * 2.0 - 2.0 * 1.0) * sm))
    want = 0.5 * ((1 - w1) * 1.0 + w1 * 4.0)
    assert np.allclose(got[0, 0], want, rtol=1e-14)


def pin_attn_gqa_head_mapping(orc):
    """Query head i reads KV head i // G: give each KV head a constant value row."""
    D, S, Hkv, G = 128, 16, 4, 2
    rng = np.random.default_rng(24)
    k = rng.integers(0, 0x70, (1, Hkv, S, D)).astype(np.uint8)
    v = np.zeros((1, Hkv, S, D), np.uint8)
    for h in range(Hkv):
        v[0, h] = 0x38 + 8 * h          # 1, 2, 4, 8
    q = bf16_bits(rng.standard_normal((1, Hkv * G, D)).astype(np.float32))
    got = orc.paged_decode_attn(q, k, v, np.array([0, 1], np.int32), np.array([0], np.int32),
                                np.array([9], np.int32), 0.1, k_scale=np.ones(Hkv, np.float32),
                                v_scale=np.ones(Hkv, np.float32))
    for i in range(Hkv * G):
        assert np.allclose(got[0, i], 2.0 ** (i // G)), i


def pin_attn_mha_textbook(orc):
    rng = np.random.default_rng(25)
    c = _rand_case(rng, 2, 3, 3, 32, [50, 64], fp8=False)
    sm = 0.2
    got = orc.paged_decode_attn(c["q"], c["k"], c["v"], c["indptr"], c["indices"], c["seq"], sm)
    want = _numpy_reference(c, sm)
    assert np.allclose(got, want, rtol=1e-11, atol=1e-13)


def pin_attn_page_permutation_invariant(orc):
    rng = np.random.default_rng(26)
    c = _rand_case(rng, 3, 8, 2, 16, [20, 33, 64], P=40)
    sm = 1 / np.sqrt(128)
    base = orc.paged_decode_attn(c["q"], c["k"], c["v"], c["indptr"], c["indices"], c["seq"], sm,
                                 k_scale=c["ks"], v_scale=c["vs"])
    perm = rng.permutation(40)
    inv = np.argsort(perm)           # new position of old page p is inv[p]
    k2 = c["k"][perm]
    v2 = c["v"][perm]
    got = orc.paged_decode_attn(c["q"], k2, v2, c["indptr"], inv[c["indices"]].astype(np.int32), c["seq"], sm,
                                k_scale=c["ks"], v_scale=c["vs"])
    assert np.array_equal(got, base)


def pin_attn_fp8_equals_bf16_on_exact_values(orc):
    """An FP8 cache with a power-of-two scale equals a BF16 cache holding the
    dequantized values (every code value times 2^k is exact in bf16)."""
    rng = np.random.default_rng(27)
    c = _rand_case(rng, 2, 8, 2, 16, [30, 17])
    c["ks"] = np.float32([0.25, 2.0 ** -5])
    c["vs"] = np.float32([0.5, 2.0 ** -3])
    sm = 1 / np.sqrt(128)
    fp8 = orc.paged_decode_attn(c["q"], c["k"], c["v"], c["indptr"], c["indices"], c["seq"], sm,
                                k_scale=c["ks"], v_scale=c["vs"])
    vals = torch_e4m3_values()
    kd = (vals[c["k"]] * np.float64(c["ks"])[None, :, None, None]).astype(np.float32)
    vd = (vals[c["v"]] * np.float64(c["vs"])[None, :, None, None]).astype(np.float32)
    kb, vb = bf16_bits(kd), bf16_bits(vd)
    assert np.array_equal(bits_to_f32(kb), kd) and np.array_equal(bits_to_f32(vb), vd)
    bf = orc.paged_decode_attn(c["q"], kb, vb, c["indptr"], c["indices"], c["seq"], sm)
    assert np.array_equal(fp8, bf)


def pin_attn_fail_closed(orc):
    """Aborted, empty, over-long and bad-page requests give zero rows and leave
    the other rows as they are."""
    rng = np.random.default_rng(28)
    c = _rand_case(rng, 5, 4, 2, 16, [10, 20, 30, 40, 12], P=30)
    sm = 0.1
    base = orc.paged_decode_attn(c["q"], c["k"], c["v"], c["indptr"], c["indices"], c["seq"], sm,
                                 k_scale=c["ks"], v_scale=c["vs"])
    seq = c["seq"].copy()
    seq[1] = 0                         # empty
    seq[3] = 16 * 3 + 1                # more tokens than its 3 pages hold
    ind = c["indices"].copy()
    ind[c["indptr"][4]] = 30           # page id outside the pool
    am = np.array([1, 0, 0, 0, 0], np.uint8)
    got = orc.paged_decode_attn(c["q"], c["k"], c["v"], c["indptr"], ind, seq, sm,
                                k_scale=c["ks"], v_scale=c["vs"], abort_mask=am)
    for r in (0, 1, 3, 4):
        assert not got[r].any(), r
    assert np.array_equal(got[2], base[2])
    # a CSR row that runs past the index list is malformed: zero row, nothing read
    nnz = int(c["indptr"][-1]) - 1
    got = orc.paged_decode_attn(c["q"], c["k"], c["v"], c["indptr"], c["indices"], c["seq"], sm,
                                k_scale=c["ks"], v_scale=c["vs"], nnz=nnz)
    assert not got[4].any()
    assert np.array_equal(got[:4], base[:4])


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
