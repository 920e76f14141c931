"""paged_decode_attn on the GPU against the oracle, element by element, on
shapes the oracle finishes in seconds: several tiles, ragged tails, every page
size, every group size up to 8, splits across many warps, and the fail-closed
cases."""
import numpy as np
import pytest

from fp8_paged_kv_decode_gb300 import workloads as W
from gpu_util import PagedCase, assert_close, bf16_out, dev

pytestmark = pytest.mark.gpu

SHAPES = [
    # (B, Hq, Hkv, S, seq)
    (4, 8, 2, 16, [1, 17, 150, 300]),
    (8, 64, 8, 64, [1, 31, 32, 33, 64, 65, 1000, 5000]),
    (3, 8, 8, 32, [17, 200, 96]),            # G = 1
    (3, 4, 2, 128, [300, 129, 5]),           # G = 2
    (2, 16, 2, 64, [40000, 12345]),          # long: split over many warps
    (5, 32, 8, 16, [4097, 1, 2, 3000, 16]),
    (3, 6, 2, 32, [700, 64, 129]),           # G = 3 (N padded to 8)
]


@pytest.mark.parametrize("kv", ["fp8", "bf16"])
@pytest.mark.parametrize("idx", range(len(SHAPES)), ids=[str(i) for i in range(len(SHAPES))])
def test_matches_oracle(orc, kv, idx):
    B, Hq, Hkv, S, seq = shape = SHAPES[idx]
    case = PagedCase(orc, B, Hq, Hkv, S, seq, kv=kv, seed=100 + 2 * idx + (kv == "bf16"))
    got = bf16_out(case.gpu())
    assert_close(got, case.oracle(orc), "kv=%s shape=%s" % (kv, shape))


@pytest.mark.parametrize("kv", ["fp8", "bf16"])
def test_tiny_workload(orc, kv):
    wl = W.WORKLOADS["tiny_gqa4"]
    hb = W.host_batch(wl)
    case = PagedCase(orc, wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.page_size, hb.seq_lens, kv=kv, seed=11)
    assert_close(bf16_out(case.gpu()), case.oracle(orc), "tiny_gqa4 " + kv)


def test_peaky_softmax(orc):
    """Logit std ~4 (q ~ 4 N(0,1)) over long contexts split across warps."""
    case = PagedCase(orc, 2, 8, 1, 64, [20000, 7000], seed=3, q_std=4.0)
    assert_close(bf16_out(case.gpu()), case.oracle(orc), "peaky")


def wide_range_q(case, mults, seed, zero_k=False):
    """Scale a few channels of every query head by large factors (the other
    channels stay N(0,1)), so one query row spans a wide dynamic range.  The
    channels are chosen per KV head and shared by its query heads; with
    ``zero_k`` the K codes of those channels are zero in the whole pool, so the
    large channels add nothing to the logits and the small ones decide them."""
    rng = np.random.default_rng(seed)
    G = case.Hq // case.Hkv
    q = W.bits_to_f32(case.q).copy()
    for h in range(case.Hkv):
        ch = rng.choice(case.D, size=len(mults), replace=False)
        for c, m in zip(ch, mults):
            q[:, h * G:(h + 1) * G, c] *= np.float32(m)
        if zero_k:
            case.kc[:, h, :, ch] = 0
    case.q = W.bf16_bits(q)


@pytest.mark.parametrize("zero_k", [False, True], ids=["k_random", "k_zero_in_large_channels"])
@pytest.mark.parametrize("G", [4, 8])
def test_wide_dynamic_range_q(orc, G, zero_k):
    """FP8 KV: the queries enter the tensor cores as f16 with a power-of-two
    scale per row; a row whose channels span 1 to 1e4 (three channels x1e3,
    x1e4, x1e4) still matches the oracle, with K random in those channels
    (a very peaky softmax) or zero there (the small channels decide)."""
    Hkv = 2
    case = PagedCase(orc, 4, G * Hkv, Hkv, 64 if G == 8 else 16, [3000, 100, 17, 800], seed=60 + G + zero_k)
    wide_range_q(case, [1e3, 1e4, 1e4], seed=70 + G, zero_k=zero_k)
    assert_close(bf16_out(case.gpu()), case.oracle(orc), "G=%d zero_k=%s" % (G, zero_k))


@pytest.mark.parametrize("m", [1e9, 1e12])
@pytest.mark.parametrize("G", [4, 8])
def test_huge_logits_stay_finite(orc, G, m):
    """Query channels x1e9 or x1e12 with K random there: logits reach ~1e10
    in log2 units.  The softmax scales each logit with the same rounded
    multiply that forms the running maximum, so the largest term is exactly
    1 and nothing overflows; the outputs are finite and match the oracle."""
    case = PagedCase(orc, 4, G * 2, 2, 64, [3000, 100, 17, 800], seed=60 + G)
    wide_range_q(case, [m, m, m / 10], seed=70 + G)
    got = bf16_out(case.gpu())
    assert np.isfinite(got).all()
    assert_close(got, case.oracle(orc), "G=%d m=%g" % (G, m))


@pytest.mark.parametrize("S", [16, 64])
def test_fail_closed_rows(orc, S):
    """Aborted, empty, over-long and bad-page requests give zero rows; the
    other rows still match; the bad page id is never dereferenced and is
    reported in the device error word.  Page size 16 runs the producer-warp
    CTA, 64 the single-warp one."""
    import fp8_paged_kv_decode_gb300 as fkv
    B = 6
    case = PagedCase(orc, B, 16, 2, S, [100, 200, 300, 400, 500, 600], seed=4)
    seq = case.seq.copy()
    seq[1] = 0
    seq[3] = S * ((400 + S - 1) // S) + 1               # one token more than its pages hold
    ind = case.indices.copy()
    ind[case.indptr[4] + 3] = case.P + 1000               # outside the pool
    am = np.array([1, 0, 0, 0, 0, 0], np.uint8)
    fkv.device_error(clear=True)
    got = bf16_out(case.gpu(abort_mask=am, seq=seq, indices=ind))
    ref = case.oracle(orc, abort_mask=am, seq=seq, indices=ind)
    for r in (0, 1, 3, 4):
        assert not ref[r].any()
        assert np.array_equal(got[r], np.zeros_like(got[r])), r
    assert_close(got, ref, "fail-closed")
    assert fkv.device_error() & fkv.DEVERR_ATTN_PAGE


def test_no_tracker_path_equals_all_clear_mask(orc):
    case = PagedCase(orc, 3, 8, 2, 64, [500, 70, 1], seed=5)
    import torch
    a = case.gpu().view(torch.int16).cpu().numpy()
    b = case.gpu(abort_mask=np.zeros(3, np.uint8)).view(torch.int16).cpu().numpy()
    assert np.array_equal(a, b)


@pytest.mark.parametrize("S", [64, 16])
def test_abort_equals_absent_bytewise(orc, S):
    """Aborting a request leaves every other row byte-identical to a batch
    without that request (the split plan depends only on the live requests),
    for both CTA shapes."""
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    case = PagedCase(orc, 5, 32, 4, S, [9000, 300, 20000, 4000, 1], seed=6)
    am = np.array([0, 0, 1, 0, 0], np.uint8)
    full = case.gpu(abort_mask=am).cpu()
    keep = [0, 1, 3, 4]
    # the same batch with request 2 removed from the page table and queries
    indptr = [0]
    ind = []
    for r in keep:
        pages = case.indices[case.indptr[r]:case.indptr[r + 1]]
        ind.extend(pages.tolist())
        indptr.append(len(ind))
    q = dev(case.q[keep], dtype=torch.bfloat16)
    out = torch.empty(len(keep), 32, 128, dtype=torch.bfloat16, device="cuda")
    ws = fkv.alloc_workspace(len(keep), 32, 4)
    fkv.paged_decode_attn(q, dev(case.kc), dev(case.vc), dev(np.array(indptr, np.int32)), dev(np.array(ind, np.int32)),
                          dev(case.seq[keep]), case.sm, out, ws, k_scale=dev(case.k_scale), v_scale=dev(case.v_scale))
    torch.cuda.synchronize()
    assert np.array_equal(full[keep].view(torch.int16).numpy(), out.cpu().view(torch.int16).numpy())
    assert not full[2].float().abs().sum()


def test_page_permutation_invariant(orc):
    """Moving pages to other physical slots changes nothing (bit for bit)."""
    import torch
    case = PagedCase(orc, 3, 16, 2, 32, [3000, 77, 1200], seed=7, spare=50)
    base = case.gpu().view(torch.int16).cpu().numpy()
    rng = np.random.default_rng(8)
    perm = rng.permutation(case.P)
    inv = np.argsort(perm)
    got = case.gpu(indices=inv[case.indices].astype(np.int32), kc=case.kc[perm], vc=case.vc[perm])
    assert np.array_equal(base, got.view(torch.int16).cpu().numpy())


def test_shared_pages_across_requests(orc):
    """Two requests listing the same physical pages (a shared prefix) read the same data."""
    case = PagedCase(orc, 2, 8, 2, 16, [160, 160], seed=9)
    ind = case.indices.copy()
    ind[case.indptr[1]:case.indptr[1] + 5] = ind[case.indptr[0]:case.indptr[0] + 5]
    got = bf16_out(case.gpu(indices=ind))
    assert_close(got, case.oracle(orc, indices=ind), "shared pages")


def test_shared_prefix_batch(orc):
    """Eight requests whose first 40 pages are the same physical pages (a shared
    2560-token prompt) on top of their own suffixes, FP8 and BF16."""
    from fp8_paged_kv_decode_gb300 import workloads as W
    for kv in ("fp8", "bf16"):
        case = PagedCase(orc, 8, 32, 4, 64, [5000, 2700, 2561, 9000, 3333, 2600, 7000, 4096], kv=kv, seed=61)
        pt = W.PageTable(case.indptr, case.indices, np.zeros(case.indices.size, np.uint32),
                         np.zeros(case.P, np.uint32), case.P)
        ind = W.share_prefix(pt, 40).indices
        assert (ind[case.indptr[3]:case.indptr[3] + 40] == case.indices[:40]).all()
        assert_close(bf16_out(case.gpu(indices=ind)), case.oracle(orc, indices=ind), "shared prefix " + kv)


def test_empty_batch_is_noop():
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    kc = torch.zeros(2, 1, 16, 128, dtype=torch.uint8, device="cuda")
    q = torch.empty(0, 8, 128, dtype=torch.bfloat16, device="cuda")
    s = torch.ones(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    i1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    fkv.paged_decode_attn(q, kc, kc, i1, i1, i1[:0], 0.1, q, ws, k_scale=s, v_scale=s)
    torch.cuda.synchronize()



def test_graph_captured_step_equals_eager(orc):
    """The step captured in a CUDA graph (append, check, attention) gives the
    same bytes as the eager calls."""
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    from fp8_paged_kv_decode_gb300 import workloads as W
    wl = W.WORKLOADS["integrity_256req"]
    db = W.device_batch(wl, "cuda", ctx=np.full(wl.batch, 300))
    P = db.pt.num_pages
    kc = torch.zeros(P, wl.num_kv_heads, wl.page_size, 128, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    ks, vs = dev(db.k_scale), dev(db.v_scale)
    fkv.kv_append_fp8(db.k_src, db.v_src, db.slots_src, ks, vs, kc, vc)
    ind, indp = dev(db.pt.indices), dev(db.pt.indptr)
    tags, exp = dev(db.pt.page_tags.view(np.int32)), dev(db.pt.expected_tags.view(np.int32))
    seq = dev(db.seq_lens)
    mask = torch.zeros(wl.batch, dtype=torch.uint8, device="cuda")
    out = torch.zeros(wl.batch, wl.num_q_heads, 128, dtype=torch.bfloat16, device="cuda")
    ws = fkv.alloc_workspace(wl.batch, wl.num_q_heads, wl.num_kv_heads)

    def step():
        fkv.kv_append_fp8(db.k_new, db.v_new, db.slots_new, ks, vs, kc, vc)
        fkv.kv_page_tag_check(tags, indp, ind, exp, mask)
        fkv.paged_decode_attn(db.q, kc, vc, indp, ind, seq, 1 / np.sqrt(128), out, ws, k_scale=ks, v_scale=vs,
                              abort_mask=mask)

    step()
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert int(mask.sum()) > 0
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


@pytest.mark.parametrize("B,kv", [(100, "fp8"), (128, "fp8"), (129, "fp8"), (129, "bf16"), (1024, "fp8"),
                                  (2000, "fp8")])
def test_large_batches_both_schedules(orc, B, kv):
    """Up to 128 requests every attention warp finds its own range from the
    inputs (past 64 in one pass over 32-request chunks, then the chunk that
    holds its first tile); larger batches read the plan kernel's prefix
    table.  Both agree
    with the oracle, with empty, aborted and ragged requests mixed in."""
    rng = np.random.default_rng(B + (kv == "bf16"))
    seq = rng.integers(0, 90, B)
    seq[rng.choice(B, 20, replace=False)] = 0
    case = PagedCase(orc, B, 8, 2, 16, seq, kv=kv, seed=B)
    abort = (rng.random(B) < 0.05).astype(np.uint8)
    got = bf16_out(case.gpu(abort_mask=abort))
    assert_close(got, case.oracle(orc, abort_mask=abort), "B=%d kv=%s" % (B, kv))


@pytest.mark.parametrize("kv", ["fp8", "bf16"])
@pytest.mark.parametrize("Hkv,seq", [(1, [3200]), (2, [3200]), (1, [3136]), (1, [3585]), (1, [25 * 512]),
                                     (1, [4243 * 64])])
def test_long_unit_merge_chunks(orc, kv, Hkv, seq):
    """One long unit split over many warps.  With whole warps per unit (two
    tiles each here), 3200 tokens are 50 tiles over 25 warps: four merge
    chunks of six parts and one that holds only the unit's last warp; 3136
    tokens (49 tiles) give ranges of one and two tiles; 12800 tokens give 17
    chunks, more than one shared-memory merge round holds.  4243 tiles are
    past the whole-warp schedule on a 152-SM part: the even split, 7 to 8
    tiles per warp."""
    case = PagedCase(orc, 1, 8 * Hkv, Hkv, 64, seq, kv=kv, seed=sum(seq) + Hkv)
    assert_close(bf16_out(case.gpu()), case.oracle(orc), "Hkv=%d seq=%s kv=%s" % (Hkv, seq, kv))


def test_batch_beyond_plan_smem_table(orc):
    """More requests than the plan kernel keeps in shared memory (4096): its
    warp search reads the prefix table from global memory."""
    rng = np.random.default_rng(4500)
    B = 4500
    seq = rng.integers(0, 40, B)
    case = PagedCase(orc, B, 2, 1, 16, seq, kv="fp8", seed=4500)
    abort = (rng.random(B) < 0.02).astype(np.uint8)
    assert_close(bf16_out(case.gpu(abort_mask=abort)), case.oracle(orc, abort_mask=abort), "B=4500")


@pytest.mark.parametrize("kv,S", [("fp8", 64), ("fp8", 16), ("bf16", 64), ("bf16", 16)])
@pytest.mark.parametrize("seq,abort", [
    ([1, 64, 65], None),
    ([30000, 100, 0, 5000, 700], [0, 1, 0, 0, 0]),
    ([106304, 106304], None),
    ([106368, 106368], None),
], ids=["one_tile_units", "mixed", "whole_warp_max", "even_split_min"])
def test_small_batch_schedules(orc, kv, S, seq, abort):
    """Small batches give every (request, KV head) unit whole warps: units of
    one or two tiles get one warp and need no merge, long ones are split
    evenly over their own warps, and empty or aborted requests get none.
    Two requests of 1661 tiles per head are the most a 152-SM part schedules
    this way (11 tiles per warp, one below the even split's minimum of 12);
    one tile more per head takes the even split of the batch's tiles.  Page size 16 runs the producer-warp
    CTA, 64 the single-warp one."""
    B = len(seq)
    case = PagedCase(orc, B, 16, 2, S, seq, kv=kv, seed=sum(seq) + S + (kv == "bf16"))
    am = None if abort is None else np.array(abort, np.uint8)
    got = bf16_out(case.gpu(abort_mask=am))
    assert_close(got, case.oracle(orc, abort_mask=am), "seq=%s kv=%s S=%d" % (seq, kv, S))


@pytest.mark.parametrize("kv", ["fp8", "bf16"])
def test_batch_of_48_even_split(orc, kv):
    """48 requests of 8 KV heads (384 units) is the shape of the 64-request
    headline: the instance without the whole-warp option, each warp finding
    its range of the even split from the requests' rows it loaded itself."""
    rng = np.random.default_rng(48 + (kv == "bf16"))
    seq = rng.integers(1, 3000, 48)
    seq[[3, 17]] = 0
    case = PagedCase(orc, 48, 64, 8, 64, seq, kv=kv, seed=480 + (kv == "bf16"))
    abort = np.zeros(48, np.uint8)
    abort[[5, 40]] = 1
    assert_close(bf16_out(case.gpu(abort_mask=abort)), case.oracle(orc, abort_mask=abort), "B=48 kv=" + kv)


@pytest.mark.parametrize("kv", ["fp8", "bf16"])
@pytest.mark.parametrize("S", [16, 64])
def test_batch_with_no_live_request(orc, kv, S):
    """Every request empty or aborted: the batch runs the whole-warp
    instance, no warp gets work, and every output row (the buffer starts as
    NaN) must still come out zero."""
    case = PagedCase(orc, 4, 16, 2, S, [100, 0, 300, 0], kv=kv, seed=77 + S)
    am = np.array([1, 0, 1, 0], np.uint8)
    got = bf16_out(case.gpu(abort_mask=am))
    assert np.array_equal(got, np.zeros_like(got))
    assert np.array_equal(case.oracle(orc, abort_mask=am), np.zeros_like(got))


@pytest.mark.parametrize("kv", ["fp8", "bf16"])
@pytest.mark.parametrize("Hq,Hkv,S,seq", [
    (32, 2, 64, [700, 3000, 65]),        # G = 16: two groups of 8 per KV head
    (24, 2, 16, [1, 500, 129, 2048]),    # G = 12: two groups of 6
    (32, 1, 32, [5000, 17]),             # G = 32: four groups of 8
    (64, 1, 64, [1500]),                 # G = 64: eight groups of 8
    (40, 4, 64, [300] * 40),             # G = 10, 40 requests: the even split
], ids=["g16", "g12", "g32", "g64", "g10_b40"])
def test_large_group_sizes(orc, kv, Hq, Hkv, S, seq):
    """Group sizes above 8 that split into a power-of-two number of groups of
    at most 8: each group is a virtual KV head reading the KV head's pages
    again, and every query row still matches the oracle."""
    case = PagedCase(orc, len(seq), Hq, Hkv, S, seq, kv=kv, seed=7 * Hq + Hkv + (kv == "bf16"))
    assert_close(bf16_out(case.gpu()), case.oracle(orc), "Hq=%d Hkv=%d S=%d kv=%s" % (Hq, Hkv, S, kv))


def test_unsplittable_group_size_is_unsupported(orc):
    """G = 9 has no power-of-two split into groups of at most 8: the call is
    refused before anything is launched."""
    import fp8_paged_kv_decode_gb300 as fkv
    case = PagedCase(orc, 2, 9, 1, 64, [100, 200], seed=9)
    with pytest.raises(fkv.FkvError, match="unsupported"):
        case.gpu()


def test_abort_equals_absent_under_whole_warp_schedule(orc):
    """Both runs take the whole-warp schedule, and its tiles per warp come from
    the live units only: 147 live tiles per KV head (requests of 100 and 47
    tiles) over 8 KV heads give 1176 tiles, which would be 3 tiles per warp
    if the aborted request's 8 units were counted (608 - 24 warps to spare on
    a 152-SM part) and are 2 either way when only live units count.  The
    live rows must be byte-identical to the batch without the request."""
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    case = PagedCase(orc, 3, 64, 8, 64, [6400, 64, 3008], seed=12)
    am = np.array([0, 1, 0], np.uint8)
    full = case.gpu(abort_mask=am).cpu()
    keep = [0, 2]
    indptr = [0]
    ind = []
    for r in keep:
        ind.extend(case.indices[case.indptr[r]:case.indptr[r + 1]].tolist())
        indptr.append(len(ind))
    q = dev(case.q[keep], dtype=torch.bfloat16)
    out = torch.empty(len(keep), 64, 128, dtype=torch.bfloat16, device="cuda")
    ws = fkv.alloc_workspace(len(keep), 64, 8)
    fkv.paged_decode_attn(q, dev(case.kc), dev(case.vc), dev(np.array(indptr, np.int32)), dev(np.array(ind, np.int32)),
                          dev(case.seq[keep]), case.sm, out, ws, k_scale=dev(case.k_scale), v_scale=dev(case.v_scale))
    torch.cuda.synchronize()
    assert np.array_equal(full[keep].view(torch.int16).numpy(), out.cpu().view(torch.int16).numpy())
    assert_close(bf16_out(full), case.oracle(orc, abort_mask=am), "aborted middle request")


def _spare_page_zero(case):
    """Relabel so that physical page 0 is a spare page (listed by no request):
    swap its contents and its id with one that is."""
    used = set(case.indices.tolist())
    if 0 in used:
        s = next(x for x in range(case.P) if x not in used)
        for pool in (case.kc, case.vc):
            pool[[0, s]] = pool[[s, 0]]
        case.indices = np.where(case.indices == 0, s, case.indices).astype(np.int32)
    return case


@pytest.mark.parametrize("kv", ["fp8", "bf16"])
@pytest.mark.parametrize("S", [16, 64])
def test_bad_page_rows_are_zero_over_nan_bytes(orc, kv, S):
    """A page id outside the pool is replaced by page 0 for the copy and the
    unit is marked bad; its row must be zeros even when page 0 holds NaN codes
    (a short request whose unit one warp covers whole, and a long one split
    over several warps), with no abort mask to catch them first."""
    import fp8_paged_kv_decode_gb300 as fkv
    case = _spare_page_zero(PagedCase(orc, 4, 32, 4, S, [150, 30000, 2000, 9000], kv=kv, seed=31, spare=4))
    if case.fp8:
        case.kc[0] = 0x7F
        case.vc[0] = 0xFF
    else:
        case.kc[0] = 0x7FC0
        case.vc[0] = 0xFFC0
    ind = case.indices.copy()
    ind[case.indptr[0]] = case.P + 7                    # request 0: one unit per KV head, one warp each
    ind[case.indptr[1] + 100] = -3                      # request 1: units split over many warps
    fkv.device_error(clear=True)
    got = bf16_out(case.gpu(indices=ind))
    ref = case.oracle(orc, indices=ind)
    for r in (0, 1):
        assert not ref[r].any()
        assert np.array_equal(got[r], np.zeros_like(got[r])), r
    assert_close(got, ref, "bad pages over NaN bytes")
    assert fkv.device_error() & fkv.DEVERR_ATTN_PAGE


def _identity_case(orc, shape, kv):
    if shape == "mixed":        # units over one warp, a few (one merge level), many (two levels)
        return PagedCase(orc, 12, 64, 8, 64, [20000, 9000, 3000, 15000, 500, 7000, 12000, 800, 25000, 4000, 6000, 1],
                         kv=kv, seed=33)
    # 160 requests of 16-token pages: the plan kernel's table and the two-warp CTA
    seq = np.random.default_rng(34).integers(1, 3000, 160)
    return PagedCase(orc, 160, 32, 4, 16, seq, kv=kv, seed=34)


@pytest.mark.parametrize("kv,shape", [("fp8", "mixed"), ("bf16", "mixed"), ("fp8", "plan")])
def test_run_to_run_byte_identity(orc, kv, shape):
    """The same call repeated gives the same bytes, although which warp
    merges a split unit, and whether it merges from its registers or through
    shared memory, depends on when the unit's parts arrive: every merge folds
    the parts in the same order with the same roundings.  Calls alternate
    with a write that evicts L2, so timings vary."""
    import torch
    case = _identity_case(orc, shape, kv)
    if shape == "mixed":
        assert_close(bf16_out(case.gpu()), case.oracle(orc), "byte-identity batch")
    import fp8_paged_kv_decode_gb300 as fkv
    q = dev(case.q, dtype=torch.bfloat16)
    cdt = None if case.fp8 else torch.bfloat16
    kt, vt = dev(case.kc, dtype=cdt), dev(case.vc, dtype=cdt)
    ks = dev(case.k_scale) if case.fp8 else None
    vs = dev(case.v_scale) if case.fp8 else None
    ip, ix, sl = dev(case.indptr), dev(case.indices), dev(case.seq)
    ws = fkv.alloc_workspace(case.B, case.Hq, case.Hkv, fkv.KV_FP8_E4M3 if case.fp8 else fkv.KV_BF16)
    out = torch.empty((case.B, case.Hq, 128), dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(64 * 2 ** 20, dtype=torch.float32, device="cuda")     # 256 MB > L2
    first = None
    for it in range(40):
        if it % 2:
            flush.fill_(float(it))
        out.fill_(float("nan"))
        fkv.paged_decode_attn(q, kt, vt, ip, ix, sl, case.sm, out, ws, k_scale=ks, v_scale=vs)
        torch.cuda.synchronize()
        got = out.view(torch.int16).cpu().numpy().copy()
        if first is None:
            first = got
        else:
            assert np.array_equal(got, first), "call %d differs from the first" % it
