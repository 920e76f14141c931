"""Host-side logic: workload generators, page allocator, replica sharding (no GPU)."""
import os

import numpy as np
import pytest

from fp8_paged_kv_decode_gb300 import workloads as W


@pytest.mark.parametrize("name", sorted(W.WORKLOADS))
def test_page_tables_are_consistent(name):
    wl = W.WORKLOADS[name]
    rng = np.random.default_rng(wl.seed)
    seq = W.context_lengths(wl, rng) + 1
    pt = W.build_page_table(wl, seq, rng)
    npages = np.diff(pt.indptr)
    assert np.array_equal(npages, (seq + wl.page_size - 1) // wl.page_size)
    assert pt.indices.min() >= 0 and pt.indices.max() < pt.num_pages
    assert np.unique(pt.indices).size == pt.indices.size, "a page has one owner"
    live_ok = pt.page_tags[pt.indices] == pt.expected_tags
    if wl.stale_frac:
        assert pt.stale_pages.size == round(wl.stale_frac * pt.indices.size)
        assert np.array_equal(~live_ok, np.isin(pt.indices, pt.stale_pages))
    else:
        assert live_ok.all()


def test_workload_shapes_match_their_description():
    w = W.WORKLOADS
    assert (w["pages_shaped_64req"].batch, w["pages_shaped_64req"].num_q_heads, w["pages_shaped_64req"].num_kv_heads,
            w["pages_shaped_64req"].page_size) == (64, 64, 8, 64)
    rng = np.random.default_rng(w["pages_shaped_64req"].seed)
    ctx = W.context_lengths(w["pages_shaped_64req"], rng)
    assert ctx.min() >= 512 and ctx.max() <= 131072
    assert 8000 < np.median(ctx) < 30000
    assert len(W.outlier_channels(w["pages_shaped_64req"], rng)) == 10       # 1% of 8 x 128 K channels
    assert w["long_ctx_131k"].q_std == 4.0
    assert w["integrity_256req"].stale_frac == 0.01


def test_tag_bump_wraps():
    rng = np.random.default_rng(0)
    pool = W.PagePool(4, rng)
    pool.tags[:] = 0xFFFFFFFF
    ids, tags = pool.alloc(2)
    assert (tags == 0).all()


def test_fp8_halves_cache_bytes():
    """The FP8 pool holds the same tokens in half the bytes of the BF16 pool
    (Cloudflare post: FP8 e4m3 instead of BF16 halves the cache)."""
    import torch
    a = torch.empty(10, 8, 64, 128, dtype=torch.uint8)
    b = torch.empty(10, 8, 64, 128, dtype=torch.bfloat16)
    assert 2 * a.numel() * a.element_size() == b.numel() * b.element_size()


def test_shards_cover_batch_once():
    for B in (1, 5, 64, 256):
        for world in (1, 2, 3, 8):
            parts = [W.shard_requests(B, r, world) for r in range(world)]
            allr = np.concatenate(parts)
            assert np.array_equal(np.sort(allr), np.arange(B))


def _gloo_worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import torch
    mine = W.shard_requests(64, rank, world)
    t = torch.zeros(64, dtype=torch.int64)
    t[mine] = 1
    dist.all_reduce(t)
    # the bench's own barrier and timing reduction: max over ranks of the
    # per-rank time
    import bench
    bench._PG = True
    bench.barrier()
    ms = bench.max_over_ranks(10.0 + rank)
    q.put((rank, t.tolist(), float(ms)))
    dist.destroy_process_group()


def test_replica_sharding_gloo_world2():
    import multiprocessing as mp
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ps = [ctx.Process(target=_gloo_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = [q.get(timeout=120) for _ in ps]
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, cover, ms in res:
        assert cover == [1] * 64
        assert ms == 11.0


def test_admission_under_a_budget():
    pages = np.array([3, 1, 4, 1, 5])
    assert W.admitted(10, pages, 0) == 0
    assert W.admitted(10, pages, 40) == 2          # 3 + 1 pages fit, the third (4) does not
    assert W.admitted(10, pages, 90) == 4
    assert W.admitted(5, pages, 40) == 3           # half the page bytes: twice the pages
    # the same budget holds twice the tokens at half the bytes per page
    wl = W.WORKLOADS["pages_shaped_64req"]
    rng = np.random.default_rng(wl.seed)
    npg = (W.context_lengths(wl, rng) + 1 + 63) // 64
    pf = 2 * 8 * 64 * 128
    budget = int(npg[:32].sum()) * 2 * pf
    assert W.admitted(2 * pf, npg, budget) == 32
    assert W.admitted(pf, npg, budget) > 32


def test_share_prefix_rewrites_only_long_requests():
    wl = W.WORKLOADS["tiny_gqa4"]
    rng = np.random.default_rng(3)
    pt = W.build_page_table(wl, np.array([100, 20, 64, 300]), rng)     # 7, 2, 4, 19 pages of 16 tokens
    assert pt.indptr.tolist() == [0, 7, 9, 13, 32]
    sp = W.share_prefix(pt, 3)
    np.testing.assert_array_equal(sp.indices[:9], pt.indices[:9])      # request 0 itself; request 1 too short
    np.testing.assert_array_equal(sp.indices[9:12], pt.indices[:3])    # request 2: first 3 pages shared
    assert sp.indices[12] == pt.indices[12]
    np.testing.assert_array_equal(sp.indices[13:16], pt.indices[:3])   # request 3
    np.testing.assert_array_equal(sp.indices[16:], pt.indices[16:])
    np.testing.assert_array_equal(sp.expected_tags[13:16], pt.expected_tags[:3])


def test_subset_batch_keeps_the_first_requests():
    db = W.device_batch(W.WORKLOADS["tiny_gqa4"], "cpu")
    sub = W.subset_batch(db, 2)
    assert sub.wl.batch == 2
    np.testing.assert_array_equal(sub.seq_lens, db.seq_lens[:2])
    np.testing.assert_array_equal(sub.pt.indptr, db.pt.indptr[:3])
    np.testing.assert_array_equal(sub.pt.indices, db.pt.indices[:db.pt.indptr[2]])
    assert sub.k_src.shape[0] == int(db.ctx[:2].sum())
    assert W.subset_batch(db, 0).wl.batch == 0
    with pytest.raises(ValueError):
        W.subset_batch(db, db.wl.batch + 1)


def test_reference_arm_runs_on_rank_zero_only():
    """Launched as two ranks, the reference arm's rank 1 exits 0 without work
    or output (rank 0 alone runs the oracle and prints the line)."""
    import subprocess
    import sys
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
