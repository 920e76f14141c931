"""Benchmark: one decode step of the FP8 paged-KV path on the 64-request workload.

A step is the whole hot path over one batch: append one new token per request
(kv_append_fp8), the per-page generation-tag check (kv_page_tag_check), and
paged decode attention (paged_decode_attn).  The workload is
``pages_shaped_64req``: 64 concurrent requests, 64 query / 8 KV heads,
head_dim 128, page 64, contexts lognormal (median 16384, sigma 0.8) clipped to
[512, 131072], FP8 e4m3 KV (~2.9 GB read per step, far larger than L2, so no
L2 flush is needed between steps).

Prints one JSON line.  ``value`` is decode tokens/s (requests x steps / time,
one layer); the roofline object is for the paged_decode_attn call, whose
algorithmic bytes are the KV bytes of every attended token plus q, out and
page ids.  The same step with a BF16 cache, the integrity-check overhead on
``integrity_256req`` and the CPU oracle on a bounded sample are reported
beside it.  ``--impl reference`` times the CPU oracle as the reference arm.

Multi-GPU (torchrun): each rank runs its own replica batch (weak scaling), no
collective on the data path; timing is max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode attn tokens/s & HBM GB/s (% of 8 TB/s) at 64 req, FP8 vs BF16 KV"
HEADLINE = "pages_shaped_64req"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--kv", default="fp8", choices=["fp8", "bf16"], help="KV cache dtype of the main line")
    ap.add_argument("--page-size", type=int, default=None, help="override the workload's page size (tokens)")
    ap.add_argument("--ctx", default=None, help="override the workload's context lengths, e.g. fixed:16384")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's request count (the same seeded draws: the first N requests)")
    ap.add_argument("--stale-frac", type=float, default=None,
                    help="override the workload's fraction of stale (reallocated) pages, e.g. 0 for a clean batch")
    ap.add_argument("--skip-extras", action="store_true", help="only the FP8 headline and e2e")
    ap.add_argument("--cpu-requests", type=int, default=8, help="requests in the oracle's bounded sample")
    ap.add_argument("--shared-prefix", action="store_true",
                    help="instead of the headline: requests sharing their first pages (a common prompt prefix)")
    ap.add_argument("--capacity-sweep", action="store_true",
                    help="instead of the headline: KV budget admission and a concurrency sweep, FP8 vs BF16")
    ap.add_argument("--configs-only", action="store_true",
                    help="instead of the headline: the attention call on every workload (the per-config table)")
    ap.add_argument("--config-reps", type=int, default=None,
                    help="timed attention calls per workload in the per-config table (default from --steps)")
    return ap.parse_args()


# ----------------------------------------------------------------------------
# environment
# ----------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def selected_workload(W, args):
    """The --workload entry, with --batch, --page-size, --ctx and --stale-frac applied when given."""
    wl = W.WORKLOADS[args.workload]
    if args.batch is not None and args.batch != wl.batch:
        wl = dataclasses.replace(wl, name="%s (first %d requests)" % (wl.name, args.batch), batch=args.batch)
    if args.ctx is not None and args.ctx != wl.ctx:
        wl = dataclasses.replace(wl, name="%s (ctx %s)" % (wl.name, args.ctx), ctx=args.ctx)
    if args.page_size is not None and args.page_size != wl.page_size:
        wl = dataclasses.replace(wl, name="%s (page %d)" % (wl.name, args.page_size), page_size=args.page_size)
    if args.stale_frac is not None and args.stale_frac != wl.stale_frac:
        wl = dataclasses.replace(wl, name="%s (stale_frac=%g)" % (wl.name, args.stale_frac),
                                 stale_frac=args.stale_frac)
    return wl


def peak_hbm():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def code_tokens(text):
    """Source text without // comments and with whitespace collapsed: edits
    to comments leave the hash of the code unchanged."""
    out = []
    for line in text.splitlines():
        i = line.find("//")
        if i >= 0:
            line = line[:i]
        line = " ".join(line.split())
        if line:
            out.append(line)
    return "\n".join(out)


def kernel_source_hash(sources=None):
    """Hash of the attention kernel's code (its two source files), which the
    recorded ncu traffic figures are keyed to."""
    h = hashlib.sha256()
    for f in ("decode_attn.cu", "fkv_common.cuh"):
        if sources is None:
            with open(os.path.join(ROOT, "fp8_paged_kv_decode_gb300", "csrc", f)) as fh:
                text = fh.read()
        else:
            text = sources[f]
        h.update(code_tokens(text).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kv, workload=HEADLINE):
    """DRAM bytes per paged_decode_attn call on ``workload`` from the committed
    ncu summary (keys ``<workload>.<kv>.dram_bytes_per_call``), if it was taken
    on the current kernel source; else None."""
    try:
        vals = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                line = line.strip()
                if line and not line.startswith("#") and "=" in line:
                    k, v = line.split("=", 1)
                    vals[k.strip()] = v.strip()
        key = "%s.%s" % (workload, kv)
        if vals.get(key + ".source_hash") == kernel_source_hash():
            return {"dram_bytes_per_call": int(vals[key + ".dram_bytes_per_call"])}
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.lines = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.dev)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# the step
# ----------------------------------------------------------------------------
class Step:
    """Device state of one workload for one KV dtype: populated cache, page
    table, tags and the per-step inputs."""

    def __init__(self, db, kv, device):
        import torch
        import fp8_paged_kv_decode_gb300 as fkv
        self.fkv, self.torch = fkv, torch
        self.db, self.kv, self.device = db, kv, device
        wl = db.wl
        self.B, self.Hq, self.Hkv, self.S, self.D = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.page_size, wl.head_dim
        P = db.pt.num_pages
        self.fp8 = kv == "fp8"
        dt = torch.uint8 if self.fp8 else torch.bfloat16
        self.k_cache = torch.zeros(P, self.Hkv, self.S, self.D, dtype=dt, device=device)
        self.v_cache = torch.zeros(P, self.Hkv, self.S, self.D, dtype=dt, device=device)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
        self.k_scale, self.v_scale = t(db.k_scale), t(db.v_scale)
        if self.fp8:
            fkv.kv_append_fp8(db.k_src, db.v_src, db.slots_src, self.k_scale, self.v_scale, self.k_cache, self.v_cache)
        else:
            fkv.kv_append_bf16(db.k_src, db.v_src, db.slots_src, self.k_cache, self.v_cache)
        self.indptr, self.indices = t(db.pt.indptr), t(db.pt.indices)
        self.page_tags = t(db.pt.page_tags.view(np.int32))
        self.expected = t(db.pt.expected_tags.view(np.int32))
        self.seq_lens = t(db.seq_lens)
        self.q, self.k_new, self.v_new, self.slots_new = db.q, db.k_new, db.v_new, db.slots_new
        self.mask = torch.zeros(self.B, dtype=torch.uint8, device=device)
        self.out = torch.empty(self.B, self.Hq, self.D, dtype=torch.bfloat16, device=device)
        self.ws = fkv.alloc_workspace(self.B, self.Hq, self.Hkv, fkv.KV_FP8_E4M3 if self.fp8 else fkv.KV_BF16, device)
        self.sm = 1.0 / np.sqrt(self.D)
        torch.cuda.synchronize(device)

    def append(self):
        if self.fp8:
            self.fkv.kv_append_fp8(self.k_new, self.v_new, self.slots_new, self.k_scale, self.v_scale, self.k_cache,
                                   self.v_cache)
        else:
            self.fkv.kv_append_bf16(self.k_new, self.v_new, self.slots_new, self.k_cache, self.v_cache)

    def check(self):
        self.fkv.kv_page_tag_check(self.page_tags, self.indptr, self.indices, self.expected, self.mask)

    def append_check(self, separate=False):
        """The step's append and integrity check: one launch
        (kv_append_fp8_tag_check / kv_append_bf16_tag_check), or with
        ``separate`` the two calls one after the other."""
        if separate:
            self.append()
            self.check()
        elif self.fp8:
            self.fkv.kv_append_fp8_tag_check(self.k_new, self.v_new, self.slots_new, self.k_scale, self.v_scale,
                                             self.k_cache, self.v_cache, self.page_tags, self.indptr, self.indices,
                                             self.expected, self.mask)
        else:
            self.fkv.kv_append_bf16_tag_check(self.k_new, self.v_new, self.slots_new, self.k_cache, self.v_cache,
                                              self.page_tags, self.indptr, self.indices, self.expected, self.mask)

    def attend(self, with_mask=True):
        self.fkv.paged_decode_attn(self.q, self.k_cache, self.v_cache, self.indptr, self.indices, self.seq_lens,
                                   self.sm, self.out, self.ws, k_scale=self.k_scale if self.fp8 else None,
                                   v_scale=self.v_scale if self.fp8 else None,
                                   abort_mask=self.mask if with_mask else None)

    def repeat_identical(self, calls=8):
        """Bytes of the attention output over ``calls`` repeated calls on the
        step's final cache and mask, between writes that evict L2: True if
        every call gave the same bytes."""
        torch = self.torch
        flush = torch.empty(64 * 2 ** 20, dtype=torch.float32, device=self.device)
        ref = None
        same = True
        for i in range(calls):
            flush.fill_(float(i))
            self.attend(True)
            torch.cuda.synchronize(self.device)
            got = self.out.view(torch.int16).clone()
            if ref is None:
                ref = got
            else:
                same = same and bool(torch.equal(got, ref))
        return same

    def launches_per_step(self, with_check=True):
        return 1 + self.fkv.kernels_per_call("paged_decode_attn")   # append (+ check), attention

    def attn_bytes(self):
        """Algorithmic bytes of one paged_decode_attn call on the live requests
        (the abort mask of the last check)."""
        return algorithmic_attn_bytes(self.db, self.kv, self.mask.cpu().numpy())

    def timed(self, steps, warmup, with_check=True, sampler=None, call_events=True):
        """Device time of ``steps`` steps and (``call_events``) the mean time of
        the attention calls within them, from a pair of events around each.
        An event recorded between two launches stops the second one from
        starting while the first runs (programmatic dependent launch), so a
        step timed with per-call events is a few microseconds longer than
        the same step without them; ``call_events=False`` times the steps
        alone (the attention mean is then None)."""
        torch = self.torch
        stream = torch.cuda.current_stream(self.device)
        for _ in range(warmup):
            self.append_check() if with_check else self.append()
            self.attend(with_check)
        torch.cuda.synchronize(self.device)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize(self.device)
        ctx = sampler if sampler is not None else _Null()
        with ctx:
            t0.record(stream)
            for i in range(steps):
                self.append_check() if with_check else self.append()
                if call_events:
                    ev[i][0].record(stream)
                self.attend(with_check)
                if call_events:
                    ev[i][1].record(stream)
            t1.record(stream)
            torch.cuda.synchronize(self.device)
        barrier()
        total_ms = t0.elapsed_time(t1)
        attn_ms = float(np.mean([a.elapsed_time(b) for a, b in ev])) if call_events else None
        return total_ms, attn_ms

    def graph(self, with_check=True, checks_only=0, attn_only=False, separate=False, repeat=1):
        """One step (or ``checks_only`` back-to-back checks, or the attention
        call alone) captured in a CUDA graph, so host launch cost is out of
        the measurement; ``repeat`` steps back to back in the one graph, as a
        serving loop runs them (graph launches themselves are paced in ~2 us
        steps, which would swamp a step of a few tens of us).  ``separate``:
        the check as its own launch after the append instead of inside the
        append's launch."""
        torch = self.torch
        if attn_only:
            one = lambda: self.attend(True)
        elif checks_only:
            one = lambda: [self.check() for _ in range(checks_only)]
        elif with_check:
            one = lambda: (self.append_check(separate), self.attend(True))
        else:
            one = lambda: (self.append(), self.attend(False))
        body = lambda: [one() for _ in range(repeat)]
        body()                                    # one-time set-up happens outside the capture
        torch.cuda.synchronize(self.device)
        s = torch.cuda.Stream(self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            body()
        torch.cuda.synchronize(self.device)
        return g

    def replay_ms(self, g, steps, warmup):
        """Device time of ``steps`` back-to-back replays of a captured graph."""
        torch = self.torch
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize(self.device)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(steps):
            g.replay()
        t1.record()
        torch.cuda.synchronize(self.device)
        return t0.elapsed_time(t1)

    def timed_graph(self, steps, warmup, with_check=True, checks_only=0, attn_only=False, repeat=1):
        """Device time of ``steps`` replays of the captured step (``repeat``
        steps per replay: divide by steps * repeat for one step)."""
        torch = self.torch
        g = self.graph(with_check, checks_only, attn_only, repeat=repeat)
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize(self.device)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        t0.record()
        for _ in range(steps):
            g.replay()
        t1.record()
        torch.cuda.synchronize(self.device)
        barrier()
        return t0.elapsed_time(t1)

    def timed_cold(self, reps, warmup, attn_only=False):
        """Median time of one captured step (append + check + attention, or
        the attention call alone) with L2 flushed before each: a read of twice
        the L2 size between steps, so the step reads its KV, page table and
        queries from HBM (a read, not a write, leaves no dirty lines for the
        step to write back)."""
        torch = self.torch
        g = self.graph(True, 0, attn_only)
        l2 = int(getattr(torch.cuda.get_device_properties(self.device), "L2_cache_size", 0)) or (128 << 20)
        flush = torch.ones(2 * l2 // 4, dtype=torch.int32, device=self.device)
        sink = torch.empty((), dtype=torch.int32, device=self.device)
        for _ in range(warmup):
            torch.amax(flush, dim=0, out=sink)
            g.replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize(self.device)
        for a, b in ev:
            torch.amax(flush, dim=0, out=sink)
            a.record()
            g.replay()
            b.record()
        torch.cuda.synchronize(self.device)
        del flush
        return float(np.median([a.elapsed_time(b) for a, b in ev]))

    def time_prefill(self, reps=5):
        """Bulk write of the whole cached context as a prefill would hand it
        over: kv_calibrate_scales on the bf16 prompt, then kv_append_fp8 of
        every token (rewrites the same bytes).  Each call is timed in a run
        of its own (median of ``reps`` after one untimed call): right after a
        bulk append, a calibration first pays for writing back the append's
        dirty L2 lines."""
        torch, fkv = self.torch, self.fkv
        db = self.db
        ks = torch.empty_like(self.k_scale)
        vs = torch.empty_like(self.v_scale)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

        def run(call):
            ts = []
            for _ in range(reps + 1):
                ev[0].record()
                call()
                ev[1].record()
                torch.cuda.synchronize(self.device)
                ts.append(ev[0].elapsed_time(ev[1]))
            return float(np.median(ts[1:]))

        cal_ms = run(lambda: fkv.kv_calibrate_scales(db.k_src, db.v_src, ks, vs))
        app_ms = run(lambda: fkv.kv_append_fp8(db.k_src, db.v_src, db.slots_src, ks, vs, self.k_cache,
                                               self.v_cache))
        ntok = int(db.slots_src.numel())
        src = 2 * ntok * self.Hkv * self.D * 2
        same = bool(torch.equal(ks, self.k_scale) and torch.equal(vs, self.v_scale))
        return {"tokens": ntok, "calibrate_ms": cal_ms, "calibrate_gbs": src / (cal_ms * 1e6),
                "bulk_append_ms": app_ms, "bulk_append_gbs": (src + src // 2) / (app_ms * 1e6),
                "scales_equal_harness": same}

    def time_realloc(self, frac, reps):
        """kv_page_realloc of a seeded ``frac`` of the in-use pages, with and
        without the scrub of their K and V bytes (CUDA-graph timed)."""
        torch, fkv = self.torch, self.fkv
        rng = np.random.default_rng(7)
        ind = self.db.pt.indices
        moved = np.sort(rng.choice(ind, size=max(1, round(frac * ind.size)), replace=False)).astype(np.int32)
        pages = torch.from_numpy(moved).to(self.device)
        new = torch.zeros(moved.size, dtype=torch.int32, device=self.device)
        res = {"pages": int(moved.size)}
        for name, kc, vc in (("tags_only", None, None), ("with_scrub", self.k_cache, self.v_cache)):
            fkv.kv_page_realloc(self.page_tags, pages, new, kc, vc)
            torch.cuda.synchronize(self.device)
            s = torch.cuda.Stream(self.device)
            s.wait_stream(torch.cuda.current_stream(self.device))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for _ in range(10):
                    fkv.kv_page_realloc(self.page_tags, pages, new, kc, vc)
            g.replay()
            torch.cuda.synchronize(self.device)
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record()
            for _ in range(reps):
                g.replay()
            t1.record()
            torch.cuda.synchronize(self.device)
            us = 1e3 * t0.elapsed_time(t1) / (10 * reps)
            res[name + "_us"] = us
        page_bytes = 2 * self.Hkv * self.S * self.D * (1 if self.fp8 else 2)
        res["scrub_gbs"] = moved.size * page_bytes / (res["with_scrub_us"] * 1e3)
        return res

    def timed_e2e(self, steps, warmup):
        """The step through host buffers: every step copies all of its inputs
        (queries, the new token's K/V and slot, seq_lens, the page table and
        both tag arrays) from pinned host memory and reads the output and abort
        mask back.  Inputs of a step are packed in one buffer (one copy each
        way) and double-buffered on a copy stream, so step i+1's inputs and
        step i-1's results move while step i computes."""
        torch, fkv = self.torch, self.fkv
        dev = self.device
        srcs = [self.q, self.k_new, self.v_new, self.slots_new, self.seq_lens, self.indptr, self.indices,
                self.expected, self.page_tags]
        offs, tot = [], 0
        for x in srcs:
            offs.append(tot)
            tot += (x.numel() * x.element_size() + 255) // 256 * 256
        out_bytes = self.out.numel() * self.out.element_size()
        obytes = out_bytes + self.mask.numel()
        d_in = [torch.empty(tot, dtype=torch.uint8, device=dev) for _ in range(2)]
        h_in = [torch.empty(tot, dtype=torch.uint8).pin_memory() for _ in range(2)]
        d_out = [torch.empty(obytes, dtype=torch.uint8, device=dev) for _ in range(2)]
        h_out = [torch.empty(obytes, dtype=torch.uint8).pin_memory() for _ in range(2)]

        def views(buf):
            v = []
            for x, o in zip(srcs, offs):
                n = x.numel() * x.element_size()
                v.append(buf[o:o + n].view(x.dtype).view(x.shape))
            return v

        for b in range(2):                       # the host holds the step's inputs
            for hv, x in zip(views(h_in[b]), srcs):
                hv.copy_(x.cpu())
        dv = [views(d_in[b]) for b in range(2)]
        ov = [(d_out[b][:out_bytes].view(torch.bfloat16).view(self.out.shape), d_out[b][out_bytes:]) for b in range(2)]
        comp = torch.cuda.current_stream(dev)
        cp = torch.cuda.Stream(dev)
        h2d = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]

        def step(i):
            b = i & 1
            q, kn, vn, sl, seq, indptr, ind, exp, tags = dv[b]
            out, mask = ov[b]
            comp.wait_event(h2d[b])
            if self.fp8:
                fkv.kv_append_fp8_tag_check(kn, vn, sl, self.k_scale, self.v_scale, self.k_cache, self.v_cache,
                                            tags, indptr, ind, exp, mask)
            else:
                fkv.kv_append_bf16_tag_check(kn, vn, sl, self.k_cache, self.v_cache, tags, indptr, ind, exp, mask)
            fkv.paged_decode_attn(q, self.k_cache, self.v_cache, indptr, ind, seq, self.sm, out, self.ws,
                                  k_scale=self.k_scale if self.fp8 else None,
                                  v_scale=self.v_scale if self.fp8 else None, abort_mask=mask)
            done[b].record(comp)
            with torch.cuda.stream(cp):
                cp.wait_event(done[b])
                h_out[b].copy_(d_out[b], non_blocking=True)      # this step's results
                d_in[b].copy_(h_in[b], non_blocking=True)        # inputs of step i + 2
                h2d[b].record(cp)

        def run(n):
            with torch.cuda.stream(cp):
                for b in range(2):
                    d_in[b].copy_(h_in[b], non_blocking=True)
                    h2d[b].record(cp)
            for i in range(n):
                step(i)
            cp.synchronize()

        run(warmup)
        torch.cuda.synchronize(dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        t0.record(cp)
        run(steps)
        t1.record(cp)
        torch.cuda.synchronize(dev)
        barrier()
        last = (steps - 1) & 1                   # the host holds the last step's output
        assert torch.equal(ov[last][0].view(torch.int16).reshape(-1).cpu(), h_out[last][:out_bytes].view(torch.int16))
        return t0.elapsed_time(t1), tot, obytes


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


_PG = None


def barrier():
    if _PG is not None:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x):
    """The largest of every rank's x (the job's time is its slowest rank's)."""
    if _PG is None:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# CPU oracle on a bounded sample
# ----------------------------------------------------------------------------
def oracle_sample(db, kv, n_requests, start=0, threads=1):
    """Time the oracle's step (append the new token, check tags, attend, all
    query heads) for ``n_requests`` requests of the batch, their cached context
    pre-encoded by the oracle itself.  Returns (seconds, requests, sample text),
    plus (seconds, threads used) of the same step with the attention rows split
    over ``threads`` host threads when ``threads`` > 1."""
    import oracle
    from fp8_paged_kv_decode_gb300 import workloads as W
    orc = oracle.default()
    B = db.wl.batch
    reqs = [(start + i) % B for i in range(n_requests)]
    cr = W.compact_requests(db, reqs)
    S, Hkv, D = db.wl.page_size, db.wl.num_kv_heads, db.wl.head_dim
    fp8 = kv == "fp8"
    dt = np.uint8 if fp8 else np.uint16
    kc = np.zeros((cr.num_pages, Hkv, S, D), dt)
    vc = np.zeros((cr.num_pages, Hkv, S, D), dt)
    # context (all but each request's last token) is in the cache before the
    # step; encoding it is set-up, not timed, so it is split over the host's
    # threads (disjoint slots; the oracle's C call releases the interpreter lock)
    import concurrent.futures as cf
    new_idx = np.cumsum(cr.seq_lens.astype(np.int64)) - 1
    ctx_sel = np.ones(cr.slots.size, bool)
    ctx_sel[new_idx] = False
    ctx_idx = np.flatnonzero(ctx_sel)

    def encode(part):
        if fp8:
            orc.kv_append_fp8(cr.k_tokens[part], cr.v_tokens[part], cr.slots[part], db.k_scale, db.v_scale, kc, vc)
        else:
            orc.kv_append_bf16(cr.k_tokens[part], cr.v_tokens[part], cr.slots[part], kc, vc)

    chunks = [c for c in np.array_split(ctx_idx, max(1, threads)) if c.size]
    with cf.ThreadPoolExecutor(max(1, len(chunks))) as ex:
        list(ex.map(encode, chunks))
    tags = db.pt.page_tags[cr.orig_pages]
    exp = np.concatenate([db.pt.expected_tags[db.pt.indptr[r]:db.pt.indptr[r + 1]] for r in reqs])
    t0 = time.perf_counter()
    if fp8:
        orc.kv_append_fp8(cr.k_tokens[new_idx], cr.v_tokens[new_idx], cr.slots[new_idx], db.k_scale, db.v_scale, kc, vc)
    else:
        orc.kv_append_bf16(cr.k_tokens[new_idx], cr.v_tokens[new_idx], cr.slots[new_idx], kc, vc)
    mask = orc.kv_page_tag_check(tags, cr.indptr, cr.indices, exp)
    orc.paged_decode_attn(cr.q, kc, vc, cr.indptr, cr.indices, cr.seq_lens, 1.0 / np.sqrt(D),
                          k_scale=db.k_scale if fp8 else None, v_scale=db.v_scale if fp8 else None, abort_mask=mask)
    dt_s = time.perf_counter() - t0
    toks = int(cr.seq_lens.sum())
    text = "%d of %d requests (%d context tokens, all %d query heads), one step each, 1 thread" % (
        len(reqs), B, toks, db.wl.num_q_heads)
    if threads <= 1:
        return dt_s, len(reqs), text, dt_s, 1
    # The same step with the attention rows ((request, query head) pairs) split
    # over host threads; the oracle's C call releases the interpreter lock.
    rows = np.arange(len(reqs) * db.wl.num_q_heads, dtype=np.int32)
    parts = [c for c in np.array_split(rows, threads) if c.size]

    def attend(part):
        return orc.paged_decode_attn(cr.q, kc, vc, cr.indptr, cr.indices, cr.seq_lens, 1.0 / np.sqrt(D),
                                     k_scale=db.k_scale if fp8 else None, v_scale=db.v_scale if fp8 else None,
                                     abort_mask=mask, rows=part)

    with cf.ThreadPoolExecutor(len(parts)) as ex:
        t0 = time.perf_counter()
        if fp8:
            orc.kv_append_fp8(cr.k_tokens[new_idx], cr.v_tokens[new_idx], cr.slots[new_idx], db.k_scale, db.v_scale,
                              kc, vc)
        else:
            orc.kv_append_bf16(cr.k_tokens[new_idx], cr.v_tokens[new_idx], cr.slots[new_idx], kc, vc)
        mask = orc.kv_page_tag_check(tags, cr.indptr, cr.indices, exp)
        list(ex.map(attend, parts))
        dt_t = time.perf_counter() - t0
    return dt_s, len(reqs), text, dt_t, len(parts)


# ----------------------------------------------------------------------------
def algorithmic_attn_bytes(db, kv, mask):
    """Algorithmic bytes of one paged_decode_attn call on the live requests
    (mask[r] == 0): K and V of every attended token, q and out, page ids and
    seq_lens."""
    wl = db.wl
    live = np.asarray(mask) == 0
    seq = db.seq_lens.astype(np.int64)
    es = 1 if kv == "fp8" else 2
    kvb = int((seq[live] * wl.num_kv_heads * wl.head_dim * 2 * es).sum())
    pages = int(((seq[live] + wl.page_size - 1) // wl.page_size).sum())
    qo = wl.batch * wl.num_q_heads * wl.head_dim * 2 * 2
    return kvb + qo + 4 * pages + 4 * wl.batch, int(seq[live].sum())


def arm_config(wl, db, kv, world, attn_bytes):
    """The ``config`` of the JSON line, the same for both arms."""
    return {"workload": workload_text(wl, db), "kv_dtype": "fp8_e4m3" if kv == "fp8" else "bf16",
            "global_batch": world * wl.batch,
            "step": "kv_append_%s_tag_check (append + integrity check, one launch) + paged_decode_attn (one layer)"
                    % kv,
            "l2": "inputs larger than L2 (%.2f GB of KV read per step); no flush" % (attn_bytes / 1e9),
            "parallelism": "replicas x%d" % world}


def workload_text(wl, db):
    return ("%s: %d req, %d q / %d kv heads, head_dim %d, page %d, ctx %s, %d tokens attended per step"
            % (wl.name, wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, wl.ctx,
               int(db.seq_lens.sum())))


def run_reference(args):
    """Reference arm: the CPU oracle as it stands.  Each step is one request's
    decode step -- its new token appended, its pages checked, all its query
    heads attended, the rows split over the host's threads -- cycling over the
    first few requests of the workload; their cached context is encoded by
    the oracle before timing."""
    world, rank, local = dist_env()
    if rank != 0:
        return
    import concurrent.futures as cf
    import torch
    import oracle
    from fp8_paged_kv_decode_gb300 import workloads as W
    orc = oracle.default()
    wl = selected_workload(W, args)
    device = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    db = W.device_batch(wl, device, seed=wl.seed)
    n_req = min(4, wl.batch)
    cr = W.compact_requests(db, list(range(n_req)))
    S, Hkv, D, Hq = wl.page_size, wl.num_kv_heads, wl.head_dim, wl.num_q_heads
    kc = np.zeros((cr.num_pages, Hkv, S, D), np.uint8)
    vc = np.zeros((cr.num_pages, Hkv, S, D), np.uint8)
    new_idx = np.cumsum(cr.seq_lens.astype(np.int64)) - 1
    ctx_sel = np.ones(cr.slots.size, bool)
    ctx_sel[new_idx] = False
    orc.kv_append_fp8(cr.k_tokens[ctx_sel], cr.v_tokens[ctx_sel], cr.slots[ctx_sel], db.k_scale, db.v_scale, kc, vc)
    tags = db.pt.page_tags[cr.orig_pages]
    exp = np.concatenate([db.pt.expected_tags[db.pt.indptr[r]:db.pt.indptr[r + 1]] for r in range(n_req)])
    sm = 1.0 / np.sqrt(D)
    threads = max(1, os.cpu_count() or 1)
    total = 0.0
    with cf.ThreadPoolExecutor(threads) as ex:
        for i in range(args.warmup + args.steps):
            j = i % n_req
            parts = [p for p in np.array_split(np.arange(j * Hq, (j + 1) * Hq, dtype=np.int32), threads) if p.size]
            t0 = time.perf_counter()
            orc.kv_append_fp8(cr.k_tokens[new_idx[j]:new_idx[j] + 1], cr.v_tokens[new_idx[j]:new_idx[j] + 1],
                              cr.slots[new_idx[j]:new_idx[j] + 1], db.k_scale, db.v_scale, kc, vc)
            mask = orc.kv_page_tag_check(tags, cr.indptr, cr.indices, exp)
            list(ex.map(lambda rows: orc.paged_decode_attn(cr.q, kc, vc, cr.indptr, cr.indices, cr.seq_lens, sm,
                                                           k_scale=db.k_scale, v_scale=db.v_scale,
                                                           abort_mask=mask, rows=rows), parts))
            if i >= args.warmup:
                total += time.perf_counter() - t0
    value = args.steps / total                 # decode tokens/s: one request's token per step
    sample = ("CPU oracle, one request's decode step per step (append, tag check, all %d query heads), cycling "
              "over the first %d requests (%d context tokens); attention rows over %d host threads"
              % (Hq, n_req, int(cr.seq_lens.sum()), threads))
    # the same config as the GPU arm's line: its algorithmic bytes from the
    # whole batch's abort mask, which the oracle computes here
    full_mask = orc.kv_page_tag_check(db.pt.page_tags, db.pt.indptr, db.pt.indices, db.pt.expected_tags)
    attn_bytes, _ = algorithmic_attn_bytes(db, "fp8", full_mask)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": arm_config(wl, db, "fp8", world, attn_bytes),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# The attention call on every workload: FP8 on all five, BF16 where the
# workload compares the two, and the integrity workload both as specified
# (1% of pages stale, most requests aborted) and with no stale page.
CONFIG_LEGS = [("tiny_gqa4", "fp8", None), ("uniform_gqa8_8k", "fp8", None), ("uniform_gqa8_8k", "bf16", None),
               ("pages_shaped_64req", "fp8", None), ("pages_shaped_64req", "bf16", None),
               ("long_ctx_131k", "fp8", None), ("integrity_256req", "fp8", None), ("integrity_256req", "fp8", 0.0)]


def l2_bytes(torch, device):
    return int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0)) or (128 << 20)


def config_table(device, rank, reps, warmup, peak, reuse=None):
    """paged_decode_attn on each entry of CONFIG_LEGS: the call's device time
    (CUDA-graph replays of the call alone), its algorithmic bytes on the live
    requests, GB/s and the fraction of the measured copy peak, plus the DRAM
    traffic of one launch from the committed ncu record when it matches the
    current kernel.  Working sets below twice the L2 size are timed with L2
    flushed before every call (a read of twice its size); larger ones stream
    from HBM on every call anyway and are timed back to back."""
    import dataclasses
    import torch
    from fp8_paged_kv_decode_gb300 import workloads as W
    l2 = l2_bytes(torch, device)
    out = {}
    for name, kv, stale in CONFIG_LEGS:
        wl = W.WORKLOADS[name]
        key = name if stale is None else "%s_stale%g" % (name, stale)
        if stale is not None:
            wl = dataclasses.replace(wl, name=key, stale_frac=stale)
        db = reuse if (reuse is not None and stale is None and reuse.wl == wl) else \
            W.device_batch(wl, device, seed=wl.seed + rank)
        st = Step(db, kv, device)
        st.check()                                   # the abort mask the timed calls read
        torch.cuda.synchronize(device)
        nbytes, attended = st.attn_bytes()
        live = int(wl.batch - int(st.mask.sum().item()))
        warm_us = 1e3 * max_over_ranks(st.timed_graph(reps, warmup, attn_only=True)) / reps
        cold_us = 1e3 * max_over_ranks(st.timed_cold(reps, warmup, attn_only=True))
        flushed = nbytes < 2 * l2
        us = cold_us if flushed else warm_us
        gbs = nbytes / (us * 1e3)
        tr = recorded_traffic(kv, key)
        extra = {}
        if name == "long_ctx_131k":
            # spread of the logits q.k / sqrt(d) the workload is drawn for
            # (std ~4): request 0, one query head per KV head, its first 4096 tokens
            q = db.q[0, ::wl.group].float()
            k = db.k_src[:4096].float()
            extra["logit_std"] = float((torch.einsum("hd,thd->th", q, k) / np.sqrt(wl.head_dim)).std())
        out["%s.%s" % (key, kv)] = {**extra,
            "workload": workload_text(wl, db), "kv": kv, "live_requests": live,
            "attn_us": us, "attn_us_back_to_back": warm_us, "attn_us_l2_flushed": cold_us,
            "timing": "L2 flushed before each call" if flushed else "back to back (working set > 2x L2)",
            "algorithmic_bytes": nbytes, "gbs": gbs, "frac": gbs / peak, "frac_of_8tbs": gbs / 8000.0,
            "tokens_per_s": live / (us * 1e-6), "context_tokens_per_s": attended / (us * 1e-6),
            "traffic": tr["dram_bytes_per_call"] if tr else None,
            "traffic_ratio": tr["dram_bytes_per_call"] / nbytes if tr else None}
        del st
        if db is not reuse:
            del db
        torch.cuda.empty_cache()
    return out


def bootstrap_ci(x, stat, n=10000, seed=0):
    """95% percentile-bootstrap interval of ``stat`` over the samples ``x``."""
    rng = np.random.default_rng(seed)
    x = np.asarray(x, np.float64)
    b = np.array([stat(x[rng.integers(0, x.size, x.size)]) for _ in range(n)])
    return [float(np.percentile(b, 2.5)), float(np.percentile(b, 97.5))]


def integrity_overhead(st, pairs, steps, warmup, repeat=1):
    """Cost of the tag check in the decode step.  Three CUDA-graph-captured
    steps -- without the check, with the check in the append's launch (the
    step as run), with the check as a launch of its own -- are timed in
    ``pairs`` interleaved rounds (the order rotates between rounds), ``steps``
    replays each; per round the overhead of each variant is (with - without)
    / without.  Returns the per-round figures, their median and mean and 95%
    bootstrap intervals of both."""
    graphs = {"off": st.graph(False, repeat=repeat), "on": st.graph(True, repeat=repeat),
              "separate": st.graph(True, separate=True, repeat=repeat)}
    for g in graphs.values():
        st.replay_ms(g, 0, warmup)
    times = {k: [] for k in graphs}
    order = list(graphs)
    for i in range(pairs):
        for k in order[i % 3:] + order[:i % 3]:
            times[k].append(max_over_ranks(st.replay_ms(graphs[k], steps, 2)) / (steps * repeat))
    t = {k: np.array(v) for k, v in times.items()}
    res = {"rounds": pairs, "steps_per_timing": steps * repeat, "steps_per_graph": repeat,
           "step_ms_without_check_median": float(np.median(t["off"])),
           "step_ms_with_check_median": float(np.median(t["on"])),
           "step_ms_with_separate_check_median": float(np.median(t["separate"]))}
    for k, name in (("on", ""), ("separate", "separate_launch_")):
        pct = 100.0 * (t[k] - t["off"]) / t["off"]
        res.update({name + "overhead_pct_per_round": [float(v) for v in pct],
                    name + "overhead_pct_median": float(np.median(pct)),
                    name + "overhead_pct_median_ci95": bootstrap_ci(pct, np.median),
                    name + "overhead_pct_mean": float(pct.mean()),
                    name + "overhead_pct_mean_ci95": bootstrap_ci(pct, np.mean)})
    return res


def capacity_rows(db, device, steps, warmup):
    """A per-layer KV budget that holds the first 32 requests of the 64-request
    workload in BF16; how many requests each KV dtype admits under it, and the
    decode step (append + check + attention) at concurrency 1..64 for both,
    for the concurrencies each dtype can hold.  Steps are CUDA-graph captured
    so small batches measure GPU time, not host launch cost; repeated steps
    over the same pages keep a small batch's KV in L2, so each row also gives
    the step time with L2 flushed before every step."""
    import torch
    from fp8_paged_kv_decode_gb300 import workloads as W
    wl = db.wl
    npages = np.diff(db.pt.indptr)
    page_fp8 = 2 * wl.num_kv_heads * wl.page_size * wl.head_dim
    page_bf16 = 2 * page_fp8
    budget = int(npages[:32].sum()) * page_bf16
    adm = {"fp8": W.admitted(page_fp8, npages, budget), "bf16": W.admitted(page_bf16, npages, budget)}
    rows = []
    for c in sorted({c for c in (1, 2, 4, 8, 16, 32, 48, 64, adm["fp8"], adm["bf16"]) if 0 < c <= npages.size}):
        row = {"requests": c, "tokens": int(db.seq_lens[:c].sum())}
        sub = W.subset_batch(db, c)
        for kv in ("fp8", "bf16"):
            if c > adm[kv]:
                row[kv] = None                      # does not fit the budget
                continue
            st = Step(sub, kv, device)
            rep = 20 if c <= 16 else 1                              # short steps: many per graph
            n = max(5, steps // rep)
            tot = st.timed_graph(n, warmup, repeat=rep) * steps / (n * rep)   # whole step, CUDA graph
            attn = st.timed_graph(n, warmup, attn_only=True, repeat=rep) * steps / (n * rep)
            cold = st.timed_cold(max(20, steps // 5), warmup)         # L2 flushed before each step
            row[kv] = {"step_ms": tot / steps, "tokens_per_s": c / (tot / steps / 1e3), "attn_ms": attn / steps,
                       "step_ms_cold_l2": cold}
            del st
            torch.cuda.empty_cache()
        rows.append(row)
    peak = {kv: max((r[kv]["tokens_per_s"] for r in rows if r[kv]), default=0.0) for kv in ("fp8", "bf16")}
    return {"workload": workload_text(wl, db), "budget_bytes_per_layer": budget,
            "budget": "BF16 pages of the first 32 requests", "admitted": adm,
            "resident_tokens": {kv: int(db.seq_lens[:adm[kv]].sum()) for kv in adm},
            "steps_per_timing": steps, "rows": rows, "peak_tokens_per_s": peak,
            "fp8_peak_over_bf16_peak": peak["fp8"] / peak["bf16"]}


def capacity_sweep(args):
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    from fp8_paged_kv_decode_gb300 import workloads as W
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    fkv.load_library()
    db = W.device_batch(W.WORKLOADS[HEADLINE], device)
    print(json.dumps({"capacity_sweep": capacity_rows(db, device, max(50, args.steps // 10), args.warmup)}),
          flush=True)


def configs_only(args):
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    fkv.load_library()
    reps = args.config_reps or max(10, min(200, args.steps))
    peak, kind = peak_hbm()
    print(json.dumps({"configs": config_table(device, 0, reps, args.warmup, peak), "peak_gbs": peak,
                      "peak_kind": kind}), flush=True)


def shared_prefix(args):
    """The 64-request workload with every request's first m pages replaced by
    request 0's (a shared prompt prefix of m*64 tokens): decode step time,
    bytes attended per second (each request's reads) and unique KV bytes
    per second (what HBM must supply at least)."""
    import dataclasses
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    from fp8_paged_kv_decode_gb300 import workloads as W
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    fkv.load_library()
    wl = W.WORKLOADS[HEADLINE]
    db = W.device_batch(wl, device)
    n0 = int(db.pt.indptr[1] - db.pt.indptr[0])
    steps = max(100, args.steps // 5)
    rows = []
    for m in sorted({0, 8, 32, 64, n0 - 1}):
        sub = dataclasses.replace(db, pt=W.share_prefix(db.pt, m))
        st = Step(sub, "fp8", device)
        tot = st.timed_graph(steps, args.warmup)
        attn = st.timed_graph(steps, args.warmup, attn_only=True) / steps
        attended, _ = st.attn_bytes()
        ind = sub.pt.indices
        used = np.concatenate([ind[sub.pt.indptr[r]:sub.pt.indptr[r] + (int(sub.seq_lens[r]) + wl.page_size - 1)
                                   // wl.page_size] for r in range(wl.batch)])
        unique = np.unique(used).size * 2 * wl.num_kv_heads * wl.page_size * wl.head_dim
        rows.append({"shared_prefix_tokens": m * wl.page_size, "step_ms": tot / steps, "attn_ms": attn,
                     "attended_gbs": attended / (attn * 1e6), "unique_kv_bytes": int(unique),
                     "unique_gbs": unique / (attn * 1e6)})
        del st
        torch.cuda.empty_cache()
    print(json.dumps({"shared_prefix": {"workload": workload_text(wl, db), "rows": rows}}), flush=True)


def main():
    global _PG
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.capacity_sweep:
        capacity_sweep(args)
        return
    if args.shared_prefix:
        shared_prefix(args)
        return
    if args.configs_only:
        configs_only(args)
        return
    world, rank, local = dist_env()
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        _PG = True
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    import fp8_paged_kv_decode_gb300 as fkv
    from fp8_paged_kv_decode_gb300 import workloads as W
    if rank == 0 and not os.path.exists(fkv.library_path()):
        from fp8_paged_kv_decode_gb300 import _build
        _build.build()
    barrier()
    fkv.load_library()

    wl = selected_workload(W, args)
    db = W.device_batch(wl, device, seed=wl.seed + rank)
    fp8 = Step(db, args.kv, device)
    fkv.device_error(clear=True)
    sampler = ClockSampler(local)
    # the headline run: K steps as a serving loop issues them, no events
    # between launches; then the same K steps again with events around every
    # attention call for the kernel's own duration (roofline)
    total_ms, _ = fp8.timed(args.steps, args.warmup, sampler=sampler, call_events=False)
    total_ms = max_over_ranks(total_ms)
    ev_total_ms, attn_ms = fp8.timed(args.steps, args.warmup)
    ev_total_ms, attn_ms = max_over_ranks(ev_total_ms), max_over_ranks(attn_ms)
    ms_per_step = total_ms / args.steps
    value = world * wl.batch * args.steps / (total_ms / 1e3)
    attn_bytes, attended = fp8.attn_bytes()
    peak, peak_kind = peak_hbm()
    achieved = attn_bytes / (attn_ms / 1e3) / 1e9
    traffic = recorded_traffic(args.kv, wl.name)

    e2e_steps = args.steps
    e2e_ms, bi, bo = fp8.timed_e2e(e2e_steps, max(3, args.warmup))
    e2e_ms = max_over_ranks(e2e_ms)
    e2e_value = world * wl.batch * e2e_steps / (e2e_ms / 1e3)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 KV -> f16 MMA, f32 accumulate" if args.kv == "fp8" else
        "bf16 KV -> bf16 MMA, f32 accumulate", "data": "synthetic",
        "config": arm_config(wl, db, args.kv, world, attn_bytes),
        "roofline": {"bound": "hbm", "kernel": "paged_decode_attn (plan + split attention with fused merge)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "traffic": traffic["dram_bytes_per_call"] if traffic else None,
                     "algorithmic_bytes": attn_bytes, "attn_ms": attn_ms,
                     "frac_of_8tbs": achieved / 8000.0,
                     "timing": "mean of CUDA event pairs around each of the %d attention calls of a second run of "
                               "the %d timed steps (%.4f ms per step with those events)"
                               % (args.steps, args.steps, ev_total_ms / args.steps)},
        "attention_tokens_per_s": world * wl.batch / (attn_ms / 1e3),
        "context_tokens_per_s": world * attended / (attn_ms / 1e3),
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                "steps": e2e_steps},
        "gpu_launches": args.steps * fp8.launches_per_step(),
        "clocks": sampler.summary(),
        "attention_repeat_bytes_identical": fp8.repeat_identical(),
    }

    if not args.skip_extras and args.kv == "fp8":
        line["prefill_bulk_write"] = fp8.time_prefill()
        bf = Step(db, "bf16", device)
        bms, _ = bf.timed(max(10, args.steps // 2), args.warmup, call_events=False)
        _, battn = bf.timed(max(10, args.steps // 2), args.warmup)
        bms, battn = max_over_ranks(bms), max_over_ranks(battn)
        bbytes, _ = bf.attn_bytes()
        bach = bbytes / (battn / 1e3) / 1e9
        line["bf16_kv"] = {"value": world * wl.batch * max(10, args.steps // 2) / (bms / 1e3), "unit": "tokens/s",
                           "ms_per_step": bms / max(10, args.steps // 2), "attn_ms": battn, "attn_gbs": bach,
                           "frac": bach / peak, "algorithmic_bytes": bbytes,
                           "traffic": (recorded_traffic("bf16", wl.name) or {}).get("dram_bytes_per_call")}
        line["fp8_over_bf16_attn_time"] = battn / attn_ms
        del bf
        torch.cuda.empty_cache()

        # integrity check cost: the 0%-stale variant of integrity_256req with
        # and without the check, each step captured in a CUDA graph; repeated
        # interleaved pairs give the spread
        import dataclasses
        iw = W.WORKLOADS["integrity_256req"]
        iw0 = dataclasses.replace(iw, stale_frac=0.0)
        idb = W.device_batch(iw0, device, seed=iw.seed + rank)
        ist = Step(idb, "fp8", device)
        n_i = max(200, args.steps // 2)
        pairs = integrity_overhead(ist, 10, n_i, args.warmup)
        reps = 20
        chk_ms = max_over_ranks(ist.timed_graph(n_i // 10 + 1, 3, checks_only=reps))
        chk_us = 1e3 * chk_ms / ((n_i // 10 + 1) * reps)
        clean_aborts = int(ist.mask.sum().item())
        del ist, idb
        torch.cuda.empty_cache()
        # the workload as specified: 1% of in-use pages reallocated (stale)
        sdb = W.device_batch(iw, device, seed=iw.seed + rank)
        sst = Step(sdb, "fp8", device)
        st_ms = max_over_ranks(sst.timed_graph(n_i, args.warmup, with_check=True))
        realloc = sst.time_realloc(frac=0.01, reps=max(20, n_i // 10))
        # the same rounds at concurrency 1, 2, 4 and 8 (the first N requests;
        # the pages report the check's cost at these concurrencies)
        cdb = W.device_batch(iw0, device, seed=iw.seed + rank)
        by_conc = {}
        for n in (1, 2, 4, 8):
            cst = Step(W.subset_batch(cdb, n), "fp8", device)
            r = integrity_overhead(cst, 10, max(10, n_i // 20), args.warmup, repeat=20)
            by_conc[str(n)] = {k: r[k] for k in ("overhead_pct_median", "overhead_pct_median_ci95",
                                                 "separate_launch_overhead_pct_median",
                                                 "step_ms_without_check_median", "step_ms_with_check_median")}
            del cst
        del cdb
        torch.cuda.empty_cache()
        line["integrity_check"] = {
            "workload": workload_text(iw, sdb),
            "by_concurrency": by_conc,
            "overhead_variant": "same shape, 0%% stale pages (%d aborted); the check runs in the append's launch "
                                "(kv_append_fp8_tag_check), separate_launch_* as its own launch" % clean_aborts,
            "overhead_pct": pairs["overhead_pct_median"], **pairs,
            "check_kernel_us": chk_us,
            "check_share_of_step_pct": 100.0 * chk_us / (1e3 * pairs["step_ms_with_check_median"]),
            "stale_1pct": {"aborted_requests": int(sst.mask.sum().item()), "step_ms": st_ms / n_i},
            "device_realloc_1pct": realloc,
            "timing": "CUDA-graph-captured steps"}
        del sst, sdb
        torch.cuda.empty_cache()

        # every workload's attention call, and the capacity / concurrency sweep
        line["configs"] = config_table(device, rank, args.config_reps or max(20, min(200, args.steps)),
                                       args.warmup, peak, reuse=db)
        del fp8
        torch.cuda.empty_cache()
        # the sweep is defined on the headline workload as drawn; another
        # selected workload (or batch / page-size change) gets its own batch
        cdb = db if db.wl == W.WORKLOADS[HEADLINE] else W.device_batch(W.WORKLOADS[HEADLINE], device)
        line["capacity_sweep"] = capacity_rows(cdb, device, max(50, args.steps // 10), args.warmup)
        del cdb

    derr = fkv.device_error()
    if derr:
        line["device_error"] = derr
    if rank == 0:
        t0 = time.perf_counter()
        s, n, text, st, nt = oracle_sample(db, args.kv, args.cpu_requests, threads=os.cpu_count() or 1)
        line["cpu_baseline"] = {"value": n / s, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": text,
                                "threaded": {"value": n / st, "unit": "tokens/s", "cores": nt,
                                             "sample": "the same step, attention rows split over %d host threads"
                                                       % nt}}
        print(json.dumps(line), flush=True)
    if _PG is not None:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
