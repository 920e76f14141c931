"""Helpers shared by the GPU parity tests (argument plumbing only)."""
from __future__ import annotations

import os
import shutil
import subprocess

import numpy as np

from fp8_paged_kv_decode_gb300 import workloads as W

ABS_TOL = 2e-3
REL_TOL = 1e-2


def tol_fail(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Elements outside tolerance: an element fails only if it is off by more
    than 2e-3 absolute AND more than 1e-2 relative to the oracle."""
    err = np.abs(got.astype(np.float64) - ref)
    return (err > ABS_TOL) & (err > REL_TOL * np.abs(ref))


def assert_close(got, ref, what=""):
    bad = tol_fail(got, ref)
    if bad.any():
        i = np.argwhere(bad)[0]
        err = np.abs(got.astype(np.float64) - ref)
        raise AssertionError("%s: %d/%d outside tolerance; first at %s got %r want %r (max abs err %g)" % (
            what, int(bad.sum()), bad.size, tuple(i), float(got[tuple(i)]), float(ref[tuple(i)]), err.max()))


def dev(a, device="cuda", dtype=None):
    import torch
    x = torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return x.view(dtype) if dtype is not None else x


def bf16_out(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


class PagedCase:
    """A random paged batch: context lengths given, pages scattered over a pool
    with spare pages, values N(0,1) bf16, caches encoded by the oracle."""

    def __init__(self, orc, B, Hq, Hkv, S, seq, kv="fp8", seed=0, spare=7, q_std=1.0, extra_pages=0):
        rng = np.random.default_rng(seed)
        D = 128
        self.B, self.Hq, self.Hkv, self.S, self.D = B, Hq, Hkv, S, D
        self.seq = np.asarray(seq, dtype=np.int32)
        npages = (self.seq.astype(np.int64) + S - 1) // S + extra_pages
        used = int(npages.sum())
        self.P = used + spare
        perm = rng.permutation(self.P).astype(np.int32)
        self.indptr = np.concatenate([[0], np.cumsum(npages)]).astype(np.int32)
        self.indices = perm[:used].copy()
        ntok = int(self.seq.sum())
        kf = rng.standard_normal((max(ntok, 1), Hkv, D)).astype(np.float32)[:ntok]
        vf = rng.standard_normal((max(ntok, 1), Hkv, D)).astype(np.float32)[:ntok]
        self.q = W.bf16_bits((q_std * rng.standard_normal((B, Hq, D))).astype(np.float32))
        k_src, v_src = W.bf16_bits(kf), W.bf16_bits(vf)
        slots = []
        for r in range(B):
            pos = np.arange(int(self.seq[r]))
            slots.append(self.indices[self.indptr[r] + pos // S].astype(np.int64) * S + pos % S)
        slots = np.concatenate(slots) if slots else np.zeros(0, np.int64)
        self.fp8 = kv == "fp8"
        if self.fp8:
            ka = np.abs(W.bits_to_f32(k_src)).max(axis=(0, 2)) if ntok else np.zeros(Hkv, np.float32)
            va = np.abs(W.bits_to_f32(v_src)).max(axis=(0, 2)) if ntok else np.zeros(Hkv, np.float32)
            self.k_scale, self.v_scale = W.scale_from_amax(ka), W.scale_from_amax(va)
            # pool bytes outside written slots hold arbitrary (finite) codes
            self.kc = rng.integers(0, 0x7F, (self.P, Hkv, S, D)).astype(np.uint8)
            self.vc = rng.integers(0, 0x7F, (self.P, Hkv, S, D)).astype(np.uint8)
            orc.kv_append_fp8(k_src, v_src, slots, self.k_scale, self.v_scale, self.kc, self.vc)
        else:
            self.k_scale = self.v_scale = None
            self.kc = W.bf16_bits(rng.standard_normal((self.P, Hkv, S, D)).astype(np.float32))
            self.vc = W.bf16_bits(rng.standard_normal((self.P, Hkv, S, D)).astype(np.float32))
            orc.kv_append_bf16(k_src, v_src, slots, self.kc, self.vc)
        self.sm = 1.0 / np.sqrt(D)

    def oracle(self, orc, abort_mask=None, seq=None, indices=None):
        return orc.paged_decode_attn(self.q, self.kc, self.vc, self.indptr,
                                     self.indices if indices is None else indices,
                                     self.seq if seq is None else seq, self.sm,
                                     k_scale=self.k_scale, v_scale=self.v_scale, abort_mask=abort_mask)

    def gpu(self, abort_mask=None, seq=None, indices=None, kc=None, vc=None):
        import torch
        import fp8_paged_kv_decode_gb300 as fkv
        q = dev(self.q, dtype=torch.bfloat16)
        if self.fp8:
            kt, vt = dev(self.kc if kc is None else kc), dev(self.vc if vc is None else vc)
            ks, vs = dev(self.k_scale), dev(self.v_scale)
        else:
            kt = dev(self.kc if kc is None else kc, dtype=torch.bfloat16)
            vt = dev(self.vc if vc is None else vc, dtype=torch.bfloat16)
            ks = vs = None
        out = torch.full((self.B, self.Hq, self.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        ws = fkv.alloc_workspace(self.B, self.Hq, self.Hkv, fkv.KV_FP8_E4M3 if self.fp8 else fkv.KV_BF16)
        am = None if abort_mask is None else dev(np.asarray(abort_mask, np.uint8))
        fkv.paged_decode_attn(q, kt, vt, dev(self.indptr), dev(self.indices if indices is None else indices),
                              dev(self.seq if seq is None else np.asarray(seq, np.int32)), self.sm, out, ws,
                              k_scale=ks, v_scale=vs, abort_mask=am)
        torch.cuda.synchronize()
        return out


TESTS_DIR = os.path.dirname(os.path.abspath(__file__))
REPO_ROOT = os.path.dirname(TESTS_DIR)


def cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.isdir(os.path.join(cand, "include")):
            return cand
    nvcc = shutil.which("nvcc")
    return os.path.dirname(os.path.dirname(nvcc)) if nvcc else None


def build_c_program(source, exe):
    """Compile a plain C test program in tests/ against libfkv.so, the CUDA
    runtime and the C oracle (gcc, no fast-math); returns the executable."""
    import fp8_paged_kv_decode_gb300 as fkv
    lib = fkv.library_path()
    assert os.path.exists(lib), "libfkv.so is not built"
    cuda = cuda_home()
    assert cuda, "CUDA toolkit not found"
    libdir = os.path.dirname(lib)
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                    "-I", os.path.join(REPO_ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    os.path.join(TESTS_DIR, source), os.path.join(REPO_ROOT, "oracle", "fkv_oracle.c"),
                    "-o", exe, "-L", libdir, "-l:" + os.path.basename(lib),
                    "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm", "-Wl,-rpath," + libdir],
                   check=True)
    return exe
