"""Build libfkv.so in-tree with nvcc for sm_103a (GB300).

Each .cu file compiles to an object in parallel, then one shared library is
linked.  No fast-math: the e4m3 quantisation relies on IEEE division.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
LIB = os.path.join(PKG, "libfkv.so")
BUILD_DIR = os.path.join(PKG, "_build")
SOURCES = ["fkv_api.cu", "kv_append.cu", "tag_check.cu", "decode_attn.cu", "decode_attn_noalloc.cu", "page_realloc.cu",
           "kv_calibrate.cu", "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hs + [os.path.join(ROOT, "include", "fkv.h")]


def build(force: bool = False, verbose: bool = False, extra_flags=(), out_lib: str = LIB,
          build_dir: str = BUILD_DIR) -> str:
    """Compile every source (only what changed) and link ``out_lib``."""
    os.makedirs(build_dir, exist_ok=True)
    exe = nvcc()
    hdrs = _headers()
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s, *hdrs]):
            jobs.append([exe, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n%s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(out_lib, objs):
        tmp = out_lib + ".tmp%d" % os.getpid()
        run([exe, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"])
        os.replace(tmp, out_lib)
    return out_lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
