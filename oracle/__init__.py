"""CPU oracle for FP8 paged-KV decode attention -- TEST INFRASTRUCTURE ONLY.

The oracle is the slow, plain reference the CUDA library is checked against.
Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import it; the library never does and has no CPU fallback.  It shares
no code with the CUDA path: the arithmetic lives in ``fkv_oracle.c`` (scalar
C, fp64), this module only builds it with gcc and marshals numpy arrays.

Parity status of each function (what pins it independently of itself is in
``tests/test_oracle_pins.py``):

* ``e4m3_decode`` / ``e4m3_encode`` -- pinned: all 256 codes against the
  E4M3 closed form, brute-force nearest-value search with ties to even,
  saturation, NaN/Inf/-0, and torch's float8_e4m3fn for in-range values.
* ``kv_append_fp8`` -- pinned: numpy's IEEE float32 division, slot placement
  against a hand-computed position, untouched bytes.
* ``kv_append_bf16`` -- pinned: every row placed by hand with numpy indexing
  (K and V pools, first / middle / last slot, padding and past-the-pool slots
  write nothing, every other element keeps its fill).
* ``kv_page_tag_check`` -- pinned: hand-derived cases in ``tests/golden``,
  brute force, tag bump and 32-bit wrap-around.
* ``kv_calibrate_scales`` -- pinned: numpy's max of |x| and IEEE float32
  division; all-zero heads; a single outlier sets its head's scale.
* ``kv_page_realloc`` -- pinned: reallocation then the (pinned) tag check
  aborts exactly the old holders; a fresh holder of the new tag passes;
  wrap-around; scrub zeroes exactly the listed pages.
* ``paged_decode_attn`` -- pinned: single-token context returns V, identical
  keys give the mean of V, numpy dense softmax on tiny inputs, G=1 per-head
  softmax, page-permutation invariance, FP8-vs-BF16 on exactly representable
  values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "fkv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_default = None

GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-Wall"]


def compile_source(src: str, out: str) -> str:
    """Compile an oracle source file to a shared library (gcc, no fast-math,
    no FMA contraction, so x86 and Arm hosts give the same bits)."""
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", *GCC_FLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, _LIB)
    return _LIB


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_div_rn_f32.restype = ctypes.c_float
        lib.oracle_div_rn_f32.argtypes = [ctypes.c_float, ctypes.c_float]
        lib.oracle_kv_append_fp8.restype = None
        lib.oracle_kv_append_fp8.argtypes = [P, P, P, i32, P, P, P, P, i32, i32, i32, i32]
        lib.oracle_kv_append_bf16.restype = None
        lib.oracle_kv_append_bf16.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32]
        lib.oracle_kv_page_tag_check.restype = None
        lib.oracle_kv_page_tag_check.argtypes = [P, i32, P, P, P, i32, i64, P]
        lib.oracle_dense_attn.restype = None
        lib.oracle_dense_attn.argtypes = [P, P, P, i32, i32, ctypes.c_double, P]
        lib.oracle_paged_decode_attn.restype = None
        lib.oracle_paged_decode_attn.argtypes = [
            P, i32, i32, P, P, i32, P, P, i32, i32, i32, i32,
            P, P, i64, P, P, ctypes.c_double, P, i32, P]
        lib.oracle_kv_calibrate_scales.restype = None
        lib.oracle_kv_calibrate_scales.argtypes = [P, P, i64, i32, i32, P, P]
        lib.oracle_kv_page_realloc.restype = None
        lib.oracle_kv_page_realloc.argtypes = [P, i32, P, i32, P, P, P, i32, i32, i32, i32]
        self.lib = lib
        self.path = path

    # ---------------- scalar formats ----------------
    def e4m3_decode(self, code: int) -> float:
        return self.lib.oracle_e4m3_decode(int(code) & 0xFF)

    def e4m3_encode(self, x: float) -> int:
        return int(self.lib.oracle_e4m3_encode(float(np.float32(x))))

    def e4m3_encode_array(self, x) -> np.ndarray:
        f = self.lib.oracle_e4m3_encode
        x = _c(x, np.float32).ravel()
        return np.fromiter((f(float(v)) for v in x), dtype=np.uint8, count=x.size)

    def e4m3_decode_table(self) -> np.ndarray:
        return np.array([self.lib.oracle_e4m3_decode(c) for c in range(256)], dtype=np.float64)

    def bf16_to_double(self, bits) -> np.ndarray:
        b = _c(bits, np.uint16)
        f = self.lib.oracle_bf16_to_double
        return np.array([f(int(v)) for v in b.ravel()], dtype=np.float64).reshape(b.shape)

    def div_rn_f32(self, x: float, s: float) -> float:
        return self.lib.oracle_div_rn_f32(float(x), float(s))

    # ---------------- the three operations ----------------
    def kv_append_fp8(self, k_new, v_new, slot_mapping, k_scale, v_scale, k_cache, v_cache):
        """In place: quantize bf16 ``k_new/v_new`` [N][Hkv][D] (uint16 bits) into
        the uint8 pools ``k_cache/v_cache`` [P][Hkv][S][D]."""
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
        P, Hkv, S, D = k_cache.shape
        kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
        sm = _c(slot_mapping, np.int64)
        ks, vs = _c(k_scale, np.float32), _c(v_scale, np.float32)
        self.lib.oracle_kv_append_fp8(_ptr(kn), _ptr(vn), _ptr(sm), int(sm.size), _ptr(ks), _ptr(vs),
                                      _ptr(k_cache), _ptr(v_cache), P, Hkv, S, D)

    def kv_append_bf16(self, k_new, v_new, slot_mapping, k_cache, v_cache):
        assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous
        P, Hkv, S, D = k_cache.shape
        kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
        sm = _c(slot_mapping, np.int64)
        self.lib.oracle_kv_append_bf16(_ptr(kn), _ptr(vn), _ptr(sm), int(sm.size),
                                       _ptr(k_cache), _ptr(v_cache), P, Hkv, S, D)

    def kv_page_tag_check(self, page_tags, page_indptr, page_indices, expected_tags,
                          num_pages=None) -> np.ndarray:
        tags = _c(page_tags, np.uint32)
        P = tags.size if num_pages is None else int(num_pages)
        assert 0 <= P <= tags.size
        indptr = _c(page_indptr, np.int32)
        indices = _c(page_indices, np.int32)
        exp = _c(expected_tags, np.uint32)
        B = indptr.size - 1
        out = np.zeros(B, dtype=np.uint8)
        self.lib.oracle_kv_page_tag_check(_ptr(tags), P, _ptr(indptr), _ptr(indices),
                                          _ptr(exp), B, int(indices.size), _ptr(out))
        return out

    def kv_calibrate_scales(self, k, v):
        """Per-KV-head scales fl32(amax / 448) (1 for an all-zero head) of bf16
        ``k``/``v`` [N][Hkv][D] (uint16 bits)."""
        kk, vv = _c(k, np.uint16), _c(v, np.uint16)
        N, Hkv, D = kk.shape
        ks = np.zeros(Hkv, np.float32)
        vs = np.zeros(Hkv, np.float32)
        self.lib.oracle_kv_calibrate_scales(_ptr(kk), _ptr(vv), N, Hkv, D, _ptr(ks), _ptr(vs))
        return ks, vs

    def kv_page_realloc(self, page_tags, pages, k_cache=None, v_cache=None):
        """In place: bump the live tag of every listed page (uint32, wraps) and,
        when caches are given, zero those pages.  Returns the new tags each
        new owner records (0 for ids outside the pool)."""
        assert page_tags.dtype == np.uint32 and page_tags.flags.c_contiguous
        pg = _c(pages, np.int32)
        new = np.zeros(pg.size, np.uint32)
        if k_cache is not None:
            P, Hkv, S, D = k_cache.shape
            eb = k_cache.dtype.itemsize
            assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        else:
            Hkv, S, D, eb = 1, 1, 1, 1
        self.lib.oracle_kv_page_realloc(_ptr(page_tags), int(page_tags.size), _ptr(pg), int(pg.size), _ptr(new),
                                        _ptr(k_cache), _ptr(v_cache), Hkv, S, D, eb)
        return new

    def dense_attn(self, q, k, v, sm_scale) -> np.ndarray:
        q, k, v = _c(q, np.float64), _c(k, np.float64), _c(v, np.float64)
        T, D = k.shape
        out = np.zeros(D, dtype=np.float64)
        self.lib.oracle_dense_attn(_ptr(q), _ptr(k), _ptr(v), T, D, float(sm_scale), _ptr(out))
        return out

    def paged_decode_attn(self, q, k_cache, v_cache, page_indptr, page_indices, seq_lens,
                          sm_scale, k_scale=None, v_scale=None, abort_mask=None, rows=None, nnz=None):
        """fp64 attention rows.  ``q`` is uint16 bf16 bits [B][Hq][D]; the caches
        are uint8 e4m3 codes (with ``k_scale/v_scale``) or uint16 bf16 bits,
        shaped [P][Hkv][S][D].  Returns [B][Hq][D], or [len(rows)][D] for a
        subset of flat row indices r*Hq + i."""
        q = _c(q, np.uint16)
        B, Hq, D = q.shape
        P, Hkv, S, D2 = k_cache.shape
        assert D2 == D and Hq % Hkv == 0
        fp8 = k_cache.dtype == np.uint8
        kc = np.ascontiguousarray(k_cache)
        vc = np.ascontiguousarray(v_cache)
        ks = _c(k_scale, np.float32) if fp8 else None
        vs = _c(v_scale, np.float32) if fp8 else None
        indptr = _c(page_indptr, np.int32)
        indices = _c(page_indices, np.int32)
        sl = _c(seq_lens, np.int32)
        am = None if abort_mask is None else _c(abort_mask, np.uint8)
        if rows is None:
            rr, n = None, B * Hq
            out = np.zeros((B, Hq, D), dtype=np.float64)
        else:
            rr = _c(rows, np.int32)
            n = rr.size
            out = np.zeros((n, D), dtype=np.float64)
        self.lib.oracle_paged_decode_attn(_ptr(q), B, Hq, _ptr(kc), _ptr(vc), int(fp8), _ptr(ks), _ptr(vs),
                                          P, Hkv, S, D, _ptr(indptr), _ptr(indices),
                                          int(indices.size if nnz is None else min(nnz, indices.size)),
                                          _ptr(sl), _ptr(am),
                                          float(sm_scale), _ptr(rr), int(n), _ptr(out))
        return out


def default() -> Oracle:
    """The oracle built from ``fkv_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def __getattr__(name):
    # module-level shortcuts: oracle.kv_page_tag_check(...) etc.
    if name.startswith("_"):
        raise AttributeError(name)
    return getattr(default(), name)
