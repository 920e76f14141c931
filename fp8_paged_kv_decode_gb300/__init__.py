"""FP8 paged-KV decode attention for GB300 (sm_103a).

Thin Python binding over the C ABI in ``include/fkv.h`` (``libfkv.so``, built
in-tree by ``_build.py``).  Every function here only checks tensor metadata and
passes raw device pointers, sizes and the current CUDA stream to the library;
all computation runs in the library's CUDA kernels.  There is no CPU path: if
the library is missing or no GPU is present the calls raise.

Entry points (same names as the C ABI):
  kv_append_fp8 / kv_append_bf16   write new tokens into the paged pools
  kv_calibrate_scales              per-KV-head FP8 scales of a prompt (bulk write)
  kv_page_tag_check                the separate per-page generation-tag check
  kv_append_fp8_tag_check          the step's FP8 append and the tag check in one launch
  kv_append_bf16_tag_check         the same for a BF16 cache
  kv_page_realloc                  bump tags (and optionally zero pages) of reallocated pages
  paged_decode_attn                decode attention over the paged cache
  paged_decode_attn_workspace_size bytes of scratch paged_decode_attn needs
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "FkvError", "KV_FP8_E4M3", "KV_BF16", "library_path", "load_library", "kv_append_fp8", "kv_append_bf16",
    "kv_calibrate_scales", "kv_page_tag_check", "kv_append_fp8_tag_check", "kv_append_bf16_tag_check", "kv_page_realloc",
    "paged_decode_attn",
    "paged_decode_attn_workspace_size",
    "alloc_workspace",
    "paged_decode_attn_noalloc",
    "device_error", "kernels_per_call", "selftest_wait", "EXPORTED_SYMBOLS",
]

KV_FP8_E4M3 = 0
KV_BF16 = 1
DEVERR_APPEND_SLOT = 0x1
DEVERR_ATTN_PAGE = 0x2
DEVERR_TIMEOUT = 0x4
DEVERR_REALLOC_PAGE = 0x8
HEAD_DIM = 128

EXPORTED_SYMBOLS = (
    "fkv_status_string", "kv_append_fp8", "kv_append_bf16", "kv_calibrate_scales", "kv_page_tag_check",
    "kv_append_fp8_tag_check", "kv_append_bf16_tag_check", "kv_page_realloc",
    "paged_decode_attn_workspace_size", "paged_decode_attn", "paged_decode_attn_noalloc", "fkv_device_error",
    "fkv_kernels_per_call", "fkv_selftest_wait",
)
ERR_SCRATCH_LIMIT = 4
NOALLOC_SCRATCH_BYTES = 16 << 20

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class FkvError(RuntimeError):
    pass


def library_path() -> str:
    """The in-tree libfkv.so (``FKV_LIBRARY_PATH`` points at another build,
    e.g. a variant compiled with different options)."""
    return os.environ.get("FKV_LIBRARY_PATH") or os.path.join(_HERE, "libfkv.so")


def load_library():
    """Load libfkv.so (raises if it has not been built)."""
    global _lib
    lib = _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise FkvError("libfkv.so is not built; run fp8_paged_kv_decode_gb300._build.build()")
        lib = ctypes.CDLL(path)
        P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        lib.fkv_status_string.restype = ctypes.c_char_p
        lib.fkv_status_string.argtypes = [ctypes.c_int]
        lib.kv_append_fp8.restype = ctypes.c_int
        lib.kv_append_fp8.argtypes = [P, P, P, i32, P, P, P, P, i32, i32, i32, i32, P]
        lib.kv_append_bf16.restype = ctypes.c_int
        lib.kv_append_bf16.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32, P]
        lib.kv_page_tag_check.restype = ctypes.c_int
        lib.kv_page_tag_check.argtypes = [P, i32, P, P, P, i32, i64, P, P]
        lib.kv_append_fp8_tag_check.restype = ctypes.c_int
        lib.kv_append_fp8_tag_check.argtypes = [P, P, P, i32, P, P, P, P, i32, i32, i32, i32, P, P, P, P, i32, i64,
                                                P, P]
        lib.kv_append_bf16_tag_check.restype = ctypes.c_int
        lib.kv_append_bf16_tag_check.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32, P, P, P, P, i32, i64, P, P]
        lib.kv_calibrate_scales.restype = ctypes.c_int
        lib.kv_calibrate_scales.argtypes = [P, P, i64, i32, i32, P, P, P]
        lib.kv_page_realloc.restype = ctypes.c_int
        lib.kv_page_realloc.argtypes = [P, i32, P, i32, P, P, P, i32, i32, i32, i32, P]
        lib.paged_decode_attn_workspace_size.restype = ctypes.c_size_t
        lib.paged_decode_attn_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        lib.paged_decode_attn.restype = ctypes.c_int
        lib.paged_decode_attn.argtypes = [P, i32, i32, P, P, i32, P, P, i32, i32, i32, i32, P, P, i64, P, P, f32,
                                          P, P, ctypes.c_size_t, P]
        lib.paged_decode_attn_noalloc.restype = ctypes.c_int
        lib.paged_decode_attn_noalloc.argtypes = [P, i32, i32, P, P, i32, P, P, i32, i32, i32, i32, P, P, i64, P, P,
                                                  f32, P, P]
        lib.fkv_device_error.restype = ctypes.c_int
        lib.fkv_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
        lib.fkv_kernels_per_call.restype = i32
        lib.fkv_kernels_per_call.argtypes = [ctypes.c_char_p]
        lib.fkv_selftest_wait.restype = ctypes.c_int
        lib.fkv_selftest_wait.argtypes = [ctypes.c_uint64, i32, P, P]
        _lib = lib
        return lib


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _ptr(t):
    # plain integers: the entry points' argtypes convert them to void *
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(cond, msg):
    if not cond:
        raise FkvError(msg)


def _dev(*ts):
    for t in ts:
        if t is not None:
            _need(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")


def _raise(status: int, name: str):
    if status != 0:
        msg = load_library().fkv_status_string(status).decode()
        raise FkvError("%s failed: %s (status %d)" % (name, msg, status))


def _is_byte_cache(t):
    import torch
    return t.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8))


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------
def kv_append_fp8(k_new, v_new, slot_mapping, k_scale, v_scale, k_cache, v_cache, stream=None):
    """Quantize bf16 ``k_new/v_new`` [N][Hkv][128] to e4m3 into ``k_cache/v_cache``
    [P][Hkv][S][128] (uint8) at ``slot_mapping`` [N] (int64, <0 = skip)."""
    import torch
    _dev(k_new, v_new, slot_mapping, k_scale, v_scale, k_cache, v_cache)
    _need(k_new.dtype == torch.bfloat16 and v_new.dtype == torch.bfloat16, "k_new/v_new must be bf16")
    _need(slot_mapping.dtype == torch.int64, "slot_mapping must be int64")
    _need(k_scale.dtype == torch.float32 and v_scale.dtype == torch.float32, "scales must be float32")
    _need(_is_byte_cache(k_cache) and _is_byte_cache(v_cache), "FP8 caches must be uint8/float8_e4m3fn")
    P, Hkv, S, D = k_cache.shape
    _need(tuple(v_cache.shape) == (P, Hkv, S, D), "k_cache/v_cache shapes differ")
    N = slot_mapping.numel()
    _need(tuple(k_new.shape) == (N, Hkv, D) and tuple(v_new.shape) == (N, Hkv, D), "k_new/v_new shape")
    _raise(load_library().kv_append_fp8(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), N, _ptr(k_scale),
                                        _ptr(v_scale), _ptr(k_cache), _ptr(v_cache), P, Hkv, S, D,
                                        _stream(stream)), "kv_append_fp8")


def kv_append_bf16(k_new, v_new, slot_mapping, k_cache, v_cache, stream=None):
    """BF16-cache counterpart of ``kv_append_fp8`` (values stored unchanged)."""
    import torch
    _dev(k_new, v_new, slot_mapping, k_cache, v_cache)
    _need(k_new.dtype == torch.bfloat16 and k_cache.dtype == torch.bfloat16, "bf16 tensors expected")
    P, Hkv, S, D = k_cache.shape
    N = slot_mapping.numel()
    _need(tuple(k_new.shape) == (N, Hkv, D) and tuple(v_new.shape) == (N, Hkv, D), "k_new/v_new shape")
    _raise(load_library().kv_append_bf16(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), N, _ptr(k_cache),
                                         _ptr(v_cache), P, Hkv, S, D, _stream(stream)), "kv_append_bf16")


def kv_page_tag_check(page_tags, page_indptr, page_indices, expected_tags, abort_mask, stream=None):
    """abort_mask[r] = 1 iff a page request r expects has a different live tag
    (or is outside the pool).  All tensors on the GPU; the mask stays there."""
    import torch
    _dev(page_tags, page_indptr, page_indices, expected_tags, abort_mask)
    _need(page_tags.dtype == torch.uint32 or page_tags.dtype == torch.int32, "page_tags must be 32-bit")
    _need(expected_tags.dtype == page_tags.dtype, "expected_tags dtype must match page_tags")
    _need(page_indptr.dtype == torch.int32 and page_indices.dtype == torch.int32, "CSR must be int32")
    _need(abort_mask.dtype == torch.uint8, "abort_mask must be uint8")
    B = page_indptr.numel() - 1
    _need(abort_mask.numel() == B and expected_tags.numel() == page_indices.numel(), "size mismatch")
    _raise(load_library().kv_page_tag_check(_ptr(page_tags), page_tags.numel(), _ptr(page_indptr),
                                            _ptr(page_indices), _ptr(expected_tags), B, page_indices.numel(),
                                            _ptr(abort_mask), _stream(stream)), "kv_page_tag_check")


def kv_append_fp8_tag_check(k_new, v_new, slot_mapping, k_scale, v_scale, k_cache, v_cache,
                            page_tags, page_indptr, page_indices, expected_tags, abort_mask, stream=None):
    """``kv_append_fp8`` then ``kv_page_tag_check`` (same arguments, same
    results) in one launch; ``page_tags`` has one entry per page of the pool."""
    import torch
    _dev(k_new, v_new, slot_mapping, k_scale, v_scale, k_cache, v_cache, page_tags, page_indptr, page_indices,
         expected_tags, abort_mask)
    _need(k_new.dtype == torch.bfloat16 and v_new.dtype == torch.bfloat16, "k_new/v_new must be bf16")
    _need(slot_mapping.dtype == torch.int64, "slot_mapping must be int64")
    _need(k_scale.dtype == torch.float32 and v_scale.dtype == torch.float32, "scales must be float32")
    _need(_is_byte_cache(k_cache) and _is_byte_cache(v_cache), "FP8 caches must be uint8/float8_e4m3fn")
    P, Hkv, S, D = k_cache.shape
    _need(tuple(v_cache.shape) == (P, Hkv, S, D), "k_cache/v_cache shapes differ")
    N = slot_mapping.numel()
    _need(tuple(k_new.shape) == (N, Hkv, D) and tuple(v_new.shape) == (N, Hkv, D), "k_new/v_new shape")
    _need(page_tags.dtype in (torch.uint32, torch.int32) and expected_tags.dtype == page_tags.dtype,
          "tags must be 32-bit, both of one dtype")
    _need(page_tags.numel() == P, "page_tags must have one entry per page of the pool")
    _need(page_indptr.dtype == torch.int32 and page_indices.dtype == torch.int32, "CSR must be int32")
    _need(abort_mask.dtype == torch.uint8, "abort_mask must be uint8")
    B = page_indptr.numel() - 1
    _need(abort_mask.numel() == B and expected_tags.numel() == page_indices.numel(), "size mismatch")
    _raise(load_library().kv_append_fp8_tag_check(
        _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), N, _ptr(k_scale), _ptr(v_scale), _ptr(k_cache),
        _ptr(v_cache), P, Hkv, S, D, _ptr(page_tags), _ptr(page_indptr), _ptr(page_indices), _ptr(expected_tags),
        B, page_indices.numel(), _ptr(abort_mask), _stream(stream)), "kv_append_fp8_tag_check")


def kv_append_bf16_tag_check(k_new, v_new, slot_mapping, k_cache, v_cache,
                             page_tags, page_indptr, page_indices, expected_tags, abort_mask, stream=None):
    """``kv_append_bf16`` then ``kv_page_tag_check`` (same arguments, same
    results) in one launch; ``page_tags`` has one entry per page of the pool."""
    import torch
    _dev(k_new, v_new, slot_mapping, k_cache, v_cache, page_tags, page_indptr, page_indices, expected_tags,
         abort_mask)
    _need(k_new.dtype == torch.bfloat16 and v_new.dtype == torch.bfloat16, "k_new/v_new must be bf16")
    _need(k_cache.dtype == torch.bfloat16 and v_cache.dtype == torch.bfloat16, "BF16 caches expected")
    _need(slot_mapping.dtype == torch.int64, "slot_mapping must be int64")
    P, Hkv, S, D = k_cache.shape
    _need(tuple(v_cache.shape) == (P, Hkv, S, D), "k_cache/v_cache shapes differ")
    N = slot_mapping.numel()
    _need(tuple(k_new.shape) == (N, Hkv, D) and tuple(v_new.shape) == (N, Hkv, D), "k_new/v_new shape")
    _need(page_tags.dtype in (torch.uint32, torch.int32) and expected_tags.dtype == page_tags.dtype,
          "tags must be 32-bit, both of one dtype")
    _need(page_tags.numel() == P, "page_tags must have one entry per page of the pool")
    _need(page_indptr.dtype == torch.int32 and page_indices.dtype == torch.int32, "CSR must be int32")
    _need(abort_mask.dtype == torch.uint8, "abort_mask must be uint8")
    B = page_indptr.numel() - 1
    _need(abort_mask.numel() == B and expected_tags.numel() == page_indices.numel(), "size mismatch")
    _raise(load_library().kv_append_bf16_tag_check(
        _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), N, _ptr(k_cache), _ptr(v_cache), P, Hkv, S, D,
        _ptr(page_tags), _ptr(page_indptr), _ptr(page_indices), _ptr(expected_tags), B, page_indices.numel(),
        _ptr(abort_mask), _stream(stream)), "kv_append_bf16_tag_check")


def kv_calibrate_scales(k, v, k_scale, v_scale, stream=None):
    """Per-KV-head scales fl32(amax / 448) of a prompt's bf16 K/V [N][Hkv][128]
    (1 for an all-zero head), written into ``k_scale``/``v_scale`` (fp32 [Hkv])."""
    import torch
    _dev(k, v, k_scale, v_scale)
    _need(k.dtype == torch.bfloat16 and v.dtype == torch.bfloat16, "k/v must be bf16")
    _need(k_scale.dtype == torch.float32 and v_scale.dtype == torch.float32, "scales must be float32")
    N, Hkv, D = k.shape
    _need(tuple(v.shape) == (N, Hkv, D) and k_scale.numel() == Hkv and v_scale.numel() == Hkv, "shape mismatch")
    _raise(load_library().kv_calibrate_scales(_ptr(k), _ptr(v), N, Hkv, D, _ptr(k_scale), _ptr(v_scale),
                                              _stream(stream)), "kv_calibrate_scales")


def kv_page_realloc(page_tags, pages, new_tags, k_cache=None, v_cache=None, stream=None):
    """Bump the live tag of each listed page (new owners record ``new_tags``)
    and, if the pools are given, zero those pages."""
    import torch
    _dev(page_tags, pages, new_tags, k_cache, v_cache)
    _need(page_tags.dtype in (torch.int32, torch.uint32) and new_tags.dtype == page_tags.dtype, "32-bit tags")
    _need(pages.dtype == torch.int32 and new_tags.numel() == pages.numel(), "pages int32, one new tag each")
    if k_cache is not None:
        _need(v_cache is not None and tuple(k_cache.shape) == tuple(v_cache.shape), "both pools, same shape")
        P, Hkv, S, D = k_cache.shape
        kv = KV_FP8_E4M3 if _is_byte_cache(k_cache) else KV_BF16
    else:
        Hkv = S = 0
        D, kv = HEAD_DIM, KV_FP8_E4M3
    _raise(load_library().kv_page_realloc(_ptr(page_tags), page_tags.numel(), _ptr(pages), pages.numel(),
                                          _ptr(new_tags), _ptr(k_cache), _ptr(v_cache), kv, Hkv, S, D,
                                          _stream(stream)), "kv_page_realloc")


def paged_decode_attn_workspace_size(batch, num_q_heads, num_kv_heads, head_dim=HEAD_DIM, kv_dtype=KV_FP8_E4M3):
    n = load_library().paged_decode_attn_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, kv_dtype)
    _need(n > 0 or batch == 0, "unsupported shape for paged_decode_attn")
    return int(n)


def alloc_workspace(batch, num_q_heads, num_kv_heads, kv_dtype=KV_FP8_E4M3, device="cuda"):
    import torch
    n = paged_decode_attn_workspace_size(batch, num_q_heads, num_kv_heads, HEAD_DIM, kv_dtype)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def paged_decode_attn(q, k_cache, v_cache, page_indptr, page_indices, seq_lens, sm_scale, out, workspace,
                      k_scale=None, v_scale=None, abort_mask=None, stream=None):
    """out[r][i] = softmax(sm_scale q k^T) v over request r's paged tokens.

    q, out: bf16 [B][Hq][128]; caches [P][Hkv][S][128] uint8 (FP8 e4m3, with
    k_scale/v_scale fp32 [Hkv]) or bf16; CSR page table int32; seq_lens int32
    [B]; abort_mask uint8 [B] or None (no tracker)."""
    import torch
    _dev(q, k_cache, v_cache, page_indptr, page_indices, seq_lens, out, workspace, k_scale, v_scale, abort_mask)
    fp8 = _is_byte_cache(k_cache)
    _need(fp8 or k_cache.dtype == torch.bfloat16, "cache must be uint8 (e4m3) or bf16")
    _need(q.dtype == torch.bfloat16 and out.dtype == torch.bfloat16, "q/out must be bf16")
    _need(seq_lens.dtype == torch.int32, "seq_lens must be int32")
    _need(abort_mask is None or abort_mask.dtype == torch.uint8, "abort_mask must be uint8")
    B, Hq, D = q.shape
    P, Hkv, S, D2 = k_cache.shape
    _need(tuple(out.shape) == (B, Hq, D) and D2 == D and page_indptr.numel() == B + 1, "shape mismatch")
    _raise(load_library().paged_decode_attn(
        _ptr(q), B, Hq, _ptr(k_cache), _ptr(v_cache), KV_FP8_E4M3 if fp8 else KV_BF16,
        _ptr(k_scale) if fp8 else None, _ptr(v_scale) if fp8 else None, P, Hkv, S, D,
        _ptr(page_indptr), _ptr(page_indices), page_indices.numel(), _ptr(seq_lens), _ptr(abort_mask),
        float(sm_scale),
        _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
        "paged_decode_attn")
    return out


def paged_decode_attn_noalloc(q, k_cache, v_cache, page_indptr, page_indices, seq_lens, sm_scale, out,
                              k_scale=None, v_scale=None, abort_mask=None, stream=None):
    """``paged_decode_attn`` without a workspace argument, for callers that
    cannot allocate device memory: its scratch is a fixed array of
    ``NOALLOC_SCRATCH_BYTES`` inside the library (shared by all calls on a
    device, so calls must not overlap on the GPU).  Shapes needing more
    scratch raise FkvError (status ERR_SCRATCH_LIMIT)."""
    import torch
    _dev(q, k_cache, v_cache, page_indptr, page_indices, seq_lens, out, k_scale, v_scale, abort_mask)
    fp8 = _is_byte_cache(k_cache)
    _need(fp8 or k_cache.dtype == torch.bfloat16, "cache must be uint8 (e4m3) or bf16")
    _need(q.dtype == torch.bfloat16 and out.dtype == torch.bfloat16, "q/out must be bf16")
    _need(seq_lens.dtype == torch.int32, "seq_lens must be int32")
    _need(abort_mask is None or abort_mask.dtype == torch.uint8, "abort_mask must be uint8")
    B, Hq, D = q.shape
    P, Hkv, S, D2 = k_cache.shape
    _need(tuple(out.shape) == (B, Hq, D) and D2 == D and page_indptr.numel() == B + 1, "shape mismatch")
    _raise(load_library().paged_decode_attn_noalloc(
        _ptr(q), B, Hq, _ptr(k_cache), _ptr(v_cache), KV_FP8_E4M3 if fp8 else KV_BF16,
        _ptr(k_scale) if fp8 else None, _ptr(v_scale) if fp8 else None, P, Hkv, S, D,
        _ptr(page_indptr), _ptr(page_indices), page_indices.numel(), _ptr(seq_lens), _ptr(abort_mask),
        float(sm_scale), _ptr(out), _stream(stream)), "paged_decode_attn_noalloc")
    return out


def device_error(clear: bool = True) -> int:
    """Sticky device error word of the current device (synchronises)."""
    v = ctypes.c_uint32(0)
    _raise(load_library().fkv_device_error(ctypes.byref(v), 1 if clear else 0), "fkv_device_error")
    return int(v.value)


def kernels_per_call(entry_point: str) -> int:
    return int(load_library().fkv_kernels_per_call(entry_point.encode()))


def selftest_wait(limit_ns: int, complete: bool = False, result=None, stream=None):
    """Run the failure path of the kernels' bounded waits on the GPU: one
    block waits, with the library's two wait helpers, on an mbarrier that
    nothing completes (``complete=False``) and gives up after ``limit_ns``,
    setting DEVERR_TIMEOUT; with ``complete=True`` the waits return at once.
    ``result``: None or a CUDA uint32 tensor of 2 (1 = the wait saw the
    barrier complete, 0 = it gave up, per warp)."""
    if result is not None:
        _dev(result)
        import torch
        _need(result.dtype in (torch.uint32, torch.int32) and result.numel() >= 2, "result: 2 x 32-bit")
    _raise(load_library().fkv_selftest_wait(int(limit_ns), 1 if complete else 0, _ptr(result), _stream(stream)),
           "fkv_selftest_wait")
