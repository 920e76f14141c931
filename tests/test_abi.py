"""The C ABI library builds, loads and exports what include/fkv.h declares (no GPU)."""
import os
import re
import subprocess

import pytest

import fp8_paged_kv_decode_gb300 as fkv
from fp8_paged_kv_decode_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    with open(os.path.join(ROOT, "include", "fkv.h")) as f:
        src = f.read()
    return sorted(set(re.findall(r"^FKV_API\s+[\w\s\*]*?\b(\w+)\s*\(", src, re.M)))


@pytest.fixture(scope="module")
def lib_path():
    return _build.build()


def test_header_declares_the_entry_points():
    decl = declared_symbols()
    assert set(decl) == set(fkv.EXPORTED_SYMBOLS)
    for name in ("kv_append_fp8", "kv_page_tag_check", "paged_decode_attn"):
        assert name in decl


def test_library_exports_every_declared_symbol(lib_path):
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [s for s in declared_symbols() if s not in exported]
    assert not missing, missing


def test_library_loads_in_tree(lib_path):
    lib = fkv.load_library()
    assert os.path.realpath(lib._name) == os.path.realpath(os.path.join(ROOT, "fp8_paged_kv_decode_gb300", "libfkv.so"))
    for s in declared_symbols():
        assert hasattr(lib, s)
    assert lib.fkv_status_string(0) == b"ok"
    assert fkv.kernels_per_call("paged_decode_attn") == 2
    assert fkv.kernels_per_call("kv_page_tag_check") == 1
    assert fkv.kernels_per_call("kv_append_fp8_tag_check") == 1
    assert fkv.kernels_per_call("kv_append_bf16_tag_check") == 1


def test_host_validation_without_gpu(lib_path):
    """Argument checks return before touching the device."""
    lib = fkv.load_library()
    # head_dim != 128 is unsupported; negative sizes invalid
    assert lib.kv_append_fp8(None, None, None, 0, None, None, None, None, 4, 2, 16, 64, None) == 2
    assert lib.kv_append_fp8(None, None, None, -1, None, None, None, None, 4, 2, 16, 128, None) == 1
    assert lib.kv_page_tag_check(None, 4, None, None, None, -1, 0, None, None) == 1
    assert lib.kv_page_tag_check(None, 4, None, None, None, 0, 0, None, None) == 0
    # the append and the check in one launch take both calls' argument checks
    assert lib.kv_append_fp8_tag_check(None, None, None, 0, None, None, None, None, 4, 2, 16, 64,
                                       None, None, None, None, 0, 0, None, None) == 2
    assert lib.kv_append_fp8_tag_check(None, None, None, 0, None, None, None, None, 4, 2, 16, 128,
                                       None, None, None, None, -1, 0, None, None) == 1
    assert lib.kv_append_fp8_tag_check(None, None, None, 0, None, None, None, None, 4, 2, 16, 128,
                                       None, None, None, None, 3, 0, None, None) == 1
    assert lib.kv_append_fp8_tag_check(None, None, None, 0, None, None, None, None, 4, 2, 16, 128,
                                       None, None, None, None, 0, 0, None, None) == 0
    assert lib.kv_append_bf16_tag_check(None, None, None, 0, None, None, 4, 2, 16, 64,
                                        None, None, None, None, 0, 0, None, None) == 2
    assert lib.kv_append_bf16_tag_check(None, None, None, 0, None, None, 4, 2, 16, 128,
                                        None, None, None, None, 3, 0, None, None) == 1
    assert lib.kv_append_bf16_tag_check(None, None, None, 0, None, None, 4, 2, 16, 128,
                                        None, None, None, None, 0, 0, None, None) == 0
    assert lib.paged_decode_attn(None, 2, 8, None, None, 0, None, None, 4, 2, 16, 64, None, None, 0, None, None,
                                 0.1, None, None, 0, None) == 2
    assert lib.paged_decode_attn(None, 2, 8, None, None, 0, None, None, 4, 2, 24, 128, None, None, 0, None, None,
                                 0.1, None, None, 0, None) == 2
    assert lib.paged_decode_attn(None, 2, 8, None, None, 0, None, None, 4, 3, 16, 128, None, None, 0, None, None,
                                 0.1, None, None, 0, None) == 1
    assert lib.paged_decode_attn(None, 2, 18, None, None, 0, None, None, 4, 2, 16, 128, None, None, 0, None, None,
                                 0.1, None, None, 0, None) == 2     # group 9: no split into groups of <= 8
    assert lib.paged_decode_attn(None, 2, 32, None, None, 0, None, None, 4, 2, 16, 128, None, None, 0, None, None,
                                 0.1, None, None, 0, None) == 1     # group 16 (two groups of 8): null pointers
    assert lib.paged_decode_attn(None, 2, 8, None, None, 0, None, None, 4, 2, 16, 128, None, None, 0, None, None,
                                 -1.0, None, None, 0, None) == 1    # sm_scale must be positive
    assert lib.fkv_selftest_wait(10_000_000_001, 0, None, None) == 1     # more than 10 s of waiting
