"""The no-allocation attention entry point (GPU).

paged_decode_attn_noalloc serves callers that cannot allocate device memory
(a plugin whose host runtime owns every allocation and passes it only its
inputs and outputs, or a serving loop that forbids cudaMalloc on its hot path
because it can synchronise the device).  It keeps its scratch in a fixed
array inside the library.

Here it is called through the package's ctypes binding, which hands the
tensors' device pointers straight to the C entry point, several times in a
row on different batches.  Each output is checked against the CPU oracle
and against paged_decode_attn on the same inputs, within the tolerance used
by every attention test.  A plain C program then drives the entry point
through the C ABI alone, across a cudaDeviceReset, and checks it against the
C oracle.  The file is named so pytest collects it last.
"""
import subprocess

import pytest

from gpu_util import PagedCase, assert_close, bf16_out, build_c_program, dev

pytestmark = pytest.mark.gpu


def _noalloc(case):
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    q = dev(case.q, dtype=torch.bfloat16)
    if case.fp8:
        kt, vt, ks, vs = dev(case.kc), dev(case.vc), dev(case.k_scale), dev(case.v_scale)
    else:
        kt, vt = dev(case.kc, dtype=torch.bfloat16), dev(case.vc, dtype=torch.bfloat16)
        ks = vs = None
    out = torch.full((case.B, case.Hq, case.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    fkv.paged_decode_attn_noalloc(q, kt, vt, dev(case.indptr), dev(case.indices), dev(case.seq), case.sm, out,
                                  k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("kv", ["fp8", "bf16"])
def test_noalloc_matches_regular_entry_point_twice(orc, kv):
    first = PagedCase(orc, 6, 64, 8, 64, [40000, 17, 3000, 1, 9000, 640], kv=kv, seed=501)
    second = PagedCase(orc, 4, 32, 8, 16, [4097, 33, 2, 1500], kv=kv, seed=502)
    third = PagedCase(orc, 3, 32, 2, 64, [5000, 40, 2100], kv=kv, seed=503)   # 16 query heads per KV head
    cases = (first, second, third)
    refs = [case.oracle(orc) for case in cases]
    for case, ref in zip(cases, refs):               # calls in a row share the scratch
        got = bf16_out(_noalloc(case))
        assert_close(got, ref, "noalloc vs oracle (%s, B=%d)" % (kv, case.B))
        want = bf16_out(case.gpu())                  # regular entry point, caller-provided workspace
        assert_close(got, want, "noalloc vs regular (%s, B=%d)" % (kv, case.B))
        assert_close(want, ref, "regular vs oracle (%s, B=%d)" % (kv, case.B))


def test_noalloc_c_abi_across_device_reset(tmp_path):
    """Plain C, no torch: two calls in a row, then cudaDeviceReset (a new
    context, in which the library looks its scratch address up again), then a
    third call; all checked against the C oracle."""
    exe = build_c_program("c_abi_noalloc.c", str(tmp_path / "c_abi_noalloc"))
    res = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "c abi noalloc ok" in res.stdout, res.stdout


def test_workspace_of_a_split_group():
    """A group of 16 query heads per KV head is served as two groups of 8: the
    workspace is that of twice the KV heads with 8 query heads each."""
    import fp8_paged_kv_decode_gb300 as fkv
    assert fkv.paged_decode_attn_workspace_size(3, 32, 2) == fkv.paged_decode_attn_workspace_size(3, 32, 4) > 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    B, Hq, Hkv = 4096, 64, 8                         # needs far more than the fixed scratch
    assert fkv.paged_decode_attn_workspace_size(B, Hq, Hkv) > fkv.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(B, Hq, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(1, Hkv, 16, 128, dtype=torch.uint8, device="cuda")
    s = torch.ones(Hkv, dtype=torch.float32, device="cuda")
    indptr = torch.zeros(B + 1, dtype=torch.int32, device="cuda")
    ind = torch.zeros(1, dtype=torch.int32, device="cuda")
    seq = torch.zeros(B, dtype=torch.int32, device="cuda")
    with pytest.raises(fkv.FkvError, match="status 4"):
        fkv.paged_decode_attn_noalloc(q, kc, kc, indptr, ind, seq, 0.1, q, k_scale=s, v_scale=s)
