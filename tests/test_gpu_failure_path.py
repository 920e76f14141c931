"""The failure path of the kernels' bounded waits, run on the GPU without a
fault (fkv_selftest_wait): a wait on an mbarrier that nothing completes gives
up after its time limit, sets DEVERR_TIMEOUT and the kernel ends normally;
the context stays usable for the calls that follow."""
import time

import pytest

from gpu_util import PagedCase, assert_close, bf16_out

pytestmark = pytest.mark.gpu


def test_completed_barrier_returns_at_once():
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    fkv.device_error(clear=True)
    res = torch.full((2,), 7, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    fkv.selftest_wait(2_000_000_000, complete=True, result=res)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert res.cpu().tolist() == [1, 1]          # both helpers saw the phase complete
    assert fkv.device_error() == 0
    assert dt < 1.0                              # nowhere near the 2 s limit


@pytest.mark.parametrize("limit_ms", [20, 200])
def test_wait_that_nothing_completes_gives_up_and_reports(orc, limit_ms):
    import torch
    import fp8_paged_kv_decode_gb300 as fkv
    fkv.device_error(clear=True)
    res = torch.full((2,), 7, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    fkv.selftest_wait(limit_ms * 1_000_000, result=res)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert res.cpu().tolist() == [0, 0]          # both helpers gave up
    assert dt >= limit_ms * 1e-3                 # ... after waiting their limit
    assert dt < limit_ms * 1e-3 + 2.0
    assert fkv.device_error() & fkv.DEVERR_TIMEOUT
    assert fkv.device_error() == 0               # the read above cleared it
    # the context is still usable: the next calls match the oracle
    case = PagedCase(orc, 3, 16, 2, 64, [700, 64, 2000], seed=41)
    assert_close(bf16_out(case.gpu()), case.oracle(orc), "attention after a timed-out wait")
    assert fkv.device_error() == 0


def test_limit_above_ten_seconds_is_refused():
    import fp8_paged_kv_decode_gb300 as fkv
    with pytest.raises(fkv.FkvError):
        fkv.selftest_wait(10_000_000_001)
