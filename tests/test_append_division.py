"""The division on kv_append_fp8's fast path is IEEE round-to-nearest division.

kv_append_fp8 writes e4m3(fl32(x / scale)).  Its kernel computes the quotient
from the correctly rounded reciprocal of the scale and one fused remainder
correction (the correction step of Markstein's division) whenever the scale
lies in [2^-30, 2^30] and |x| <= 2^64, and with __fdiv_rn otherwise.  The
correction step's textbook precondition does not hold for every operand pair
here, so this test proves the claim by exhaustion on the host:
``recip_division_check.c`` runs the same sequence in IEEE single precision for
every bf16 significand against every fp32 significand (2^30 pairs), across the
admitted exponent range, and for the tiny inputs whose code is a signed zero.
The GPU tests then check the kernel's codes bit for bit against the oracle.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_recip_division_matches_ieee_division(tmp_path):
    exe = str(tmp_path / "recip_division_check")
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-pthread",
                    os.path.join(HERE, "recip_division_check.c"), "-o", exe, "-lm"], check=True)
    res = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    lines = dict(line.split(" ", 1) for line in res.stdout.strip().splitlines())
    assert lines["exhaustive_pairs=1073741824"] == "bad=0", res.stdout
    for key, val in lines.items():
        assert val == "bad=0", res.stdout
    assert res.returncode == 0, res.stdout
