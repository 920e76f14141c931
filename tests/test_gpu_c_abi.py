"""The C ABI on its own: a plain C program (no Python, no torch) runs one
decode step through libfkv.so and checks it against the C oracle."""
import subprocess

import pytest

from gpu_util import build_c_program

pytestmark = pytest.mark.gpu


def test_decode_step_through_c_abi(tmp_path):
    exe = build_c_program("c_abi_decode_step.c", str(tmp_path / "c_abi_decode_step"))
    res = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "c abi decode step ok" in res.stdout
