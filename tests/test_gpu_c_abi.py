"""The C ABI on its own: a plain C program (no Python, no torch) runs one
decode step through libfkv.so and checks it against the C oracle."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.isdir(os.path.join(cand, "include")):
            return cand
    nvcc = shutil.which("nvcc")
    return os.path.dirname(os.path.dirname(nvcc)) if nvcc else None


def test_decode_step_through_c_abi(tmp_path):
    import fp8_paged_kv_decode_gb300 as fkv
    lib = fkv.library_path()
    assert os.path.exists(lib), "libfkv.so is not built"
    cuda = _cuda_home()
    assert cuda, "CUDA toolkit not found"
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "c_abi_decode_step")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    os.path.join(HERE, "c_abi_decode_step.c"), os.path.join(ROOT, "oracle", "fkv_oracle.c"),
                    "-o", exe, "-L", libdir, "-l:" + os.path.basename(lib),
                    "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm", "-Wl,-rpath," + libdir],
                   check=True)
    res = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "c abi decode step ok" in res.stdout
