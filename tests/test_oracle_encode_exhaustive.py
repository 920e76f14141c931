"""The oracle's E4M3 encoder on every binary32 value whose code is neither a
signed zero nor saturated (|x| in [2^-16, 2^10), both signs: 436 M values), and
on a sample of the rest, against a nearest-value search over the 127 listed
magnitudes of the OCP FP8 E4M3 definition (ties to the even code, satfinite,
NaN keeps its sign).  The search shares nothing with the encoder but the
format; see ``e4m3_encode_exhaustive.c``."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_encode_matches_nearest_value_search_exhaustively(tmp_path):
    exe = str(tmp_path / "e4m3_encode_exhaustive")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-pthread",
                    os.path.join(HERE, "e4m3_encode_exhaustive.c"), os.path.join(ROOT, "oracle", "fkv_oracle.c"),
                    "-o", exe, "-lm"], check=True)
    res = subprocess.run([exe], capture_output=True, text=True, timeout=900)
    lines = {ln.split()[0]: ln.split()[1:] for ln in res.stdout.strip().splitlines()}
    assert lines["exhaustive"] == [str(26 * 2 ** 24), "bad=0"], res.stdout
    assert lines["sampled"][1] == "bad=0", res.stdout
    assert int(lines["sampled"][0]) > 10 ** 7
    assert res.returncode == 0, res.stdout


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("mutant", ["encode_ties_away", "encode_mantissa_truncates"])
def test_exhaustive_check_catches_encode_mutants(tmp_path, mutant):
    """The same check on a copy of the oracle with a plausible encoder mistake
    planted (the mistakes of test_oracle_mutants) must fail."""
    from test_oracle_mutants import MUTANTS
    old, new = MUTANTS[mutant]
    src = open(os.path.join(ROOT, "oracle", "fkv_oracle.c")).read()
    assert src.count(old) == 1
    mutated = tmp_path / "fkv_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    exe = str(tmp_path / "e4m3_encode_exhaustive_mutant")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-pthread",
                    os.path.join(HERE, "e4m3_encode_exhaustive.c"), str(mutated), "-o", exe, "-lm"], check=True)
    res = subprocess.run([exe], capture_output=True, text=True, timeout=900)
    assert res.returncode == 1, res.stdout
    assert "exhaustive %d bad=0" % (26 * 2 ** 24) not in res.stdout
