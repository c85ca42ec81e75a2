"""Host proof of the act_quant kernel's exact-division shortcut: the kernel replaces each
x / s by a reciprocal multiply plus one Markstein correction step (two FMAs). quotient_check.c
enumerates every bf16 block maximum and every bf16 element below it and checks that the result
equals the IEEE binary32 quotient wherever it can influence the e4m3 code."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_quotient_identity_exhaustive(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "quotient_check")
    src = os.path.join(HERE, "quotient_check.c")
    base = [cc, "-O2", "-std=c11", "-ffp-contract=off", "-o", exe, src, "-lm"]
    if subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True).returncode != 0:
        subprocess.run(base, check=True)
    res = subprocess.run([exe], capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stdout[-2000:]
    assert "violations 0" in res.stdout
