"""The kvi8r store build computes its fp16 scale s = RN(a / 127) and the code
multiplier RN(1 / (s sqrt(128))) without the library's correctly rounded
division and reciprocal: a Markstein correction step for the quotient, and
one fma refinement of the hardware's approximate reciprocal.  Both must be
correctly rounded.  exact_division_check.c checks that exhaustively on the
host: the quotient for every non-negative finite fp32 a, the reciprocal for
every positive finite fp16 scale and every starting value within two ulp of
the true reciprocal (the hardware approximation is within one).

The kvf8s build's V codes e4m3(v / s_v) take the exact quotient's rounding
from fp32 arithmetic plus a residual test near each e4m3 rounding boundary.
e4m3_quotient_check.c restates that procedure and checks it against exact
rational rounding for every bf16 absmax and every bf16 value up to it."""
import os
import platform
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_store_build_scale_arithmetic_is_correctly_rounded(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "exact_division_check")
    flags = ["-O2", "-ffp-contract=off"]
    if platform.machine() in ("x86_64", "AMD64"):
        flags.append("-mfma")  # a hardware fused multiply-add for fmaf
    subprocess.run([cc, *flags, "-o", exe, os.path.join(HERE, "exact_division_check.c"), "-lm"], check=True)
    p = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stdout + p.stderr
    assert "division by 127: 0 of 2139095040 mismatch" in p.stdout
    assert "reciprocal of fp16 scale * sqrt(128): 0 of 158715 mismatch" in p.stdout


def test_kvf8s_v_codes_are_the_exact_quotient_rounding(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "e4m3_quotient_check")
    flags = ["-O2", "-ffp-contract=off"]
    if platform.machine() in ("x86_64", "AMD64"):
        flags.append("-mfma")
    subprocess.run([cc, *flags, "-o", exe, os.path.join(HERE, "e4m3_quotient_check.c"), "-lm"], check=True)
    p = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stdout + p.stderr
    assert "pairs 532701119" in p.stdout
    assert "absmax >= 2^-100: 0 mismatch" in p.stdout
    assert "sign symmetry: 0 mismatch" in p.stdout
