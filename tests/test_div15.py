"""The quantize kernel divides by 15 with a multiply and one FMA correction
instead of an IEEE division; this checks, on the CPU, that the sequence equals
the correctly rounded quotient for every finite non-negative fp32 input."""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_division_by_15_is_correctly_rounded_for_every_float():
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "div15")
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-o", exe,
                        os.path.join(HERE, "div15_exhaustive.c"), "-lm"], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=600).stdout
    assert out.strip() == "0", f"{out.strip()} inputs differ from IEEE division"
