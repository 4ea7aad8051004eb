"""The NVFP4 quantizer's x / deq(scale) (Markstein's correction in quant_nvfp4.cu) equals IEEE
division: an exhaustive GPU check of the product's own function (tests/probes/div_exhaustive.cu
includes the kernel source) over every E4M3 divisor and every dividend with a quotient in
[2^-3, 16), both signs, plus 2^32 random cases; quotient bits and E2M1 codes must all agree."""
import os
import re
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_division_equals_ieee_exhaustively():
    from precision_attention_diffusion_gb300 import build
    exe = os.path.join(tempfile.mkdtemp(prefix="fa_lp_div_"), "div_exhaustive")
    src = os.path.join(HERE, "probes", "div_exhaustive.cu")
    subprocess.run([build.nvcc()] + build.ARCH + ["-O3", "-std=c++17", "--expt-relaxed-constexpr",
                    "-I", os.path.join(os.path.dirname(HERE), "include"), src, "-o", exe],
                   check=True, capture_output=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    m = re.search(r"cases (\d+) quotient_mismatches (\d+) code_mismatches (\d+) zero_sign (\d)",
                  r.stdout)
    assert m, r.stdout
    cases, bq, bc, zs = map(int, m.groups())
    assert cases > 1.9e10
    assert bq == 0 and bc == 0 and zs == 1
