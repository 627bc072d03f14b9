"""The kernels divide by a per-tensor scale with one multiply by the rounded
reciprocal and one FMA correction (Markstein's theorem) instead of a full
division per element.  This test compares that division with CUDA's correctly
rounded __fdiv_rn over every fp32 dividend: the quotients must agree bit for
bit wherever the quotient's magnitude is in [2^-40, 2^20), and the E4M3 codes
everywhere (NaN and infinite dividends included).  The packed two-wide
magnitude version that the Q/K kernel uses, with the sign put back on the
code byte, must give the scalar version's magnitudes and codes."""
import os
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "nvfp4_quant_gb300", "csrc")


def _divisors():
    rng = np.random.default_rng(0)
    fixed = [1.0, 0.05, 0.0123456, 0.37, 1.0 / 448.0, 448.0, 6.0, 3.0e-5, 65504.0,
             float(np.nextafter(np.float32(2.0), np.float32(0.0))),  # all-ones significand
             float(np.nextafter(np.float32(1.0), np.float32(2.0))), 1.5 * 2.0 ** -100,
             2.0 ** 100, 0.75, 1e-3]
    rand = list(np.exp(rng.uniform(np.log(1e-6), np.log(1e3), 25)))
    return ["%.9g" % float(np.float32(d)) for d in fixed + rand]


def test_shared_divisor_division_is_correctly_rounded(tmp_path):
    exe = str(tmp_path / "div_check")
    subprocess.run(["nvcc", "-std=c++17", "-O3", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-I" + CSRC, os.path.join(HERE, "cuda", "div_check.cu"), "-o", exe],
                   check=True)
    out = subprocess.run([exe, *_divisors()], check=True, capture_output=True, text=True,
                         timeout=600).stdout
    lines = [l.split() for l in out.splitlines() if l.startswith("divisor")]
    assert len(lines) == len(_divisors())
    for f in lines:
        assert f[3] == "0", "quotient differs from __fdiv_rn: " + " ".join(f)
        assert f[5] == "0", "E4M3 code differs: " + " ".join(f)
        assert f[9] == "0", "packed magnitude division differs from the scalar one: " + " ".join(f)
