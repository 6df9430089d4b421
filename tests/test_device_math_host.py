"""Host-side checks of the device math constants (no GPU needed).

The bf16 kernels evaluate log1p(e), e in [0, 1], as e * (1 + e * r(e)) with a
fitted degree-7 polynomial r (see csrc/fit_log1p.py).  These tests read the
coefficients out of device_math.cuh, evaluate the same Horner scheme in fp32,
and check the relative error against log1p, so that a mistyped constant
cannot pass unnoticed.
"""
import os
import re
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "selective_state_space_126_b300", "csrc")


def device_coefficients():
    src = open(os.path.join(CSRC, "device_math.cuh")).read()
    body = src[src.index("float log1p_unit(float e)"):src.index("log1p_unit2")]
    nums = [float(x) for x in re.findall(r"(-?\d\.\d+e[-+]\d+)f", body)]
    # Horner order in the source: highest degree first
    return np.array(nums[::-1], dtype=np.float32)


def eval_fp32(coef, e):
    x = e.astype(np.float32)
    acc = np.full_like(x, coef[-1])
    for c in coef[-2::-1]:
        acc = (acc * x + c).astype(np.float32)
    return ((acc * x + np.float32(1)) * x).astype(np.float32).astype(np.float64)


def test_log1p_polynomial_relative_error():
    coef = device_coefficients()
    assert len(coef) == 8
    e = np.concatenate([np.geomspace(1e-30, 1e-3, 20001), np.linspace(1e-3, 1, 200001)]).astype(np.float32)
    got = eval_fp32(coef, e)
    ref = np.log1p(e.astype(np.float64))
    rel = np.abs(got - ref) / ref
    assert rel.max() < 5e-7, rel.max()


def test_fit_script_reproduces_the_constants():
    out = subprocess.run([sys.executable, os.path.join(CSRC, "fit_log1p.py")], capture_output=True, text=True,
                         check=True).stdout
    fitted = np.array([float(x.rstrip("f")) for x in out.strip().splitlines()[-1].split(",")], dtype=np.float32)
    np.testing.assert_allclose(fitted, device_coefficients(), rtol=1e-6, atol=0)


def test_softplus_identity_through_the_polynomial():
    """max(s,0) + log1p(e^-|s|) with the polynomial equals log(1 + e^s) to fp32 relative accuracy,
    including Delta far below 1e-3 (s << 0), where an absolute-error form would lose all digits."""
    coef = device_coefficients()
    s = np.linspace(-40, 20, 120001)
    e = np.exp(-np.abs(s))
    got = np.maximum(s, 0) + eval_fp32(coef, e)
    ref = np.logaddexp(0, s)
    rel = np.abs(got - ref) / ref
    assert rel.max() < 1e-6, rel.max()
