"""CPU check of the polynomial tanh the kernels evaluate on the FMA pipe.

The coefficients are read from the kernel header and evaluated in float32
exactly as the kernels do (Horner in w = u^2); the result must stay within
5e-8 of tanh over the whole range |u| <= 0.5 where the kernels use it, well
below the tanh.approx instruction's error, and the fit script must reproduce
the committed constants."""

import os
import re
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "soft_capped_attention_gb300", "csrc", "softmax_elem.cuh")


def _consts():
    text = open(HDR).read()
    c = [float(re.search(rf"kTanhC{k}\s*=\s*([-0-9.e]+)f", text).group(1)) for k in range(4)]
    umax = float(re.search(r"kTanhPolyMaxU\s*=\s*([0-9.]+)f", text).group(1))
    return np.array(c, dtype=np.float32), umax


def test_polynomial_tanh_error_bound():
    c, umax = _consts()
    u = np.linspace(-umax, umax, 1_000_001).astype(np.float32)
    w = (u * u).astype(np.float32)
    p = c[3]
    for k in (2, 1, 0):
        p = (p * w + c[k]).astype(np.float32)
    t = (u + (u * w).astype(np.float32) * p).astype(np.float32)
    err = np.abs(t.astype(np.float64) - np.tanh(u.astype(np.float64)))
    assert err.max() < 5e-8, err.max()


def test_fit_script_reproduces_constants():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "soft_capped_attention_gb300", "csrc",
                                                       "fit_tanh_poly.py")],
                         capture_output=True, text=True, check=True).stdout
    got = [float(x.rstrip("f")) for x in out.splitlines()[0].split(":")[1].split(",")]
    c, _ = _consts()
    np.testing.assert_allclose(got, c, rtol=1e-6)
