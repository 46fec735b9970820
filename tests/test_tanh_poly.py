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


def folded_x(X, inv, mul, add, c):
    """x = X Q(X^2) + add with the argument scale inv and output scale mul folded
    into the coefficients, evaluated in float32 in the kernels' order."""
    inv, mul, add = np.float32(inv), np.float32(mul), np.float32(add)
    w = np.float32(inv * inv)
    a0 = np.float32(mul * inv)
    k = [a0]
    wp = np.float32(1.0)
    for j in range(4):
        wp = np.float32(wp * w)
        k.append(np.float32(np.float32(a0 * wp) * c[j]))
    z = (X * X).astype(np.float32)
    q = np.float32(k[4])
    for j in (3, 2, 1, 0):
        q = (q * z + k[j]).astype(np.float32)
    return (X * q + add).astype(np.float32)


def test_folded_polynomial_matches_scaled_tanh():
    """mul * tanh(in X) + add through the folded coefficients stays within
    2e-7 * mul of the exact value over the polynomial's range, for argument
    scales from 1e-4 (smallest before the K4 guard) to 0.5."""
    c, umax = _consts()
    for inv in (1e-4, 1.7677669529663688e-3, 0.01, 0.1, 0.5):
        for mul in (0.5, 72.13475204444817):
            X = np.linspace(-umax / inv, umax / inv, 400_001).astype(np.float32)
            x = folded_x(X, inv, mul, -3.0, c)
            ref = mul * np.tanh(np.float64(np.float32(inv)) * X.astype(np.float64)) - 3.0
            err = np.abs(x.astype(np.float64) - ref).max()
            assert err < 2e-7 * mul + 5e-7, (inv, mul, err)
