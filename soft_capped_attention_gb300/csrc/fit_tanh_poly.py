"""Fits the odd polynomial the kernels use for tanh on |u| <= 0.5.

    python soft_capped_attention_gb300/csrc/fit_tanh_poly.py

tanh(u) = u + u^3 * (c0 + w (c1 + w (c2 + w c3))),  w = u^2.

The fit is an iteratively reweighted least-squares approximation of the
minimax polynomial in w over Chebyshev nodes of [0, 0.25], on the residual
(tanh(u) - u) / u^3 weighted by u^3 (absolute error of tanh).  It prints the
coefficients as float32 and the maximum absolute error of the float32 Horner
evaluation over a dense grid (about 2.5e-8), which is what the kernels'
constants in softmax_elem.cuh were taken from.
"""

import numpy as np

U0 = 0.5
DEG = 3


def fit():
    n = 4000
    w = np.sort((np.cos(np.pi * (np.arange(n) + 0.5) / n) + 1) / 2 * U0 * U0)
    u = np.sqrt(w)
    u[u == 0] = 1e-9
    target = (np.tanh(u) - u) / u ** 3
    wt = np.ones_like(w)
    A = np.vstack([w ** k for k in range(DEG + 1)]).T
    for _ in range(60):
        c, *_ = np.linalg.lstsq(A * (wt * u ** 3)[:, None], target * wt * u ** 3, rcond=None)
        err = u + u ** 3 * (A @ c) - np.tanh(u)
        wt = wt * (np.abs(err) / np.abs(err).max() + 1e-3) ** 0.5
        wt /= wt.max()
    return c.astype(np.float32)


def max_error_fp32(c):
    uu = np.linspace(-U0, U0, 400001).astype(np.float32)
    ww = uu * uu
    p = np.float32(c[DEG])
    for k in range(DEG - 1, -1, -1):
        p = (p * ww + c[k]).astype(np.float32)
    t = (uu + (uu * ww).astype(np.float32) * p).astype(np.float32)
    return float(np.abs(t.astype(np.float64) - np.tanh(uu.astype(np.float64))).max())


if __name__ == "__main__":
    c = fit()
    print("coefficients:", ", ".join(f"{float(x):.9g}f" for x in c))
    print("max |error| (fp32 evaluation):", max_error_fp32(c))
