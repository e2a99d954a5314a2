"""Derive the polynomials used by the kernels' softplus.

softplus(x) = max(x, 0) + log1p(w),  w = 2^(-|x| log2 e) in (0, 1].
log1p(w) is evaluated as w * P(w) with P a polynomial fitted to log1p(w)/w on
[0, 1]: weighted least squares on Chebyshev nodes, refined by Lawson
iterations toward the minimax relative error. Prints, for degree 4, 6 and 7,
the coefficients (lowest order first) and the max relative error of the fp32
Horner evaluation (about 5.7e-5, 1.4e-6 and 3.5e-7). Degree 4 serves bf16
inputs, whose own rounding (2^-9) is far coarser. Run: python fit_log1p_poly.py
"""
import numpy as np


def fit(DEG):
    k = np.arange(4000)
    x = 0.5 + 0.5 * np.cos(np.pi * (k + 0.5) / 4000)
    f = np.log1p(x) / x
    V = np.vander(x, DEG + 1, increasing=True) / f[:, None]
    w = np.ones_like(x)
    for _ in range(200):
        c, *_ = np.linalg.lstsq(V * np.sqrt(w)[:, None], np.sqrt(w), rcond=None)
        err = np.abs(V @ c - 1)
        w = w * (err + 1e-30)
        w /= w.sum()
    c32 = c.astype(np.float32)
    t = np.linspace(0, 1, 200001).astype(np.float32)[1:]
    p = np.full_like(t, c32[-1])
    for cc in c32[-2::-1]:
        p = (p.astype(np.float64) * t + cc).astype(np.float32)
    lp = (t.astype(np.float64) * p).astype(np.float32).astype(np.float64)
    ref = np.log1p(t.astype(np.float64))
    print("coefficients:", ", ".join("%.9ef" % v for v in c32))
    print("max relative error (fp32 Horner): %.3g" % np.max(np.abs(lp - ref) / ref))


for deg in (4, 6, 7):
    print("degree", deg)
    fit(deg)
