"""Coefficients of the cubic used for software exp2 in the prefill softmax.

2^x = 2^n * 2^f with n = round(x) and f = x - n in [-1/2, 1/2] (Cody and
Waite's range reduction).  2^f is approximated by c0 + c1 f + c2 f^2 + c3 f^3,
fitted here by least squares on the relative error over 20001 points of
[-1/2, 1/2], with weight 1/2^f; the script prints the coefficients (as fp32)
and the maximum relative error of the fp32-rounded cubic.  Run:
    python fit_exp2_poly.py
"""
import numpy as np

f = np.linspace(-0.5, 0.5, 20001)
y = np.exp2(f)
A = np.stack([f ** k for k in range(4)], axis=1) / y[:, None]
c, *_ = np.linalg.lstsq(A, np.ones_like(f), rcond=None)
c32 = c.astype(np.float32).astype(np.float64)
p = ((c32[3] * f + c32[2]) * f + c32[1]) * f + c32[0]
rel = np.abs(p / y - 1).max()
for k, v in enumerate(c.astype(np.float32)):
    print(f"c{k} = {float(v)!r:>22}  (0x{np.float32(v).view(np.uint32):08x})")
print(f"max relative error on [-1/2, 1/2]: {rel:.3e}")
