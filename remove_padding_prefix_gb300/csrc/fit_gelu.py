"""Derives the polynomial of the device GELU (gelu_erf in common.cuh).

erfc(t) = exp(P(t) - t^2) with P a degree-9 least-squares Chebyshev fit of
log(erfcx(t)) on [0, 3.9] (erfcx(t) = exp(t^2) erfc(t), smooth and slowly varying
there), converted to the power basis in t for Horner evaluation in fp32.  The script
prints the coefficients (lowest degree first) and the worst error of the resulting
fp32 GELU against the fp64 definition x * Phi(x) on a dense grid of [-8, 8].
"""
import numpy as np
from scipy.special import erfc, erfcx

TMAX = 3.9
DEG = 9


def fit():
    k = np.arange(4000)
    tn = np.cos(np.pi * (k + 0.5) / 4000)           # Chebyshev nodes on [-1, 1]
    t = (tn + 1) * TMAX / 2
    c = np.polynomial.chebyshev.chebfit(tn, np.log(erfcx(t)), DEG)
    P = np.polynomial.Polynomial(np.polynomial.chebyshev.cheb2poly(c))
    return P(np.polynomial.Polynomial([-1, 2 / TMAX])).coef.astype(np.float32)


def gelu_fp32(x, coef):
    t = np.minimum(np.abs(x) * np.float32(0.70710678118654752), np.float32(TMAX)).astype(np.float32)
    acc = np.full_like(t, coef[-1])
    for cc in coef[-2::-1]:
        acc = (acc * t + cc).astype(np.float32)
    e = np.exp2(((acc - t * t) * np.float32(1.4426950408889634)).astype(np.float32).astype(np.float64))
    h = (np.float32(0.5) * x * e.astype(np.float32)).astype(np.float32)
    return np.where(x > 0, x - h, h)


if __name__ == "__main__":
    coef = fit()
    print(", ".join(f"{v:.9e}f" for v in coef))
    x = np.linspace(-8, 8, 400001).astype(np.float32)
    ref = 0.5 * x.astype(np.float64) * erfc(-x.astype(np.float64) / np.sqrt(2))
    print("max abs error", np.abs(gelu_fp32(x, coef) - ref).max())
