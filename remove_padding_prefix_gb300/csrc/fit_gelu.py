"""Derives the polynomial of the device GELU (gelu_erf in common.cuh).

With t = min(|x| / sqrt(2), 3.9), erfc(t) = exp(P(t) - t^2) where P is a degree-7
least-squares Chebyshev fit of log(erfcx(t)) on [0, 3.9] (erfcx(t) = exp(t^2) erfc(t),
smooth and slowly varying there), converted to the power basis in t.  The device
evaluates e = erfc(t) / 2 = 2^(Q(t) - log2(e) t^2) with Q = log2(e) P - 1 (the base
change and the halving folded into the coefficients), then

    GELU(x) = x Phi(x) = x / 2 + |x| (1/2 - e),

which is x (1 - e) for x > 0 and x e for x < 0.  The script prints Q's coefficients
(lowest degree first) and the worst error of that fp32 evaluation against the fp64
definition x * Phi(x) on a dense grid of [-8, 8].
"""
import numpy as np
from scipy.special import erfc, erfcx

TMAX = 3.9
DEG = 7
LOG2E = 1.4426950408889634


def fit():
    """Q's coefficients in the power basis of t, fp32."""
    k = np.arange(4000)
    tn = np.cos(np.pi * (k + 0.5) / 4000)           # Chebyshev nodes on [-1, 1]
    t = (tn + 1) * TMAX / 2
    c = np.polynomial.chebyshev.chebfit(tn, np.log(erfcx(t)), DEG)
    P = np.polynomial.Polynomial(np.polynomial.chebyshev.cheb2poly(c))
    q = P(np.polynomial.Polynomial([-1, 2 / TMAX])).coef * LOG2E
    q[0] -= 1.0
    q[2] -= LOG2E
    return q.astype(np.float32)


def gelu_fp32(x, coef):
    """The device evaluation order, in fp32 (ex2 taken exact)."""
    x = x.astype(np.float32)
    ax = np.abs(x)
    t = np.minimum(ax * np.float32(0.70710678118654752), np.float32(TMAX)).astype(np.float32)
    q = np.full_like(t, coef[-1])
    for cc in coef[-2::-1]:
        q = (q.astype(np.float64) * t + cc).astype(np.float32)       # fused multiply-adds
    e = np.exp2(q.astype(np.float64)).astype(np.float32)
    half_minus_e = (np.float32(0.5) - e).astype(np.float32)
    return (x.astype(np.float64) * 0.5 + ax * half_minus_e).astype(np.float32)   # one fused multiply-add


if __name__ == "__main__":
    coef = fit()
    print(", ".join(f"{v:.9e}f" for v in coef))
    x = np.linspace(-8, 8, 400001).astype(np.float32)
    ref = 0.5 * x.astype(np.float64) * erfc(-x.astype(np.float64) / np.sqrt(2))
    print("max abs error", np.abs(gelu_fp32(x, coef) - ref).max())
