"""Derives the polynomials of the device GELU (gelu_erf<DEG> in common.cuh).

GELU(x) = x Phi(x) = x erfc(-x / sqrt(2)) / 2.  With a = min(|x|, A) and
e = erfc(a / sqrt(2)) / 2, it equals x (1 - e) for x > 0 and x e for x < 0, i.e.

    GELU(x) = relu(x) - |x| e.

With t = a / sqrt(2), erfc(t) = exp(P(t) - t^2) where P is a least-squares Chebyshev
fit of log(erfcx(t)) on [0, A / sqrt(2)] (erfcx(t) = exp(t^2) erfc(t), smooth and
slowly varying there).  The device evaluates e = 2^Q(a): the base change, the -t^2
term, the halving and the 1 / sqrt(2) scale are all folded into Q's coefficients (power
basis in a).  Two fits: degree 7 (fp32 outputs, int8 codes) and degree 5 (fp16 / bf16
outputs, whose rounding is 2^-11 relative or coarser).  The script prints each set
(lowest degree first), its clamp A and the worst error of the fp32 evaluation against
the fp64 definition on a dense grid of [-10, 10].
"""
import numpy as np
from scipy.special import erfc, erfcx

LOG2E = 1.4426950408889634
FITS = {7: 4.2, 5: 3.9}   # degree -> clamp of t = a / sqrt(2)


def fit(deg, tmax):
    """Q's coefficients in the power basis of a = |x|, fp32."""
    k = np.arange(4000)
    tn = np.cos(np.pi * (k + 0.5) / 4000)           # Chebyshev nodes on [-1, 1]
    t = (tn + 1) * tmax / 2
    c = np.polynomial.chebyshev.chebfit(tn, np.log(erfcx(t)), deg)
    P = np.polynomial.Polynomial(np.polynomial.chebyshev.cheb2poly(c))
    q = P(np.polynomial.Polynomial([-1, 2 / tmax])).coef * LOG2E     # log2(erfcx(t)) in t
    q[0] -= 1.0                                                     # the halving
    q[2] -= LOG2E                                                   # the -t^2 term
    q = q * (1 / np.sqrt(2)) ** np.arange(len(q))                   # t = a / sqrt(2)
    return q.astype(np.float32)


def gelu_fp32(x, coef, amax):
    """The device evaluation order, in fp32 (ex2 taken exact)."""
    x = x.astype(np.float32)
    ax = np.abs(x)
    a = np.minimum(ax, np.float32(amax))
    q = np.full_like(a, coef[-1])
    for cc in coef[-2::-1]:
        q = (q.astype(np.float64) * a + cc).astype(np.float32)       # fused multiply-adds
    e = np.exp2(q.astype(np.float64)).astype(np.float32)
    relu = np.maximum(x, np.float32(0))
    return (relu.astype(np.float64) - ax.astype(np.float64) * e).astype(np.float32)   # one fused multiply-add


if __name__ == "__main__":
    x = np.linspace(-10, 10, 800001).astype(np.float32)
    ref = 0.5 * x.astype(np.float64) * erfc(-x.astype(np.float64) / np.sqrt(2))
    for deg, tmax in FITS.items():
        coef = fit(deg, tmax)
        amax = np.float32(tmax * np.sqrt(2))
        print(f"degree {deg}, A = {amax:.9e}f")
        print("  " + ", ".join(f"{v:.9e}f" for v in coef))
        print("  max abs error", np.abs(gelu_fp32(x, coef, amax) - ref).max())
