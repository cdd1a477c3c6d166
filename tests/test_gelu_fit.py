"""The device GELU's polynomials: the coefficients in common.cuh are exactly the ones
csrc/fit_gelu.py derives, and the fp32 evaluation in the device's order stays within the
error bounds the header states (checked on the CPU against the fp64 definition
x * Phi(x) = x erfc(-x / sqrt(2)) / 2)."""
import importlib.util
import pathlib
import re

import numpy as np
import pytest

scipy_special = pytest.importorskip("scipy.special")

CSRC = pathlib.Path(__file__).resolve().parents[1] / "remove_padding_prefix_gb300" / "csrc"


def _fit_module():
    spec = importlib.util.spec_from_file_location("fit_gelu", CSRC / "fit_gelu.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _header_fits():
    """{degree: (clamp, coefficients lowest degree first)} parsed from gelu_erf<DEG>."""
    src = (CSRC / "common.cuh").read_text()
    body = src[src.index("__device__ __forceinline__ float gelu_erf(float x)"):]
    body = body[:body.index("return fmaf(-ax, e, fmaxf(x, 0.f));")]
    i7 = body.index("if constexpr (DEG == 7) {")
    i5 = body.index("} else {", i7)
    iend = body.index("const float e =", i5)
    fits = {}
    for deg, blk in ((7, body[i7:i5]), (5, body[i5:iend])):
        clamp = float(re.search(r"fminf\(ax, ([-+0-9.e]+)f\)", blk).group(1))
        nums = [float(v) for v in re.findall(r"([-+]?[0-9]\.[0-9]+e[-+][0-9]+)f", blk)]
        coefs = nums[1:]                   # first number: the clamp; then the Horner chain, highest first
        fits[deg] = (clamp, np.array(coefs[::-1], np.float32))
    return fits


@pytest.mark.parametrize("deg,bound", [(7, 6.4e-7), (5, 3.8e-5)])
def test_header_coefficients_match_the_fit(deg, bound):
    fg = _fit_module()
    clamp, coef = _header_fits()[deg]
    tmax = fg.FITS[deg]
    assert len(coef) == deg + 1
    assert np.array_equal(coef, fg.fit(deg, tmax))
    assert np.float32(clamp) == np.float32(tmax * np.sqrt(2))
    x = np.linspace(-10, 10, 400001).astype(np.float32)
    ref = 0.5 * x.astype(np.float64) * scipy_special.erfc(-x.astype(np.float64) / np.sqrt(2))
    err = np.abs(fg.gelu_fp32(x, coef, np.float32(clamp)) - ref)
    assert err.max() <= bound


def test_fit_form_matches_definition_at_closed_forms():
    """relu(x) - |x| erfc(|x| / sqrt 2) / 2 is x Phi(x): Phi(1) and Phi(-1) from the tables."""
    fg = _fit_module()
    coef = fg.fit(7, fg.FITS[7])
    amax = np.float32(fg.FITS[7] * np.sqrt(2))
    got = fg.gelu_fp32(np.array([1.0, -1.0, 0.0, 12.0, -12.0], np.float32), coef, amax)
    assert got[0] == pytest.approx(0.8413447460685429, abs=1e-6)
    assert got[1] == pytest.approx(-0.15865525393145707, abs=1e-6)
    assert got[2] == 0.0
    assert got[3] == pytest.approx(12.0, abs=1e-6)
    assert abs(got[4]) < 1e-6
