"""Helpers shared by the GPU parity tests: uploads, comparisons and tolerances."""
import numpy as np
import torch

import remove_padding_prefix_gb300 as rpp

# stated tolerances: fp16/bf16 max-abs 2e-2, mean-abs 2e-3; int8 final outputs 5e-2.
# fp32 (not stated): derived from fp32 rounding of K <= 4096 accumulations of O(1)
# terms, ~1e-6 relative; 1e-4 / 1e-5 leaves two orders of margin.
TOL = {"fp16": (2e-2, 2e-3), "bf16": (2e-2, 2e-3), "fp32": (1e-4, 1e-5), "int8": (5e-2, 5e-3)}

TDT = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16, "int8": torch.float16}


def dev():
    return torch.device("cuda:0")


def up(a, dtype, device=None):
    """Upload a float32 array (already rounded to `dtype`) as a device tensor of that dtype."""
    t = torch.as_tensor(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(device or dev()).to(TDT[dtype]).contiguous()


def down(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(got, ref, dtype, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    d = np.abs(got - ref)
    mx, mean = TOL[dtype]
    assert d.max() <= mx and d.mean() <= mean, f"{what}: max-abs {d.max():.3e} mean-abs {d.mean():.3e} ({dtype})"
    return d.max(), d.mean()


def check_err(err):
    code = rpp.get_device_error(err)
    assert code == 0, f"device error word {code}"
