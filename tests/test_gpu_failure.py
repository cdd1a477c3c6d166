"""Failure detection of the bounded waits, on the GPU, without a GPU fault.

Every mbarrier wait inside the library's tensor-core kernels gives up after a time
limit, records RPP_DERR_TIMEOUT in the caller's error word, drains what it has in
flight, frees its tensor memory and returns, so the context stays usable.  The test
makes a wait run out on purpose through a test-only hook: the next GEMM launch issues
no operand loads (its barriers are never signalled) and its pipeline waits give up
after a few milliseconds.  It then checks the error word, that later kernels given the
set word do no work, and that the next call with the word cleared computes correctly.
"""
import numpy as np
import pytest
import torch

import oracle
import remove_padding_prefix_gb300 as rpp
from gpu_util import dev, up, down, assert_close

pytestmark = pytest.mark.gpu


def _gemm_inputs(M, N, K, seed):
    from workloads import round_to_dtype
    rng = np.random.default_rng(seed)
    a = round_to_dtype(rng.standard_normal((M, K), dtype=np.float32), "bf16")
    w = round_to_dtype(0.05 * rng.standard_normal((K, N), dtype=np.float32), "bf16")
    b = round_to_dtype(0.1 * rng.standard_normal(N, dtype=np.float32), "bf16")
    return a, w, b


def test_gemm_wait_runs_out_and_reports_timeout():
    M, N, K = 300, 256, 192
    a, w, b = _gemm_inputs(M, N, K, 3)
    ad, wd = up(a, "bf16"), up(np.ascontiguousarray(w.T), "bf16")
    bd = torch.as_tensor(b, device=dev())
    lib = rpp.lib()
    err = rpp.new_error_word()
    out = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=dev())
    assert lib.rpp_test_stall_next_gemm(5000) == 0          # waits give up after 5 ms
    rpp.linear(ad, wd, bd, out=out, err=err)
    torch.cuda.synchronize()
    assert rpp.get_device_error(err) == rpp._abi.RPP_DERR_TIMEOUT
    assert bool((out == 7.0).all())                         # the stalled launch stored nothing
    # with the word still set, the next launch does no work at all
    rpp.linear(ad, wd, bd, out=out, err=err)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    # the hook was consumed by the one launch; with the word cleared the GEMM is correct
    err.zero_()
    rpp.linear(ad, wd, bd, out=out, err=err)
    torch.cuda.synchronize()
    assert rpp.get_device_error(err) == 0
    ref = oracle.linear(a, w, b)
    assert_close(down(out), ref, "bf16", "GEMM after a timed-out launch")
