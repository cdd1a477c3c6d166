"""The allocation-free int8 GEMM entry point (rpp_gemm_i8_i32_noalloc).

Some callers cannot allocate device memory -- a plugin whose host framework owns all
of it, a latency-critical path that must not call cudaMalloc, a foreign-function
caller without a device allocator -- so the library offers a variant of its int8 GEMM
that keeps its scratch in a fixed array inside the library.  This test calls that
entry point through the C ABI twice in a row and checks each result against the
regular entry point, which uses a caller-provided workspace; both are exact integer
products, so the comparison is bit for bit.  It also checks that a problem too large
for the fixed scratch is refused.  The file is named to be collected last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import remove_padding_prefix_gb300 as rpp

pytestmark = pytest.mark.gpu


def _call_noalloc(a, w, acc, err):
    M, K = a.shape
    N = w.shape[0]
    return rpp.lib().rpp_gemm_i8_i32_noalloc(a.data_ptr(), w.data_ptr(), acc.data_ptr(), M, N, K, err.data_ptr(),
                                             torch.cuda.current_stream().cuda_stream)


def test_noalloc_int8_gemm_matches_workspace_entry_point_twice():
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    err = rpp.new_error_word(dev)
    cases = [(300, 256, 1024, 11), (129, 64, 3072, 12)]   # second call: other sizes, chunked K
    for M, N, K, seed in cases:
        rng = np.random.default_rng(seed)
        a = torch.as_tensor(rng.integers(-127, 128, size=(M, K), dtype=np.int64).astype(np.int8), device=dev)
        w = torch.as_tensor(rng.integers(-127, 128, size=(N, K), dtype=np.int64).astype(np.int8), device=dev)
        ref = rpp.gemm_i8_i32(a, w, err=err)
        acc = torch.full((M, N), -1, dtype=torch.int32, device=dev)
        assert _call_noalloc(a, w, acc, err) == 0
        torch.cuda.synchronize()
        assert rpp.get_device_error(err) == 0
        assert torch.equal(acc, ref)


def test_noalloc_int8_gemm_rejects_problems_larger_than_its_scratch():
    dev = torch.device("cuda:0")
    M, N, K = 1024, 1024, 4096          # 16 MiB of re-encoded operands > 8 MiB scratch
    a = torch.zeros(M, K, dtype=torch.int8, device=dev)
    w = torch.zeros(N, K, dtype=torch.int8, device=dev)
    acc = torch.full((M, N), 7, dtype=torch.int32, device=dev)
    err = rpp.new_error_word(dev)
    assert _call_noalloc(a, w, acc, err) == rpp._abi.RPP_EWORKSPACE
    torch.cuda.synchronize()
    assert bool((acc == 7).all())     # nothing was launched
