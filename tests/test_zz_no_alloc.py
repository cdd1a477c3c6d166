"""The allocation-free int8 GEMM entry point (rpp_gemm_i8_i32_noalloc).

Some callers cannot allocate device memory -- a plugin whose host framework owns all
of it, a latency-critical path that must not call cudaMalloc, a foreign-function
caller without a device allocator -- so the library offers a variant of its int8 GEMM
that keeps its scratch in a fixed array inside the library.  This test calls that
entry point through the C ABI twice in a row and checks each result against the
regular entry point, which uses a caller-provided workspace, and once against the
CPU oracle's exact integer product; all are exact integer products, so the
comparison is bit for bit.  It also checks that a problem too large
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
    """Two calls back to back on one stream with a single synchronisation after both
    (the second call reuses the scratch array the first one left behind, in stream
    order); each result equals the workspace entry point's, and the first also equals
    the oracle's exact integer product."""
    import oracle
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    err = rpp.new_error_word(dev)
    cases = [(300, 256, 1024, 11), (129, 64, 3072, 12)]   # second call: other sizes, chunked K
    ops = []
    for M, N, K, seed in cases:
        rng = np.random.default_rng(seed)
        a_h = rng.integers(-127, 128, size=(M, K), dtype=np.int64).astype(np.int8)
        w_h = rng.integers(-127, 128, size=(N, K), dtype=np.int64).astype(np.int8)
        a, w = torch.as_tensor(a_h, device=dev), torch.as_tensor(w_h, device=dev)
        ref = rpp.gemm_i8_i32(a, w, err=err)
        acc = torch.full((M, N), -1, dtype=torch.int32, device=dev)
        ops.append((a_h, w_h, a, w, ref, acc))
    torch.cuda.synchronize()
    for _, _, a, w, _, acc in ops:          # no synchronisation between the two calls
        assert _call_noalloc(a, w, acc, err) == 0
    torch.cuda.synchronize()
    assert rpp.get_device_error(err) == 0
    for i, (a_h, w_h, _, _, ref, acc) in enumerate(ops):
        assert torch.equal(acc, ref)
        if i == 0:
            exact = oracle.int8_gemm(a_h, w_h.T)
            assert np.array_equal(acc.cpu().numpy().astype(np.int64), exact)


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
