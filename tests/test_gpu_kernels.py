"""GPU parity of the layer's building blocks against the oracle: the tcgen05 GEMM with
each fused epilogue, the fp32 GEMM, LayerNorm and the varlen attention kernel.

Sizes span several 128-row tiles plus a ragged tail, every tile width the heuristic
picks, and the device-side row count used inside the layer."""
import numpy as np
import pytest
import torch

import oracle
import remove_padding_prefix_gb300 as rpp
from workloads import round_to_dtype
from gpu_util import dev, up, down, assert_close, check_err, TDT

pytestmark = pytest.mark.gpu


def _gemm_case(dtype, M, N, K, epi, seed=0, rows=None):
    rng = np.random.default_rng(seed)
    a = round_to_dtype(rng.standard_normal((M, K), dtype=np.float32), dtype)
    W = round_to_dtype(0.02 * rng.standard_normal((K, N), dtype=np.float32), dtype)   # [in, out]
    b = round_to_dtype(0.02 * rng.standard_normal(N, dtype=np.float32), dtype)
    r = round_to_dtype(rng.standard_normal((M, N), dtype=np.float32), dtype)
    err = rpp.new_error_word()
    rows_t = torch.tensor([rows], dtype=torch.int32, device=dev()) if rows is not None else None
    out = torch.full((M, N), float("nan"), dtype=TDT[dtype], device=dev())
    res_t = up(r, dtype) if epi == rpp.RPP_EPI_BIAS_RESIDUAL else None
    rpp.linear(up(a, dtype), up(W.T, dtype), torch.as_tensor(b, device=dev()), epilogue=epi, residual=res_t,
               out=out, rows=rows_t, err=err)
    check_err(err)
    ref = oracle.linear(a, W, b)
    if epi == rpp.RPP_EPI_BIAS_GELU:
        ref = oracle.gelu(ref)
    if epi == rpp.RPP_EPI_BIAS_RESIDUAL:
        ref = ref + r
    m = M if rows is None else rows
    if m:
        assert_close(down(out[:m]), ref[:m], dtype, f"linear {dtype} {M}x{N}x{K} epi{epi}")
    if rows is not None:   # rows past the device count are never written
        assert torch.isnan(out[m:].float()).all()


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("epi", [0, 1, 2])
def test_tc_gemm_epilogues(dtype, epi):
    _gemm_case(dtype, 300, 256, 192, epi, seed=epi)


@pytest.mark.parametrize("M,N,K", [(1, 16, 8), (129, 2304, 768), (2304, 768, 3072), (517, 3072, 1024),
                                   (1000, 288, 96), (384, 96, 384), (255, 144, 64)])
def test_tc_gemm_shapes(M, N, K):
    _gemm_case("fp16", M, N, K, rpp.RPP_EPI_BIAS, seed=M)


@pytest.fixture
def cluster_mode():
    """Set the GEMM's CTA-pair mode for one test, back to automatic afterwards."""
    def set_mode(m):
        assert rpp.lib().rpp_set_gemm_cluster_mode(m) == 0
    yield set_mode
    set_mode(0)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("M,N,K,epi,rows", [
    (1, 16, 8, 0, None),          # one row tile: with pairs forced, the partner tile is empty
    (300, 256, 192, 1, None),     # three row tiles: the last pair is half empty
    (517, 3072, 1024, 0, None),
    (2304, 768, 3072, 2, None),
    (1000, 768, 256, 2, 613),     # device row count, odd number of live tiles
    (384, 144, 64, 0, 129),
])
def test_tc_gemm_cluster_modes(cluster_mode, mode, M, N, K, epi, rows):
    """Unpaired and paired GEMMs (a two-CTA cluster, each CTA loading its own A rows and half
    of the W tile for cta_group::2 MMAs), each against
    the oracle, on shapes with an odd number of row tiles."""
    cluster_mode(mode)
    _gemm_case("bf16" if epi == 2 else "fp16", M, N, K, epi, seed=M + mode, rows=rows)


def test_tc_gemm_device_row_count():
    _gemm_case("bf16", 1000, 768, 256, rpp.RPP_EPI_BIAS_RESIDUAL, rows=613)
    _gemm_case("fp16", 512, 128, 64, rpp.RPP_EPI_BIAS, rows=0)


@pytest.mark.parametrize("epi", [0, 1, 2])
def test_f32_gemm(epi):
    _gemm_case("fp32", 150, 256, 1024, epi, seed=10 + epi)


@pytest.mark.parametrize("dtype,H", [("fp32", 256), ("fp16", 768), ("bf16", 1024), ("fp16", 96), ("bf16", 96),
                                     ("fp16", 256), ("bf16", 512), ("fp16", 1536)])
def test_layernorm(dtype, H):
    rng = np.random.default_rng(H)
    M = 333
    x = round_to_dtype(rng.standard_normal((M, H), dtype=np.float32) * 2 + 0.5, dtype)
    g = round_to_dtype(1 + 0.1 * rng.standard_normal(H, dtype=np.float32), dtype)
    b = round_to_dtype(0.1 * rng.standard_normal(H, dtype=np.float32), dtype)
    eps = 1e-5 if H == 96 else 1e-12
    err = rpp.new_error_word()
    y = rpp.layernorm(up(x, dtype), torch.as_tensor(g, device=dev()), torch.as_tensor(b, device=dev()), eps, err=err)
    check_err(err)
    assert_close(down(y), oracle.layernorm(x, g, b, eps), dtype, f"layernorm {dtype} H={H}")


@pytest.mark.parametrize("dtype,H", [("fp16", 1024), ("bf16", 768)])
def test_layernorm_device_rows_in_place(dtype, H):
    """Rows past the device row count stay untouched; y may alias x (each row is read
    before it is written)."""
    rng = np.random.default_rng(H + 7)
    M_max, M = 700, 611
    x = round_to_dtype(rng.standard_normal((M_max, H), dtype=np.float32) * 3 - 1, dtype)
    g = (1 + 0.1 * rng.standard_normal(H)).astype(np.float32)
    b = (0.1 * rng.standard_normal(H)).astype(np.float32)
    err = rpp.new_error_word()
    xd = up(x, dtype)
    rows = torch.tensor([M], dtype=torch.int32, device=dev())
    rpp.layernorm(xd, torch.as_tensor(g, device=dev()), torch.as_tensor(b, device=dev()), 1e-12, out=xd, rows=rows,
                  err=err)
    check_err(err)
    got = down(xd)
    assert_close(got[:M], oracle.layernorm(x[:M], g, b, 1e-12), dtype, f"in-place layernorm {dtype} H={H}")
    assert np.array_equal(got[M:], x[M:])


def _attention_case(dtype, lengths, nh, seed=0, max_len=None, poison=False, qk_scale=1.0):
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, np.int32)
    L = int(max_len or max(1, lengths.max()))
    T = int(lengths.sum())
    T_max = max(T, 1) + 5   # capacity larger than T: rows past T must be ignored
    d = 64
    qkv = rng.standard_normal((T_max, 3 * nh * d), dtype=np.float32)
    qkv[:, :2 * nh * d] *= np.float32(qk_scale)
    qkv = round_to_dtype(qkv, dtype)
    lt = torch.as_tensor(lengths, device=dev())
    err = rpp.new_error_word()
    cu, _ = rpp.build_offsets(lt, L, err=err)
    out = torch.full((T_max, nh * d), float("nan"), dtype=TDT[dtype], device=dev())
    qkv_d = up(qkv, dtype)
    if poison == "nan":   # capacity rows past T hold NaN: a kernel must never let them reach a valid output
        qkv_d[T:] = float("nan")
    elif poison == "large":
        # capacity rows past T hold large finite values of both signs: the query rows past
        # the last sequence's end (computed, never stored) then see row maxima that jump
        # between key tiles in some rows of a warp and not in others
        big = 300.0 * np.sign(rng.standard_normal((T_max - T, 3 * nh * d))) * rng.uniform(0.5, 1.0, (T_max - T, 1))
        qkv_d[T:] = torch.as_tensor(big, dtype=torch.float32, device=dev()).to(qkv_d.dtype)
    rpp.attention_varlen(qkv_d, cu, len(lengths), L, nh, out=out, err=err)
    check_err(err)
    cu_ref, _, _ = oracle.build_offsets(lengths, L)
    H = nh * d
    ref = oracle.attention_varlen(qkv[:T, :H], qkv[:T, H:2 * H], qkv[:T, 2 * H:], cu_ref, nh)
    if T:
        assert_close(down(out[:T]), ref, dtype, f"attention {dtype} lens={lengths.tolist()[:6]}")
    assert torch.isnan(out[T:].float()).all()


@pytest.mark.parametrize("dtype", ["fp16", "bf16", "fp32"])
def test_attention_ragged(dtype):
    _attention_case(dtype, [1, 63, 64, 65, 128, 129, 200, 7], nh=4, seed=1)


@pytest.mark.parametrize("dtype", ["fp16", "bf16", "fp32"])
def test_attention_ignores_non_finite_capacity_rows(dtype):
    # the last sequence ends inside a key tile, so its last tile spans rows past T
    _attention_case(dtype, [130, 57, 201], nh=2, seed=5, poison="nan")
    _attention_case(dtype, [3], nh=1, seed=6, poison="nan")


@pytest.mark.parametrize("dtype", ["fp16", "bf16", "fp32"])
def test_attention_rows_past_sequence_end_with_large_values(dtype):
    """Rows past T hold large values: the out-of-sequence query rows of the last query
    tile rescale their running maximum while the valid rows of the same warp do not.
    The valid outputs must not change and the kernel must run to completion."""
    _attention_case(dtype, [130, 57, 201], nh=2, seed=8, poison="large")
    _attention_case(dtype, [64, 300], nh=3, seed=9, poison="large")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_attention_wide_score_range(dtype):
    """Q and K scaled by 3 (scores spread over tens of log2 units): row maxima move
    between 32-key chunks of one tile and between tiles, so the lazy rescaling of O, the
    running sum and the P chunks already written runs often; outputs still match."""
    _attention_case(dtype, [300, 77, 129, 1, 256], nh=3, seed=31, qk_scale=3.0)


def test_attention_is_deterministic():
    """The same inputs give bit-identical outputs on every call (BERT-large length mix,
    16 heads, three calls; each CTA's work and arithmetic order are fixed by cu_seqlens)."""
    rng = np.random.default_rng(41)
    lens = np.concatenate([rng.integers(32, 129, 32), rng.integers(256, 385, 32)])
    T = int(lens.sum())
    nh = 16
    qkv = up(round_to_dtype(rng.standard_normal((T, 3 * nh * 64), dtype=np.float32), "bf16"), "bf16")
    err = rpp.new_error_word()
    cu, _ = rpp.build_offsets(torch.as_tensor(lens.astype(np.int32), device=dev()), 384, err=err)
    outs = [rpp.attention_varlen(qkv, cu, len(lens), 384, nh, err=err) for _ in range(3)]
    check_err(err)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_attention_after_nan_in_tensor_memory():
    """A GEMM over NaN inputs runs on every SM just before the attention, so the tensor
    memory the attention allocates holds NaN bit patterns.  Whatever the attention does
    not overwrite (the P rows of warps with no query row, the S columns past a partial
    tile) must never reach a valid output: five calls, each bit-identical to the first
    and within tolerance of the oracle."""
    rng = np.random.default_rng(43)
    lens = np.concatenate([rng.integers(32, 129, 32), rng.integers(256, 385, 32)]).astype(np.int32)
    rng.shuffle(lens)
    T = int(lens.sum())
    nh = 16
    H = nh * 64
    qkv_h = round_to_dtype(rng.standard_normal((T, 3 * H), dtype=np.float32), "bf16")
    qkv = up(qkv_h, "bf16")
    err = rpp.new_error_word()
    cu, _ = rpp.build_offsets(torch.as_tensor(lens, device=dev()), 384, err=err)
    a_nan = torch.full((2 * 152 * 128, 64), float("nan"), dtype=torch.bfloat16, device=dev())
    w = torch.zeros(512, 64, dtype=torch.bfloat16, device=dev())
    bias = torch.zeros(512, dtype=torch.float32, device=dev())
    outs = []
    for _ in range(5):
        rpp.linear(a_nan, w, bias)
        outs.append(rpp.attention_varlen(qkv, cu, len(lens), 384, nh, err=err))
    check_err(err)
    cu_h = cu.cpu().numpy()
    ref = oracle.attention_varlen(qkv_h[:, :H], qkv_h[:, H:2 * H], qkv_h[:, 2 * H:], cu_h, nh)
    assert_close(down(outs[0]), ref, "bf16", "attention after NaN in tensor memory")
    assert all(torch.equal(outs[0], o) for o in outs[1:])


def test_attention_bert_large_lengths():
    rng = np.random.default_rng(7)
    lens = np.concatenate([rng.integers(32, 129, 8), rng.integers(256, 385, 8)])
    _attention_case("bf16", lens, nh=16, seed=2, max_len=384)


def test_attention_many_sequences_and_long_tile_counts():
    """Batches the persistent longest-first kernel takes (up to 2048 sequences, up to 64
    key tiles) and beyond them (2050 sequences: the one-CTA-per-query-tile kernel), each
    against the oracle; plus one sequence spanning many key tiles (lazy rescaling over
    nine tiles)."""
    rng = np.random.default_rng(21)
    _attention_case("fp16", rng.integers(0, 4, 2048), nh=1, seed=22, max_len=3)
    _attention_case("bf16", rng.integers(0, 4, 2050), nh=1, seed=23, max_len=3)
    _attention_case("bf16", [1100, 5, 300], nh=2, seed=24, max_len=1100)


def test_attention_at_the_persistent_kernels_key_limit():
    """One 8192-token sequence, the most the persistent kernel takes (64 query tiles over
    64 key tiles, lazy rescaling along whole rows), and an 8200-token one, which goes to the
    one-CTA-per-query-tile kernel; both against the oracle."""
    _attention_case("bf16", [8192], nh=1, seed=31, max_len=8192)
    _attention_case("fp16", [8200, 3], nh=1, seed=32, max_len=8200)


def test_attention_empty_and_zero_length_sequences():
    _attention_case("fp16", [0, 5, 0, 0, 70], nh=2, seed=3)
    _attention_case("fp16", [0, 0], nh=2, seed=4, max_len=8)


def test_attention_rejects_length_above_max_len():
    lengths = np.array([10, 40], np.int32)
    qkv = torch.zeros(50, 3 * 64, dtype=torch.float16, device=dev())
    err = rpp.new_error_word()
    cu, _ = rpp.build_offsets(torch.as_tensor(lengths, device=dev()), 64, err=err)
    rpp.attention_varlen(qkv, cu, 2, 32, 1, err=err)   # max_len 32 < 40
    assert rpp.get_device_error(err) == rpp.RPP_DERR_LENGTH


def test_device_gelu_against_exact_definition():
    """The GEMM epilogue's GELU (exp of a fitted log-erfcx polynomial) against the fp64
    definition x * Phi(x): an fp32 GEMM with identity weights makes the accumulator
    exactly x, so the output is the device GELU of x itself."""
    x = np.concatenate([np.linspace(-8, 8, 64 * 1000), [0.0, -0.0, 1e-20, -1e-20, 3.9 * 2 ** 0.5, -30.0, 30.0,
                                                         1e4, -1e4] + [0.0] * 55]).astype(np.float32)
    a = x.reshape(-1, 64)
    eye = np.eye(64, dtype=np.float32)
    out = rpp.linear(up(a, "fp32"), up(eye, "fp32"), torch.zeros(64, device=dev()), epilogue=rpp.RPP_EPI_BIAS_GELU)
    got = down(out).reshape(-1)
    ref = oracle.gelu(x.astype(np.float64))
    err = np.abs(got - ref)
    assert np.all(err <= 5e-7 * (1.0 + np.abs(x))), (err.max(), x[np.argmax(err)])


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_device_gelu_16bit_outputs(dtype):
    """16-bit outputs take the degree-5 fit (at most 3.8e-5 from x * Phi(x)): with identity
    weights the accumulator is exactly x, and each output is within half a step of its
    dtype plus that fit error of the fp64 definition."""
    rng = np.random.default_rng(11)
    x = round_to_dtype(np.concatenate([np.linspace(-8, 8, 64 * 500), rng.standard_normal(64 * 500) * 2]
                                      ).astype(np.float32), dtype)
    a = x.reshape(-1, 64)
    eye = np.eye(64, dtype=np.float32)
    out = rpp.linear(up(a, dtype), up(eye, dtype), torch.zeros(64, device=dev()), epilogue=rpp.RPP_EPI_BIAS_GELU)
    got = down(out).reshape(-1).astype(np.float64)
    ref = oracle.gelu(x.astype(np.float64))
    mant = 10 if dtype == "fp16" else 7
    half_step = np.ldexp(1.0, np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -14))).astype(int) - mant - 1)
    err = np.abs(got - ref)
    assert np.all(err <= half_step + 4e-5), (err.max(), x[np.argmax(err - half_step)])
