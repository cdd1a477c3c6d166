"""GPU parity of the INT8 path: weight and activation quantisation bit-exact, int32
accumulators of the int8 GEMM bit-exact (including adversarial all-extreme inputs at
the largest K), the calibration pass, and the int8 encoder layer within the int8
tolerance (5e-2 on final outputs)."""
import numpy as np
import pytest
import torch

import oracle
import remove_padding_prefix_gb300 as rpp
from workloads import CONFIGS, make_bert_workload, make_calibration_batch, round_to_dtype
from gpu_util import dev, up, down, assert_close, check_err

pytestmark = pytest.mark.gpu
INT8 = CONFIGS[3]


@pytest.mark.parametrize("K,N", [(1024, 3072), (4096, 1024), (96, 48)])
def test_weight_quantisation_bit_exact(K, N):
    rng = np.random.default_rng(K + N)
    W = round_to_dtype(0.02 * rng.standard_normal((K, N), dtype=np.float32), "fp16")
    W[:, 3] = 0.0
    W[7, 5] = 2.0 * np.abs(W[:, 5]).max()        # one dominant entry
    q, s = rpp.quantize_weight(up(W, "fp16"))
    q_ref, s_ref = oracle.quantize_weight_per_channel(W)
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref.T)


def test_activation_quantisation_bit_exact():
    rng = np.random.default_rng(0)
    x = round_to_dtype(3 * rng.standard_normal((777, 1024), dtype=np.float32), "fp16")
    scale = np.float32(np.abs(x).max() / 127 * 0.7)   # some values clamp
    x[0, :8] = np.array([0.5, 1.5, 2.5, -0.5, -1.5, 126.5, -126.5, 0.0], np.float32) * scale
    x = round_to_dtype(x, "fp16")
    q = rpp.quantize_activation(up(x, "fp16"), torch.tensor([scale], device=dev()))
    assert np.array_equal(q.cpu().numpy(), oracle.quantize_activation(x, scale))


@pytest.mark.parametrize("M,N,K", [(300, 256, 1024), (129, 1024, 4096), (1, 16, 16), (2000, 3072, 1024),
                                   (517, 64, 3072)])
def test_int8_gemm_int32_accumulators_bit_exact(M, N, K):
    rng = np.random.default_rng(M)
    a = rng.integers(-127, 128, size=(M, K), dtype=np.int64).astype(np.int8)
    w = rng.integers(-127, 128, size=(N, K), dtype=np.int64).astype(np.int8)
    acc = rpp.gemm_i8_i32(torch.as_tensor(a, device=dev()), torch.as_tensor(w, device=dev()))
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), oracle.int8_gemm(a, w.T))


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("M,N,K", [(300, 256, 1024), (385, 128, 4096), (8300, 1024, 1024)])
def test_int8_gemm_cluster_modes_bit_exact(mode, M, N, K):
    """The integer GEMM under every CTA-pair mode setting (it runs unpaired in all of
    them), one and four exact K chunks, odd numbers of row tiles: int32 accumulators
    bit-exact."""
    rng = np.random.default_rng(M + K + mode)
    a = rng.integers(-127, 128, size=(M, K), dtype=np.int64).astype(np.int8)
    w = rng.integers(-127, 128, size=(N, K), dtype=np.int64).astype(np.int8)
    assert rpp.lib().rpp_set_gemm_cluster_mode(mode) == 0
    try:
        acc = rpp.gemm_i8_i32(torch.as_tensor(a, device=dev()), torch.as_tensor(w, device=dev()))
    finally:
        rpp.lib().rpp_set_gemm_cluster_mode(0)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), oracle.int8_gemm(a, w.T))


def test_int8_gemm_adversarial_extremes():
    """All-+-127 operands: every chunk partial reaches +-(1024 * 127^2) = +-16 516 096, just
    under 2^24, and the full sum reaches +-66 064 384 for K = 4096."""
    M, N, K = 256, 128, 4096
    rng = np.random.default_rng(5)
    a = np.where(rng.random((M, K)) < 0.5, 127, -127).astype(np.int8)
    a[:64] = 127
    a[64:128] = -127
    w = np.where(rng.random((N, K)) < 0.5, 127, -127).astype(np.int8)
    w[:32] = 127
    w[32:48] = -127
    acc = rpp.gemm_i8_i32(torch.as_tensor(a, device=dev()), torch.as_tensor(w, device=dev()))
    ref = oracle.int8_gemm(a, w.T)
    assert ref.max() == 127 * 127 * K and ref.min() == -127 * 127 * K
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), ref)


def _int8_case(wl, scales):
    cfg = wl["cfg"]
    layer = wl["layers"][0]
    ecfg = rpp.encoder_cfg(cfg.H, cfg.nh, cfg.F, cfg.eps, "fp16", int8=True)
    prepared = rpp.EncoderLayer(ecfg, layer)
    lengths = torch.as_tensor(wl["lengths"], device=dev())
    err = rpp.new_error_word()
    cu, po = rpp.build_offsets(lengths, cfg.L, err=err)
    x = rpp.remove_padding(up(wl["x_padded"].reshape(-1, cfg.H), "fp16"), po, cu, cfg.B, cfg.L, err=err)
    y = rpp.encoder_layer_forward(prepared, x, cu, cfg.B, cfg.L, act_scales=torch.as_tensor(scales, device=dev()),
                                  err=err)
    check_err(err)
    return down(y), cu.cpu().numpy(), down(x)


def test_int8_layer_small():
    cfg = INT8
    wl = make_bert_workload(cfg, B=4, L=160, lengths=np.array([160, 1, 64, 129], np.int32), affine=True)
    s = oracle.calibrate_int8(wl["x_padded"], wl["lengths"], wl["layers"][0], cfg.nh, cfg.eps)
    got, cu, x = _int8_case(wl, s)
    T = int(cu[-1])
    ref = oracle.bert_layer_int8(x[:T], cu, oracle.prepare_int8_layer(wl["layers"][0]), s, cfg.nh, cfg.eps)
    assert_close(got[:T], ref, "int8", "int8 layer small")


def test_int8_layer_full_config_all_sequences():
    """The BERT-large-shaped int8 layer (B=64, L=256) at full size, every sequence of the
    batch against the oracle's int8 layer (one packed call), scales from the oracle's
    calibration on the seeded calibration batch."""
    cfg = INT8
    wl = make_bert_workload(cfg)
    cal = make_calibration_batch(cfg)
    s = oracle.calibrate_int8(cal["x_padded"], cal["lengths"], wl["layers"][0], cfg.nh, cfg.eps)
    got, cu, x = _int8_case(wl, s)
    q = oracle.prepare_int8_layer(wl["layers"][0])
    T = int(cu[-1])
    ref = oracle.bert_layer_int8(x[:T], cu, q, s, cfg.nh, cfg.eps)
    assert_close(got[:T], ref, "int8", "int8 layer, all 64 sequences")


def test_calibration_matches_oracle():
    wl = make_bert_workload(INT8, B=8, L=128)
    cfg = wl["cfg"]
    layer = wl["layers"][0]
    prepared = rpp.EncoderLayer(rpp.encoder_cfg(cfg.H, cfg.nh, cfg.F, cfg.eps, "fp16"), layer)
    lengths = torch.as_tensor(wl["lengths"], device=dev())
    err = rpp.new_error_word()
    cu, po = rpp.build_offsets(lengths, cfg.L, err=err)
    x = rpp.remove_padding(up(wl["x_padded"].reshape(-1, cfg.H), "fp16"), po, cu, cfg.B, cfg.L, err=err)
    amax = rpp.encoder_layer_calibrate(prepared, x, cu, cfg.B, cfg.L, err=err)
    check_err(err)
    ref = oracle.calibrate_int8(wl["x_padded"], wl["lengths"], layer, cfg.nh, cfg.eps) * 127.0
    got = amax.cpu().numpy()
    assert got[0] == np.float32(np.abs(wl["x_padded"][np.arange(cfg.L)[None, :] < wl["lengths"][:, None]]).max())
    assert np.allclose(got, ref, rtol=1e-2), (got, ref)
