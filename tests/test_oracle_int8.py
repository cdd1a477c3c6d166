"""Pins for the oracle's INT8 flow.

Closed forms and invariants: codes stay in [-127, 127] and each column's largest
magnitude maps to 127; round-half-to-even on exact ties; the dequantised weight is
within half a step of the float weight; the integer product equals an exact float64
product of small integers; on grid-aligned inputs the quantise -> int8 GEMM ->
dequantise chain is lossless and equals the float linear layer; calibration scales
are the max-abs over valid tokens only; the whole int8 layer stays within the
quantisation-noise bound of the float layer.
"""
import numpy as np
import pytest

import oracle
from workloads import CONFIGS, make_bert_workload, make_calibration_batch

INT8 = CONFIGS[3]


def test_weight_quantisation_properties():
    rng = np.random.default_rng(0)
    W = (0.02 * rng.standard_normal((64, 48))).astype(np.float16).astype(np.float32)
    W[:, 5] = 0.0
    Wq, s = oracle.quantize_weight_per_channel(W)
    assert Wq.dtype == np.int8 and s.dtype == np.float32
    assert np.abs(Wq.astype(int)).max() <= 127
    nz = [n for n in range(48) if n != 5]
    assert np.all(np.abs(Wq[:, nz].astype(int)).max(axis=0) == 127)
    assert np.all(Wq[:, 5] == 0) and s[5] == 1.0
    err = np.abs(Wq.astype(np.float64) * s.astype(np.float64) - W)
    assert np.all(err <= 0.5 * s.astype(np.float64) * (1 + 1e-6) + 1e-12)


def test_activation_quantisation_ties_and_clamp():
    s = np.float32(0.5)                 # 1/s = 2 exactly
    x = np.array([0.25, 0.75, 1.25, -0.25, -0.75, 100.0, -100.0, 63.25], np.float32)
    # x * 2 = 0.5, 1.5, 2.5, -0.5, -1.5, 200, -200, 126.5 -> half-even: 0, 2, 2, -0, -2, clamp, clamp, 126
    assert oracle.quantize_activation(x, s).tolist() == [0, 2, 2, 0, -2, 127, -127, 126]


def test_int8_gemm_exact():
    rng = np.random.default_rng(1)
    a = rng.integers(-127, 128, size=(33, 1024)).astype(np.int8)
    b = rng.integers(-127, 128, size=(1024, 17)).astype(np.int8)
    acc = oracle.int8_gemm(a, b)
    ref = a.astype(np.int64) @ b.astype(np.int64)     # integer arithmetic route
    assert acc.dtype == np.int64 and np.array_equal(acc, ref)
    worst = oracle.int8_gemm(np.full((1, 4096), 127, np.int8), np.full((4096, 1), -127, np.int8))
    assert worst[0, 0] == -127 * 127 * 4096
    # brute force on a tiny case
    a2, b2 = a[:3, :5].astype(int), b[:5, :2].astype(int)
    bf = [[sum(a2[i, k] * b2[k, j] for k in range(5)) for j in range(2)] for i in range(3)]
    assert oracle.int8_gemm(a2, b2).tolist() == bf


def test_int8_linear_lossless_on_grid():
    rng = np.random.default_rng(2)
    s_a = np.float32(0.03125)          # power of two: x = k * s_a and 1/s_a exact
    k = rng.integers(-127, 128, size=(20, 64))
    x = k.astype(np.float32) * s_a
    Wq = rng.integers(-127, 128, size=(64, 32)).astype(np.int8)
    s_w = (2.0 ** -rng.integers(6, 10, size=32)).astype(np.float32)
    W = Wq.astype(np.float64) * s_w.astype(np.float64)
    b = rng.standard_normal(32)
    assert np.allclose(oracle.int8_linear(x, s_a, Wq, s_w, b), oracle.linear(x, W, b), atol=1e-12)


def test_calibration_uses_valid_tokens_only():
    cfg = INT8
    wl = make_bert_workload(cfg, B=3, L=16, lengths=np.array([16, 4, 9]))
    cal = make_calibration_batch(cfg)
    x = wl["x_padded"].copy()
    lens = wl["lengths"]
    valid = np.arange(16)[None, :] < lens[:, None]
    x[~valid] = 1e3                     # pads would dominate the max-abs if they were counted
    s = oracle.calibrate_int8(x, lens, wl["layers"][0], cfg.nh, cfg.eps)
    assert s[0] == np.float32(np.abs(x[valid]).max() / 127)
    assert np.all(s > 0) and s.dtype == np.float32
    assert cal["x_padded"].shape == (cfg.B, cfg.L, cfg.H)


def test_int8_layer_close_to_float_layer():
    cfg = INT8
    wl = make_bert_workload(cfg, B=3, L=32, lengths=np.array([32, 17, 5]))
    layer = wl["layers"][0]
    s = oracle.calibrate_int8(wl["x_padded"], wl["lengths"], layer, cfg.nh, cfg.eps)
    cu, po, T = oracle.build_offsets(wl["lengths"], 32)
    x = oracle.remove_padding(wl["x_padded"], po).astype(np.float64)
    yq = oracle.bert_layer_int8(x, cu, oracle.prepare_int8_layer(layer), s, cfg.nh, cfg.eps)
    yf = oracle.bert_layer(x, cu, layer, cfg.nh, cfg.eps)
    err = np.abs(yq - yf)
    # int8 noise: a few percent of a unit-variance output, far from a structural error
    assert err.mean() < 0.05 and err.max() < 0.5
    # a structural mistake (say, a dropped residual) would move outputs by O(1)
    assert not np.allclose(yq, oracle.layernorm(x, np.ones(cfg.H), np.zeros(cfg.H), cfg.eps), atol=0.3)
