"""GPU parity of the INT8 path: weight and activation quantisation bit-exact, int32
accumulators of the int8 GEMM bit-exact (including adversarial all-extreme inputs at
the largest K), the calibration pass, the int8 encoder layer within the int8
tolerance (5e-2 on final outputs; the attention writes the codes of its output, or a
separate kernel quantises it beyond the persistent attention's limits), and the
all-int8 flow: attention on codes (P's
codes read back bit-exact where no code lies near a rounding tie, the output within
the bound of a few flipped codes elsewhere) and the layer with int8 attention."""
import numpy as np
import pytest
import torch

import oracle
import remove_padding_prefix_gb300 as rpp
from workloads import make_bert_workload, make_calibration_batch, round_to_dtype, config_by_name
from gpu_util import dev, up, down, assert_close, check_err

pytestmark = pytest.mark.gpu
INT8 = config_by_name("bert_large_int8")


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


def test_int8_layer_beyond_persistent_attention_limits():
    """2050 short sequences (beyond the persistent attention's 2048): the int8 layer takes
    the one-CTA-per-query-tile attention and a separate quantisation of its output instead
    of the codes written by the persistent kernel; every sequence against the oracle."""
    import dataclasses
    cfg = dataclasses.replace(INT8, H=128, nh=2, F=512)
    rng = np.random.default_rng(2050)
    lengths = rng.integers(0, 5, size=2050).astype(np.int32)
    wl = make_bert_workload(cfg, B=2050, L=4, lengths=lengths, affine=True)
    s = oracle.calibrate_int8(wl["x_padded"], wl["lengths"], wl["layers"][0], cfg.nh, cfg.eps)
    got, cu, x = _int8_case(wl, s)
    T = int(cu[-1])
    ref = oracle.bert_layer_int8(x[:T], cu, oracle.prepare_int8_layer(wl["layers"][0]), s, cfg.nh, cfg.eps)
    assert_close(got[:T], ref, "int8", "int8 layer, 2050 sequences")


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
    ref_qkv = oracle.calibrate_int8_qkv(wl["x_padded"], wl["lengths"], layer, cfg.nh) * 127.0
    got = amax.cpu().numpy()
    assert got.shape == (7,)
    assert got[0] == np.float32(np.abs(wl["x_padded"][np.arange(cfg.L)[None, :] < wl["lengths"][:, None]]).max())
    assert np.allclose(got[:4], ref, rtol=1e-2), (got, ref)
    assert np.allclose(got[4:], ref_qkv, rtol=1e-2), (got, ref_qkv)


# ---------------------------------------------------------------- int8 attention
def _codes_case(seed, lengths, nh, spread=1.0):
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, np.int32)
    T = int(lengths.sum())
    T_max = max(T, 1) + 3
    codes = rng.integers(-127, 128, size=(T_max, 3 * nh * 64)).astype(np.int64)
    codes[:, :2 * nh * 64] = np.rint(codes[:, :2 * nh * 64] * spread).astype(np.int64)
    codes = np.clip(codes, -127, 127)
    err = rpp.new_error_word()
    cu, _ = rpp.build_offsets(torch.as_tensor(lengths, device=dev()), int(max(1, lengths.max())), err=err)
    return codes, cu, err, T


def _run_i8_attention(codes, scales, cu, B, max_len, nh, err):
    qkv = torch.as_tensor(codes.astype(np.float32), device=dev()).to(torch.bfloat16)
    out = rpp.attention_varlen_i8(qkv, torch.as_tensor(np.asarray(scales, np.float32), device=dev()), cu, B, max_len,
                                  nh, err=err)
    torch.cuda.synchronize()
    check_err(err)
    return out.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("lengths,nh", [([384, 1, 200, 129, 0, 64], 4), ([1000, 17], 2), ([128] * 40, 16)])
def test_int8_attention_vs_oracle(lengths, nh):
    """Random codes over ragged lengths (partial and whole tiles, one-token and empty
    sequences, 1000 keys): the output within the effect of a few P codes flipped at a
    rounding tie (each flip moves an output by at most s_v), nearly all outputs well inside."""
    codes, cu, err, T = _codes_case(len(lengths) + nh, lengths, nh)
    scales = (0.03, 0.025, 0.013)   # scores with a spread of several units: codes from 0 to 127
    got = _run_i8_attention(codes, scales, cu, len(lengths), max(lengths), nh, err)
    H = nh * 64
    cc = codes[:T].astype(np.int8)
    ref = oracle.attention_varlen_int8(cc[:, :H], cc[:, H:2 * H], cc[:, 2 * H:], *scales, cu.cpu().numpy(), nh)
    d = np.abs(got[:T] - ref)
    s_v = scales[2]
    assert d.max() <= 3 * s_v, d.max()
    assert (d > 2e-3 * s_v * 127).mean() < 0.02
    assert d.mean() < s_v / 50


def test_int8_attention_codes_read_back_exactly():
    """V = 127 x one-hot rows (key j has code 127 in column j, head size 64, so up to 64
    keys): O[q, j] = Pc[q, j] s_v, which reads P's codes back from the kernel.  Every code
    whose 127 P (fp64) lies at least 1e-3 from a half-integer -- beyond the kernel's fp32
    rounding of P -- must be reproduced bit-exactly (the integer scores Qc Kc^T, the
    softmax and the coding are all checked); a code nearer a tie may be either neighbour."""
    nh, lengths = 2, [64, 37, 5, 1, 50]
    B, T = len(lengths), sum(lengths)
    H = nh * 64
    cu_np = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    scales = (0.02, 0.015, 0.5)
    codes, cu, err, _ = _codes_case(1000, lengths, nh, spread=0.6)
    codes[:, 2 * H:] = 0
    for b in range(B):
        for i in range(lengths[b]):
            codes[cu_np[b] + i, 2 * H + i::64] = 127   # key i of its sequence: column i of every head
    cc = codes[:T].astype(np.int8)
    near_tie = np.zeros((T, H), bool)
    for b in range(B):
        lo, hi = cu_np[b], cu_np[b + 1]
        for h in range(nh):
            cs = slice(h * 64, (h + 1) * 64)
            S = oracle.int8_gemm(cc[lo:hi, cs], cc[lo:hi, H:2 * H][:, cs].T).astype(np.float64)
            z = S * scales[0] * scales[1] / 8.0
            P = np.exp(z - z.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            frac = P * 127 - np.floor(P * 127)
            near_tie[lo:hi, h * 64:h * 64 + (hi - lo)] = np.abs(frac - 0.5) < 1e-3
    got = _run_i8_attention(codes, scales, cu, B, max(lengths), nh, err)
    ref = oracle.attention_varlen_int8(cc[:, :H], cc[:, H:2 * H], cc[:, 2 * H:], *scales, cu_np, nh)
    got_codes = np.rint(got[:T] / scales[2]).astype(np.int64)
    ref_codes = np.rint(ref / scales[2]).astype(np.int64)
    assert np.array_equal(got_codes[~near_tie], ref_codes[~near_tie])
    assert np.abs(got_codes - ref_codes).max() <= 1
    assert near_tie.mean() < 0.01
    assert np.abs(got[:T] - got_codes * scales[2]).max() == 0   # outputs are exact multiples of s_v
    assert ref_codes.max() > 60 and (ref_codes[:, :64] == 0).mean() > 0.1   # large and zero codes both occur


def _int8_attn_case(wl, scales7):
    cfg = wl["cfg"]
    ecfg = rpp.encoder_cfg(cfg.H, cfg.nh, cfg.F, cfg.eps, "fp16", int8=2)
    prepared = rpp.EncoderLayer(ecfg, wl["layers"][0])
    lengths = torch.as_tensor(wl["lengths"], device=dev())
    err = rpp.new_error_word()
    cu, po = rpp.build_offsets(lengths, cfg.L, err=err)
    x = rpp.remove_padding(up(wl["x_padded"].reshape(-1, cfg.H), "fp16"), po, cu, cfg.B, cfg.L, err=err)
    y = rpp.encoder_layer_forward(prepared, x, cu, cfg.B, cfg.L, act_scales=torch.as_tensor(scales7, device=dev()),
                                  err=err)
    check_err(err)
    return down(y), cu.cpu().numpy(), down(x)


@pytest.mark.parametrize("full", [False, True])
def test_int8_attention_layer(full):
    """The all-int8 layer (QKV codes from the GEMM epilogue, attention on codes) against
    the oracle's seven-scale layer: a small ragged batch, and the BERT-large-shaped int8
    config with every sequence."""
    cfg = INT8
    if full:
        wl = make_bert_workload(cfg)
        cal = make_calibration_batch(cfg)
    else:
        wl = make_bert_workload(cfg, B=4, L=160, lengths=np.array([160, 1, 64, 129], np.int32), affine=True)
        cal = wl
    layer = wl["layers"][0]
    s7 = np.concatenate([oracle.calibrate_int8(cal["x_padded"], cal["lengths"], layer, cfg.nh, cfg.eps),
                         oracle.calibrate_int8_qkv(cal["x_padded"], cal["lengths"], layer, cfg.nh)])
    got, cu, x = _int8_attn_case(wl, s7)
    T = int(cu[-1])
    ref = oracle.bert_layer_int8(x[:T], cu, oracle.prepare_int8_layer(layer), s7, cfg.nh, cfg.eps)
    assert_close(got[:T], ref, "int8", f"all-int8 layer full={full}")
