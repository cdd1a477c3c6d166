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
from workloads import make_bert_workload, make_calibration_batch, config_by_name

INT8 = config_by_name("bert_large_int8")


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


# ---------------------------------------------------------------- exact pins of the int8 flow
# A small layer (H = 8, two heads of 4, F = 8) built so that every GEMM input of the
# float layer lies exactly on the grid of its activation scale, with odd codes and codes
# above 63 in each.  Then quantisation is lossless with the right scale and lossy with
# any other power-of-two scale (a coarser one cannot hold the odd codes, a finer one
# clamps the large codes), so the int8 layer must equal the float layer to rounding,
# and a scale taken for the wrong tensor or a residual taken from the wrong place must
# show up in the output.
#
# Construction (sigma = [1, -1, 1, -1, ...], P = projection onto span{sigma, 1},
# Pp = I - P; scales s0 = 2^-4 (QKV input), s1 = 2^-2 (attention output), s2 = 2^-5
# (FC1 input), s3 = 2^-3 (FC2 input)):
#   Q weights 0 -> every score is 0 -> attention is the plain mean of V over the
#     sequence (lengths 1 and 2, pairs differing by an even-coded multiple of
#     sigma and 1);
#   V weights 4 I -> attention output 4 * mean(x) on the s1 grid;
#   Wo = -Pp / 4 -> x + proj = x P, a row a sigma + b 1: LayerNorm with eps = 0 maps it
#     to sign(a) sigma exactly, so LN1's output is +-gamma1 sigma + beta1 (dyadic);
#   W1 = 8 I, b1 chosen so each column's pre-GELU value is >= 9 (GELU(h) = h in fp64)
#     or <= -9 (GELU(h) = 0), the positive ones on the s3 grid.
_SIG = np.array([1.0, -1.0] * 4)
_S = (2.0 ** -4, 2.0 ** -2, 2.0 ** -5, 2.0 ** -3)   # s0, s1, s2, s3: four distinct scales


def _grid_case():
    H, F, nh = 8, 8, 2
    s0, s1, s2, s3 = _S
    rng = np.random.default_rng(77)
    # x codes: three single-token sequences and two pairs; pair rows differ by
    # 2 * (p sigma + q 1) codes, so the pair mean has integer codes
    rows, lengths = [], []
    for _ in range(3):
        c = rng.integers(-120, 121, size=H)
        c[0] = 125 if c[0] >= 0 else -125    # a large code: a 2x finer scale clamps it
        c[1] |= 1                             # an odd code: a 2x coarser scale loses it
        rows.append(c)
        lengths.append(1)
    for p, q in ((3, -5), (-7, 2)):
        a = rng.integers(-90, 91, size=H)
        a[2] = 97
        a[3] |= 1
        rows += [a, a + 2 * (p * _SIG + q).astype(np.int64)]
        lengths.append(2)
    xcodes = np.array(rows, np.int64)
    assert np.abs(xcodes).max() <= 127
    x = xcodes * s0
    cu = np.concatenate([[0], np.cumsum(lengths)])

    P = (np.outer(_SIG, _SIG) + np.ones((H, H))) / H
    Pp = np.eye(H) - P
    # weights as codes x per-column power-of-two scales (the float layer is codes * scale)
    wqkv_codes = np.zeros((H, 3 * H), np.int64)
    wqkv_s = np.ones(3 * H)
    wqkv_codes[:, H:2 * H] = rng.integers(-127, 128, size=(H, H))   # K: anything (Q = 0)
    wqkv_s[H:2 * H] = 2.0 ** -7
    wqkv_codes[:, 2 * H:] = 64 * np.eye(H, dtype=np.int64)          # V = 4 x
    wqkv_s[2 * H:] = 2.0 ** -4
    wo_codes = np.rint(-Pp * 4).astype(np.int64)                     # -Pp / 4 = codes / 16
    assert np.array_equal(wo_codes / 16.0, -Pp / 4)
    wo_s = np.full(H, 2.0 ** -4)
    gamma1 = np.array([2.5, 1.75, 3.0, 1.78125, 1.75, 2.0, 1.96875, 2.25])
    beta1 = np.array([0.9375, -0.5, 0.25, 0.03125, -1.0, 0.5, 0.0, -1.71875])
    w1_codes = 32 * np.eye(H, dtype=np.int64)                        # W1 = 8 I
    w1_s = np.full(F, 2.0 ** -2)
    targets = np.array([9.25, 10.125, 11.0, 12.375, 13.5, 14.625, 15.0, 15.875])
    b1 = np.zeros(F)
    for f in range(F):   # the larger of the two possible LN1 outputs of column f maps to its target
        hi = max(gamma1[f] + beta1[f], -gamma1[f] + beta1[f])
        b1[f] = targets[f] - 8 * hi
    w2_codes = rng.integers(-127, 128, size=(F, H))
    w2_s = 2.0 ** -rng.integers(6, 9, size=H).astype(np.float64)
    b2 = rng.integers(-64, 65, size=H) * 2.0 ** -8

    f32 = lambda a: np.asarray(a, np.float32)
    layer = {"Wqkv": wqkv_codes * wqkv_s, "bqkv": np.zeros(3 * H), "Wo": wo_codes * wo_s, "bo": np.zeros(H),
             "W1": w1_codes * w1_s, "b1": b1, "W2": w2_codes * w2_s, "b2": b2,
             "gamma1": gamma1, "beta1": beta1, "gamma2": np.ones(H), "beta2": np.zeros(H)}
    qlayer = {"Wqkv_q": wqkv_codes.astype(np.int8), "Wqkv_s": f32(wqkv_s), "Wo_q": wo_codes.astype(np.int8),
              "Wo_s": f32(wo_s), "W1_q": w1_codes.astype(np.int8), "W1_s": f32(w1_s),
              "W2_q": w2_codes.astype(np.int8), "W2_s": f32(w2_s)}
    for k in ("bqkv", "bo", "b1", "b2", "gamma1", "beta1", "gamma2", "beta2"):
        qlayer[k] = layer[k]
    return x, cu, layer, qlayer, nh


def _on_grid(t, s, what):
    codes = np.asarray(t, np.float64) / s
    assert np.array_equal(codes, np.rint(codes)), f"{what} off the grid"
    assert np.abs(codes).max() <= 127, f"{what} beyond 127 codes"
    c = np.rint(codes).astype(np.int64)
    assert (c % 2 != 0).any() and np.abs(c).max() > 63, f"{what} must hold odd and large codes"


def test_grid_case_construction_is_exact():
    """The construction above really puts each GEMM input of the float layer on its grid
    (checked with the oracle's float pieces, which have their own pins)."""
    x, cu, layer, _, nh = _grid_case()
    s0, s1, s2, s3 = _S
    H = x.shape[1]
    _on_grid(x, s0, "QKV input")
    qkv = oracle.linear(x, layer["Wqkv"], layer["bqkv"])
    assert np.all(qkv[:, :H] == 0)
    attn = oracle.attention_varlen(qkv[:, :H], qkv[:, H:2 * H], qkv[:, 2 * H:], cu, nh)
    _on_grid(attn, s1, "attention output")
    y = x + oracle.linear(attn, layer["Wo"], layer["bo"])
    x1 = oracle.layernorm(y, layer["gamma1"], layer["beta1"], 0.0)
    _on_grid(x1, s2, "LN1 output")
    h = oracle.linear(x1, layer["W1"], layer["b1"])
    assert np.all((h >= 9) | (h <= -9))
    g = oracle.gelu(h)
    assert np.array_equal(g, np.where(h > 0, h, 0.0))
    _on_grid(g, s3, "GELU output")


def test_int8_layer_equals_float_layer_on_grid():
    """With every GEMM input on its scale's grid the int8 layer is the float layer."""
    x, cu, layer, qlayer, nh = _grid_case()
    yq = oracle.bert_layer_int8(x, cu, qlayer, np.array(_S, np.float32), nh, 0.0)
    yf = oracle.bert_layer(x, cu, layer, nh, 0.0)
    assert np.abs(yq - yf).max() < 1e-12


@pytest.mark.parametrize("i,j", [(0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3)])
def test_int8_layer_grid_case_sees_every_scale_swap(i, j):
    """The pin above is sensitive: exchanging any two of the four scales moves the
    output far beyond rounding (so a scale wired to the wrong tensor cannot pass it)."""
    x, cu, layer, qlayer, nh = _grid_case()
    s = list(_S)
    s[i], s[j] = s[j], s[i]
    yq = oracle.bert_layer_int8(x, cu, qlayer, np.array(s, np.float32), nh, 0.0)
    yf = oracle.bert_layer(x, cu, layer, nh, 0.0)
    assert np.abs(yq - yf).max() > 1e-3


def test_int8_layer_grid_case_sees_the_residual_source():
    """The FC2 residual is LN1's output, not the layer input: the two differ here by
    O(1), so a layer that took the wrong one could not match the float layer."""
    x, cu, layer, _, nh = _grid_case()
    x1 = oracle.layernorm(x + oracle.linear(oracle.attention_varlen(
        *np.split(oracle.linear(x, layer["Wqkv"], layer["bqkv"]), 3, axis=1), cu, nh), layer["Wo"], layer["bo"]),
        layer["gamma1"], layer["beta1"], 0.0)
    assert np.abs(x1 - x).max() > 1.0


def test_calibration_scales_hand_checked():
    """calibrate_int8 on the grid case: the four max-abs values written out by hand from
    the construction (mean of V, +-gamma1 + beta1, the GELU targets)."""
    x, cu, layer, _, nh = _grid_case()
    lengths = np.diff(cu)
    L = int(lengths.max())
    B = len(lengths)
    xp = np.zeros((B, L, x.shape[1]))
    for b in range(B):
        xp[b, :lengths[b]] = x[cu[b]:cu[b + 1]]
    s = oracle.calibrate_int8(xp, lengths, layer, nh, 0.0)
    # QKV input: the largest |x|
    assert s[0] == np.float32(np.abs(x).max() / 127)
    # attention output: 4 x the per-sequence mean of x (Q = 0: uniform weights)
    means = np.concatenate([np.repeat(x[cu[b]:cu[b + 1]].mean(axis=0, keepdims=True), lengths[b], axis=0)
                            for b in range(B)])
    assert s[1] == np.float32(np.abs(4 * means).max() / 127)
    # LN1 output: +-gamma1 sigma + beta1 with the sign of the row's sigma component
    sign = np.sign(x @ _SIG)   # x + proj = x P, whose sigma component has the sign of x . sigma
    x1 = sign[:, None] * _SIG[None, :] * layer["gamma1"][None, :] + layer["beta1"][None, :]
    assert s[2] == np.float32(np.abs(x1).max() / 127)
    # FC2 input: GELU(8 x1 + b1) = the positive targets, 0 for the negative side
    h = 8 * x1 + layer["b1"]
    assert s[3] == np.float32(np.where(h > 0, h, 0).max() / 127)
    # the four tensors have different maxima, so a scale taken from a neighbouring
    # tensor (say the pre-LN sum for the FC1 input, the pre-GELU value for the FC2
    # input) cannot pass
    assert len(set(np.float32(v) for v in s)) == 4


def test_calibration_scales_match_library_route():
    """calibrate_int8 on the int8 configuration's shapes (small batch) against torch's own
    scaled_dot_product_attention (padded batch, key mask), layer_norm and exact gelu in
    fp64: all four scales, within fp32 rounding of the max-abs / 127."""
    import torch
    torch.set_grad_enabled(False)
    cfg = INT8
    wl = make_bert_workload(cfg, B=3, L=24, lengths=np.array([24, 7, 13]))
    layer, lens = wl["layers"][0], wl["lengths"]
    B, L, H, nh, d = 3, 24, cfg.H, cfg.nh, cfg.d
    s = oracle.calibrate_int8(wl["x_padded"], lens, layer, nh, cfg.eps)
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    xp = t(wl["x_padded"])
    valid = torch.from_numpy(np.arange(L)[None, :] < lens[:, None])
    qkv = xp @ t(layer["Wqkv"]) + t(layer["bqkv"])
    q, k, v = [qkv[..., i * H:(i + 1) * H].reshape(B, L, nh, d).transpose(1, 2) for i in range(3)]
    attn = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=valid[:, None, None, :])
    attn = attn.transpose(1, 2).reshape(B, L, H)
    x1 = torch.nn.functional.layer_norm(xp + attn @ t(layer["Wo"]) + t(layer["bo"]), (H,), t(layer["gamma1"]),
                                        t(layer["beta1"]), eps=cfg.eps)
    g = torch.nn.functional.gelu(x1 @ t(layer["W1"]) + t(layer["b1"]), approximate="none")
    want = [float(a[valid].abs().max()) / 127 for a in (xp, attn, x1, g)]
    assert np.allclose(s.astype(np.float64), want, rtol=2e-7, atol=0)
    # neighbouring tensors are far apart: pre-LN sum vs LN output, pre-GELU vs GELU
    pre_ln = xp + attn @ t(layer["Wo"]) + t(layer["bo"])
    pre_gelu = x1 @ t(layer["W1"]) + t(layer["b1"])
    assert abs(float(pre_ln[valid].abs().max()) / 127 - s[2]) > 1e-3 * s[2]
    assert abs(float(pre_gelu[valid].abs().max()) / 127 - s[3]) > 1e-3 * s[3]


# ---------------------------------------------------------------- int8 attention

def _brute_int8_attention(qc, kc, vc, s_q, s_k, s_v, cu, nh):
    """The all-int8 attention restated with scalar Python loops (math.exp, Python's
    round-half-to-even `round`), for tiny shapes."""
    import math
    T, Hd = qc.shape
    d = Hd // nh
    out = np.zeros((T, Hd))
    for b in range(len(cu) - 1):
        lo, hi = int(cu[b]), int(cu[b + 1])
        for h in range(nh):
            for i in range(lo, hi):
                sc = []
                for j in range(lo, hi):
                    acc = 0
                    for c in range(h * d, (h + 1) * d):
                        acc += int(qc[i, c]) * int(kc[j, c])
                    sc.append(acc * float(s_q) * float(s_k) / math.sqrt(d))
                m = max(sc)
                e = [math.exp(v - m) for v in sc]
                tot = sum(e)
                codes = [min(127, max(0, round(127 * v / tot))) for v in e]
                for c in range(h * d, (h + 1) * d):
                    acc = 0
                    for jj, j in enumerate(range(lo, hi)):
                        acc += codes[jj] * int(vc[j, c])
                    out[i, c] = acc * float(s_v) / 127
    return out


def _int8_attention_case(seed, lengths, nh=2, d=4):
    rng = np.random.default_rng(seed)
    T = int(np.sum(lengths))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    qc, kc, vc = (rng.integers(-127, 128, size=(T, nh * d)).astype(np.int8) for _ in range(3))
    return qc, kc, vc, cu


def test_int8_attention_matches_brute_force():
    qc, kc, vc, cu = _int8_attention_case(3, [3, 5, 1, 4])
    s_q, s_k, s_v = np.float32(0.011), np.float32(0.0043), np.float32(0.021)
    got = oracle.attention_varlen_int8(qc, kc, vc, s_q, s_k, s_v, cu, 2)
    ref = _brute_int8_attention(qc, kc, vc, s_q, s_k, s_v, cu, 2)
    assert np.abs(got - ref).max() < 1e-12


@pytest.mark.parametrize("n,code", [(1, 127), (2, 64), (3, 42), (4, 32), (5, 25), (7, 18)])
def test_int8_attention_uniform_scores_closed_form(n, code):
    """Q = 0: every score is 0, P = 1/n, its code is rne(127/n) (n = 2: 63.5 -> 64, the
    even neighbour), and O = code * sum_j v_j * s_v / 127."""
    rng = np.random.default_rng(n)
    nh, d = 1, 8
    qc = np.zeros((n, d), np.int8)
    kc = rng.integers(-127, 128, size=(n, d)).astype(np.int8)
    vc = rng.integers(-127, 128, size=(n, d)).astype(np.int8)
    s_v = np.float32(0.5)
    got = oracle.attention_varlen_int8(qc, kc, vc, 1.0, 1.0, s_v, np.array([0, n]), nh)
    expect = code * vc.astype(np.int64).sum(axis=0) * 0.5 / 127
    assert np.abs(got - np.tile(expect, (n, 1))).max() < 1e-12


def test_int8_attention_close_to_float_attention():
    """Against the float attention of the dequantised Q, K, V: P's codes are within half
    a step (1/254) of P, so each output is within sum_j |v_j| / 254 of the float one
    (and strictly nearer than the bound for most rows)."""
    qc, kc, vc, cu = _int8_attention_case(11, [17, 40, 2, 64], nh=2, d=16)
    s_q, s_k, s_v = np.float32(0.02), np.float32(0.03), np.float32(0.01)
    got = oracle.attention_varlen_int8(qc, kc, vc, s_q, s_k, s_v, cu, 2)
    ref = oracle.attention_varlen(qc * np.float64(s_q), kc * np.float64(s_k), vc * np.float64(s_v), cu, 2)
    d = 16
    for b in range(len(cu) - 1):
        lo, hi = cu[b], cu[b + 1]
        for h in range(2):
            cs = slice(h * d, (h + 1) * d)
            bound = np.abs(vc[lo:hi, cs].astype(np.float64) * s_v).sum(axis=0) / 254 + 1e-12
            assert np.all(np.abs(got[lo:hi, cs] - ref[lo:hi, cs]) <= bound[None, :])
    assert np.abs(got - ref).max() > 0   # the quantisation of P is visible


def test_int8_attention_sequences_are_isolated():
    qc, kc, vc, cu = _int8_attention_case(5, [6, 9, 3])
    a = oracle.attention_varlen_int8(qc, kc, vc, 0.01, 0.02, 0.03, cu, 2)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[6:15] = -kc2[6:15]
    vc2[6:15] = 7
    b = oracle.attention_varlen_int8(qc, kc2, vc2, 0.01, 0.02, 0.03, cu, 2)
    assert np.array_equal(a[:6], b[:6]) and np.array_equal(a[15:], b[15:])
    assert not np.array_equal(a[6:15], b[6:15])


def test_int8_attention_layer_on_grid():
    """The all-int8 layer on the grid case with s_v = the grid of V (4 s0): a one-token
    sequence has P = 1, code 127, attention output V exactly, so its rows equal the float
    layer; a two-token sequence has P = 1/2, code 64, attention output
    64 (v_1 + v_2) s_v / 127 in place of the mean."""
    x, cu, layer, qlayer, nh = _grid_case()
    s_v = 4 * _S[0]
    scales7 = np.array(list(_S) + [2.0 ** -3, 2.0 ** -6, s_v], np.float32)
    y7 = oracle.bert_layer_int8(x, cu, qlayer, scales7, nh, 0.0)
    yf = oracle.bert_layer(x, cu, layer, nh, 0.0)
    assert np.abs(y7[:3] - yf[:3]).max() < 1e-12
    assert np.abs(y7[3:] - yf[3:]).max() > 1e-3
    # the pairs' attention output, from the same pieces the layer uses
    H = x.shape[1]
    qkv = oracle.int8_linear(x, _S[0], qlayer["Wqkv_q"], qlayer["Wqkv_s"], qlayer["bqkv"])
    vc = oracle.quantize_activation(qkv[:, 2 * H:], s_v).astype(np.int64)
    att = oracle.attention_varlen_int8(oracle.quantize_activation(qkv[:, :H], 2.0 ** -3),
                                       oracle.quantize_activation(qkv[:, H:2 * H], 2.0 ** -6),
                                       vc.astype(np.int8), 2.0 ** -3, 2.0 ** -6, s_v, cu, nh)
    for lo in (3, 5):
        expect = 64 * (vc[lo] + vc[lo + 1]) * s_v / 127
        assert np.abs(att[lo] - expect).max() < 1e-12 and np.abs(att[lo + 1] - expect).max() < 1e-12
    # a wrong V scale breaks the one-token rows
    bad = scales7.copy()
    bad[6] = 2 * s_v
    yb = oracle.bert_layer_int8(x, cu, qlayer, bad, nh, 0.0)
    assert np.abs(yb[:3] - yf[:3]).max() > 1e-3


def test_calibrate_int8_qkv_hand_checked():
    """Scales of Q, K and V: max |.| / 127 over valid tokens of x Wqkv + b, per part."""
    rng = np.random.default_rng(4)
    H = 8
    lengths = np.array([2, 0, 3], np.int32)
    x = rng.standard_normal((3, 4, H))
    x[0, 2:] = 1e6   # padding: never counted
    x[2, 3:] = 1e6
    layer = {"Wqkv": rng.standard_normal((H, 3 * H)), "bqkv": rng.standard_normal(3 * H)}
    s = oracle.calibrate_int8_qkv(x, lengths, layer, 2)
    rows = np.concatenate([x[0, :2], x[2, :3]])
    qkv = rows @ layer["Wqkv"] + layer["bqkv"]
    for i in range(3):
        assert s[i] == np.float32(np.abs(qkv[:, i * H:(i + 1) * H]).max() / 127)
