"""Pins for the oracle's encoder-layer pieces and the whole post-LN layer.

Each check reaches the result by a route other than the oracle's own code: closed
forms (GELU at known points, LayerNorm of a two-point row), library routines that
reduce to the same definition (torch's fp64 layer_norm, scaled_dot_product_attention
with a key-padding mask, nn.TransformerEncoderLayer on the padded batch), and
invariants the pages fix (padding removal changes no valid output; sequences are
independent; softmax weights sum to one).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import make_bert_workload, config_by_name

torch.set_grad_enabled(False)


def test_gelu_closed_forms():
    # Phi(1) = 0.841344746068542948585..., Phi(-1) = 1 - Phi(1)  (normal CDF tables)
    assert oracle.gelu(np.array([1.0]))[0] == pytest.approx(0.8413447460685429, abs=1e-15)
    assert oracle.gelu(np.array([-1.0]))[0] == pytest.approx(-0.15865525393145707, abs=1e-15)
    assert oracle.gelu(np.array([0.0]))[0] == 0.0
    x = np.linspace(-6, 6, 101)
    # odd-part identity: GELU(x) - GELU(-x) = x
    assert np.allclose(oracle.gelu(x) - oracle.gelu(-x), x, atol=1e-14)
    assert oracle.gelu(np.array([40.0]))[0] == 40.0
    # the tanh approximation is a different function: differs by > 1e-4 somewhere
    tanh_form = 0.5 * x * (1 + np.tanh(math.sqrt(2 / math.pi) * (x + 0.044715 * x ** 3)))
    assert np.abs(oracle.gelu(x) - tanh_form).max() > 1e-4


def test_layernorm_closed_form_and_library():
    # row [1, -1]: mean 0, biased variance 1 -> x / sqrt(1 + eps)
    y = oracle.layernorm(np.array([[1.0, -1.0]]), np.ones(2), np.zeros(2), 1.0)
    assert np.allclose(y, [[1 / math.sqrt(2), -1 / math.sqrt(2)]], atol=1e-15)
    rng = np.random.default_rng(0)
    x = rng.standard_normal((37, 96)) * 3 + 1.5
    g = 1 + 0.1 * rng.standard_normal(96)
    b = 0.1 * rng.standard_normal(96)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (96,), torch.from_numpy(g),
                                         torch.from_numpy(b), eps=1e-5).numpy()
    assert np.allclose(oracle.layernorm(x, g, b, 1e-5), ref, atol=1e-12)
    y = oracle.layernorm(x, np.ones(96), np.zeros(96), 1e-12)
    assert np.allclose(y.mean(-1), 0, atol=1e-12) and np.allclose(y.var(-1), 1, atol=1e-9)


def test_linear_matches_library_orientation():
    rng = np.random.default_rng(1)
    x, W, b = rng.standard_normal((5, 7)), rng.standard_normal((7, 3)), rng.standard_normal(3)
    ref = torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(W.T.copy()),
                                     torch.from_numpy(b)).numpy()
    assert np.allclose(oracle.linear(x, W, b), ref, atol=1e-13)


def _rand_qkv(rng, lengths, nh, d):
    T = int(sum(lengths))
    return [rng.standard_normal((T, nh * d)) for _ in range(3)]


def test_attention_matches_padded_sdpa():
    rng = np.random.default_rng(2)
    lengths = [5, 1, 13, 8]
    nh, d = 3, 16
    L = 13
    cu, po, T = oracle.build_offsets(lengths, L)
    q, k, v = _rand_qkv(rng, lengths, nh, d)
    out = oracle.attention_varlen(q, k, v, cu, nh)
    # library route: pad, mask keys, torch SDPA in fp64
    def padded(t):
        p = oracle.rebuild_padding(t, cu, len(lengths), L)
        return torch.from_numpy(p).view(len(lengths), L, nh, d).transpose(1, 2)
    keymask = torch.from_numpy(np.arange(L)[None, :] < np.array(lengths)[:, None])
    ref = torch.nn.functional.scaled_dot_product_attention(
        padded(q), padded(k), padded(v), attn_mask=keymask[:, None, None, :])
    ref = ref.transpose(1, 2).reshape(len(lengths), L, nh * d).numpy()
    assert np.allclose(out, oracle.remove_padding(ref, po), atol=1e-12)


def test_attention_invariants():
    rng = np.random.default_rng(4)
    lengths = [4, 9, 1]
    nh, d = 2, 8
    cu, _, T = oracle.build_offsets(lengths, 9)
    q, k, v = _rand_qkv(rng, lengths, nh, d)
    # weights sum to one: all-ones V gives exactly one
    assert np.allclose(oracle.attention_varlen(q, k, np.ones_like(v), cu, nh), 1.0, atol=1e-14)
    # q = 0: uniform weights -> mean of the sequence's own values
    out = oracle.attention_varlen(np.zeros_like(q), k, v, cu, nh)
    for b in range(3):
        lo, hi = cu[b], cu[b + 1]
        assert np.allclose(out[lo:hi], v[lo:hi].mean(0), atol=1e-14)
    # sequences are independent: each alone gives the same rows
    full = oracle.attention_varlen(q, k, v, cu, nh)
    for b in range(3):
        lo, hi = cu[b], cu[b + 1]
        alone = oracle.attention_varlen(q[lo:hi], k[lo:hi], v[lo:hi], np.array([0, hi - lo]), nh)
        assert np.allclose(alone, full[lo:hi], atol=1e-14)
    # permuting keys and values together inside a sequence changes nothing
    perm = np.arange(T)
    perm[cu[1]:cu[2]] = cu[1] + rng.permutation(lengths[1])
    assert np.allclose(oracle.attention_varlen(q, k[perm], v[perm], cu, nh), full, atol=1e-13)
    # single-token sequence returns its own value
    assert np.allclose(full[cu[2]], v[cu[2]], atol=1e-15)


def test_attention_brute_force_tiny():
    rng = np.random.default_rng(5)
    lengths = [3, 2]
    nh, d = 2, 4
    cu, _, _ = oracle.build_offsets(lengths, 3)
    q, k, v = _rand_qkv(rng, lengths, nh, d)
    out = oracle.attention_varlen(q, k, v, cu, nh)
    for b in range(2):
        for h in range(nh):
            for i in range(cu[b], cu[b + 1]):
                logits = [sum(q[i, h * d + c] * k[j, h * d + c] for c in range(d)) / math.sqrt(d)
                          for j in range(cu[b], cu[b + 1])]
                mx = max(logits)
                w = [math.exp(z - mx) for z in logits]
                den = sum(w)
                for c in range(d):
                    val = sum(w[jj] * v[cu[b] + jj, h * d + c] for jj in range(len(w))) / den
                    assert abs(val - out[i, h * d + c]) < 1e-13


def _torch_layer(layer, H, nh, F, eps):
    m = torch.nn.TransformerEncoderLayer(d_model=H, nhead=nh, dim_feedforward=F, dropout=0.0,
                                         activation="gelu", layer_norm_eps=eps, batch_first=True,
                                         norm_first=False, dtype=torch.float64)
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64).copy())
    m.self_attn.in_proj_weight.copy_(t(layer["Wqkv"].T))
    m.self_attn.in_proj_bias.copy_(t(layer["bqkv"]))
    m.self_attn.out_proj.weight.copy_(t(layer["Wo"].T))
    m.self_attn.out_proj.bias.copy_(t(layer["bo"]))
    m.linear1.weight.copy_(t(layer["W1"].T))
    m.linear1.bias.copy_(t(layer["b1"]))
    m.linear2.weight.copy_(t(layer["W2"].T))
    m.linear2.bias.copy_(t(layer["b2"]))
    m.norm1.weight.copy_(t(layer["gamma1"]))
    m.norm1.bias.copy_(t(layer["beta1"]))
    m.norm2.weight.copy_(t(layer["gamma2"]))
    m.norm2.bias.copy_(t(layer["beta2"]))
    m.train()   # the standard (non-fused) code path; dropout is 0
    return m


@pytest.mark.parametrize("affine", [False, True])
def test_bert_layer_matches_torch_encoder_layer_on_padded_batch(affine):
    cfg = config_by_name("tiny_fp32")
    wl = make_bert_workload(cfg, B=3, L=20, affine=affine, lengths=np.array([20, 7, 1]))
    layer = wl["layers"][0]
    y_pad, cu, po = oracle.bert_forward(wl["x_padded"], wl["lengths"], wl["layers"], cfg.nh, cfg.eps)
    m = _torch_layer(layer, cfg.H, cfg.nh, cfg.F, cfg.eps)
    pad_mask = torch.from_numpy(np.arange(20)[None, :] >= wl["lengths"][:, None])
    ref = m(torch.from_numpy(wl["x_padded"].astype(np.float64)), src_key_padding_mask=pad_mask).numpy()
    valid = ~pad_mask.numpy()
    assert np.allclose(y_pad[valid], ref[valid], atol=1e-11)
    assert np.all(y_pad[~valid] == 0)


def test_bert_layer_padding_removal_changes_nothing_and_sequences_independent():
    cfg = config_by_name("tiny_fp32")
    wl = make_bert_workload(cfg, B=4, L=16, lengths=np.array([16, 3, 9, 12]))
    x = wl["x_padded"].copy()
    valid = np.arange(16)[None, :] < wl["lengths"][:, None]
    y1, _, _ = oracle.bert_forward(x, wl["lengths"], wl["layers"], cfg.nh, cfg.eps)
    x2 = x.copy()
    x2[~valid] = 1e4                                    # pad contents never matter
    y2, _, _ = oracle.bert_forward(x2, wl["lengths"], wl["layers"], cfg.nh, cfg.eps)
    assert np.array_equal(y1, y2)
    x3 = x.copy()
    x3[2, :9] += 0.5                                    # perturb sequence 2 only
    y3, _, _ = oracle.bert_forward(x3, wl["lengths"], wl["layers"], cfg.nh, cfg.eps)
    for b in (0, 1, 3):
        assert np.array_equal(y1[b], y3[b])
    assert not np.allclose(y1[2, :9], y3[2, :9])
    # a two-layer stack equals two single-layer passes
    wl2 = make_bert_workload(cfg, B=2, L=8, layers=2, lengths=np.array([8, 5]))
    ys, cu, po = oracle.bert_forward(wl2["x_padded"], wl2["lengths"], wl2["layers"], cfg.nh, cfg.eps)
    ya, _, _ = oracle.bert_forward(wl2["x_padded"], wl2["lengths"], wl2["layers"][:1], cfg.nh, cfg.eps)
    yb, _, _ = oracle.bert_forward(ya, wl2["lengths"], wl2["layers"][1:], cfg.nh, cfg.eps)
    assert np.allclose(ys, yb, atol=1e-13)
