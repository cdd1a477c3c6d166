"""Pins for the oracle's Swin pieces.

Routes other than the oracle's own loops: torch.roll and the reshape/permute window
partition for the index maps, the relative-coordinate construction of the bias
index, the slice-based region labelling and the "no attention across the cyclic wrap
seam" meaning of the shift mask, torch's scaled_dot_product_attention with an
additive float mask for the window attention, and special cases (no shift, one
window covering the whole image) that reduce to plain multi-head attention.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import make_swin_workload, config_by_name

torch.set_grad_enabled(False)
SWIN = config_by_name("swin_t_stage1_fp16")


def test_shift_matches_torch_roll_and_inverts():
    rng = np.random.default_rng(0)
    img = rng.standard_normal((14, 14, 3))
    for s in (0, 1, 3, 6):
        ref = torch.roll(torch.from_numpy(img), shifts=(-s, -s), dims=(0, 1)).numpy()
        assert np.array_equal(oracle.shift(img, s), ref)
        assert np.array_equal(oracle.unshift(oracle.shift(img, s), s), img)


def test_partition_matches_reshape_permute_and_inverts():
    rng = np.random.default_rng(1)
    I, w, C = 14, 7, 5
    img = rng.standard_normal((I, I, C))
    ref = img.reshape(I // w, w, I // w, w, C).transpose(0, 2, 1, 3, 4).reshape(-1, w * w, C)
    win = oracle.window_partition(img, w)
    assert np.array_equal(win, ref)
    assert np.array_equal(oracle.window_reverse(win, I, w), img)
    # the full chain shift -> partition -> reverse -> unshift is the identity
    for s in (0, 3):
        back = oracle.unshift(oracle.window_reverse(oracle.window_partition(oracle.shift(img, s), w), I, w), s)
        assert np.array_equal(back, img)


def test_relative_position_bias_index():
    w, nh = 7, 3
    rng = np.random.default_rng(2)
    table = rng.standard_normal(((2 * w - 1) ** 2, nh))
    B = oracle.relative_position_bias(table, w)
    # relative-coordinate construction (vectorised, independent of the oracle's loops)
    coords = np.stack(np.meshgrid(np.arange(w), np.arange(w), indexing="ij")).reshape(2, -1)
    rel = coords[:, :, None] - coords[:, None, :] + (w - 1)
    idx = rel[0] * (2 * w - 1) + rel[1]
    assert np.array_equal(B, table[idx].transpose(2, 0, 1))
    # diagonal is the zero-offset entry, (w-1)(2w-1) + (w-1) = 84 for w = 7
    for t in range(w * w):
        assert np.array_equal(B[:, t, t], table[84])
    # one column to the right (u = t + 1 inside a row): dx = -1 -> entry 83
    assert np.array_equal(B[:, 0, 1], table[83])
    # one row down (u = t + w): dy = -1 -> entry 84 - 13 = 71
    assert np.array_equal(B[:, 0, w], table[71])


def _slice_region_mask(I, w, s):
    img = np.zeros((I, I), np.int64)
    cnt = 0
    for hs in (slice(0, -w), slice(-w, -s), slice(-s, None)):
        for ws in (slice(0, -w), slice(-w, -s), slice(-s, None)):
            img[hs, ws] = cnt
            cnt += 1
    lab = img.reshape(I // w, w, I // w, w).transpose(0, 2, 1, 3).reshape(-1, w * w)
    return lab[:, :, None] == lab[:, None, :]


@pytest.mark.parametrize("I,w,s", [(56, 7, 3), (14, 7, 3), (21, 7, 2), (8, 4, 2)])
def test_shift_mask(I, w, s):
    allow = oracle.shift_attend_mask(I, w, s)
    assert np.array_equal(allow, _slice_region_mask(I, w, s))
    # meaning: two tokens attend iff neither axis separates them across the wrap seam
    yy, xx = oracle.window_coords(I, w)
    wy, wx = (yy + s) >= I, (xx + s) >= I
    seam = (wy[:, :, None] == wy[:, None, :]) & (wx[:, :, None] == wx[:, None, :])
    assert np.array_equal(allow, seam)
    nWs = I // w
    interior = [a * nWs + b for a in range(nWs - 1) for b in range(nWs - 1)]
    assert allow[interior].all()
    # bottom-right window: 4 groups of sizes (w-s)^2, (w-s)s, s(w-s), s^2
    last = allow[-1]
    sizes = sorted(set(int(r.sum()) for r in last))
    assert sizes == sorted({(w - s) * (w - s), (w - s) * s, s * s})
    assert oracle.shift_attend_mask(I, w, 0).all()


def _library_window_attention(qkv, I, w, s, nh, bias_np, allow_np):
    # torch.roll + reshape/permute partition + SDPA with an additive float mask
    B, T, C3 = qkv.shape
    C = C3 // 3
    d = C // nh
    t = torch.from_numpy(qkv).view(B, I, I, C3)
    t = torch.roll(t, shifts=(-s, -s), dims=(1, 2))
    win = t.view(B, I // w, w, I // w, w, C3).permute(0, 1, 3, 2, 4, 5).reshape(-1, w * w, C3)
    nW = (I // w) ** 2
    q, k, v = [win[..., i * C:(i + 1) * C].reshape(-1, w * w, nh, d).transpose(1, 2) for i in range(3)]
    add = torch.from_numpy(bias_np)[None].expand(B * nW, -1, -1, -1).clone()
    allow = torch.from_numpy(allow_np).repeat(B, 1, 1)[:, None]
    add = add.masked_fill(~allow, float("-inf"))
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=add)
    o = o.transpose(1, 2).reshape(B, I // w, I // w, w, w, C).permute(0, 1, 3, 2, 4, 5).reshape(B, I, I, C)
    o = torch.roll(o, shifts=(s, s), dims=(1, 2))
    return o.reshape(B, T, C).numpy()


@pytest.mark.parametrize("I,s", [(14, 3), (14, 0), (21, 3)])
def test_window_attention_matches_library_route(I, s):
    rng = np.random.default_rng(3)
    w, nh, C = 7, 3, 24
    qkv = rng.standard_normal((2, I * I, 3 * C))
    table = 0.5 * rng.standard_normal(((2 * w - 1) ** 2, nh))
    bias = oracle.relative_position_bias(table, w)
    out = oracle.window_attention(qkv, I, w, s, nh, bias)
    ref = _library_window_attention(qkv, I, w, s, nh, bias, oracle.shift_attend_mask(I, w, s))
    assert np.allclose(out, ref, atol=1e-12)


def test_one_window_no_shift_no_bias_is_plain_mha():
    rng = np.random.default_rng(4)
    I = w = 7
    nh, C = 2, 16
    qkv = rng.standard_normal((1, I * I, 3 * C))
    out = oracle.window_attention(qkv, I, w, 0, nh, np.zeros((nh, 49, 49)))
    cu = np.array([0, 49])
    ref = oracle.attention_varlen(qkv[0, :, :C], qkv[0, :, C:2 * C], qkv[0, :, 2 * C:], cu, nh)
    assert np.allclose(out[0], ref, atol=1e-13)


def _library_swin_block(x, wt, I, w, s, nh, eps):
    # torch modules end to end: LayerNorm, Linear, GELU, roll, SDPA with additive mask
    B, T, C = x.shape
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64).copy())
    xt = t(x)
    h = torch.nn.functional.layer_norm(xt, (C,), t(wt["gamma1"]), t(wt["beta1"]), eps)
    qkv = torch.nn.functional.linear(h, t(wt["Wqkv"].T), t(wt["bqkv"])).numpy()
    bias = oracle.relative_position_bias(wt["table"], w)
    a = _library_window_attention(qkv, I, w, s, nh, bias, _slice_region_mask(I, w, s) if s else
                                  np.ones(((I // w) ** 2, w * w, w * w), bool))
    xa = xt + torch.nn.functional.linear(t(a), t(wt["Wo"].T), t(wt["bo"]))
    h2 = torch.nn.functional.layer_norm(xa, (C,), t(wt["gamma2"]), t(wt["beta2"]), eps)
    m = torch.nn.functional.linear(torch.nn.functional.gelu(
        torch.nn.functional.linear(h2, t(wt["W1"].T), t(wt["b1"]))), t(wt["W2"].T), t(wt["b2"]))
    return (xa + m).numpy()


@pytest.mark.parametrize("affine", [False, True])
def test_swin_block_matches_library_route(affine):
    wl = make_swin_workload(SWIN, B=2, I=14, affine=affine)
    cfg = wl["cfg"]
    y = oracle.swin_block(wl["x"], wl["weights"], cfg.I, cfg.w, cfg.s, cfg.nh, cfg.eps)
    ref = _library_swin_block(wl["x"], wl["weights"], cfg.I, cfg.w, cfg.s, cfg.nh, cfg.eps)
    assert np.allclose(y, ref, atol=1e-11)


def test_swin_block_images_independent():
    wl = make_swin_workload(SWIN, B=3, I=14)
    cfg = wl["cfg"]
    x = wl["x"].copy()
    y1 = oracle.swin_block(x, wl["weights"], cfg.I, cfg.w, cfg.s, cfg.nh, cfg.eps)
    x[1] += 1.0
    y2 = oracle.swin_block(x, wl["weights"], cfg.I, cfg.w, cfg.s, cfg.nh, cfg.eps)
    assert np.array_equal(y1[0], y2[0]) and np.array_equal(y1[2], y2[2])


def _patch_merge_torch(x, I, gamma, beta, W, eps):
    """Library route: the 2 x 2 neighbourhoods by view/permute (channel block k = 2 dx + dy),
    torch layer_norm and matmul in fp64."""
    B, _, C = x.shape
    t = torch.as_tensor(x, dtype=torch.float64).view(B, I // 2, 2, I // 2, 2, C)   # [B, py, dy, px, dx, C]
    t = t.permute(0, 1, 3, 4, 2, 5).reshape(B, (I // 2) ** 2, 4 * C)               # [B, py, px, dx, dy, C]
    t = torch.nn.functional.layer_norm(t, (4 * C,), torch.as_tensor(gamma, dtype=torch.float64),
                                       torch.as_tensor(beta, dtype=torch.float64), eps)
    return (t @ torch.as_tensor(W, dtype=torch.float64)).numpy()


@pytest.mark.parametrize("I,C", [(4, 8), (8, 96), (14, 24)])
def test_patch_merge_matches_library_route(I, C):
    rng = np.random.default_rng(I * C)
    B = 2
    x = rng.standard_normal((B, I * I, C))
    gamma = 1 + 0.1 * rng.standard_normal(4 * C)
    beta = 0.1 * rng.standard_normal(4 * C)
    W = 0.05 * rng.standard_normal((4 * C, 2 * C))
    got = oracle.patch_merge(x, I, gamma, beta, W, 1e-5)
    assert got.shape == (B, (I // 2) ** 2, 2 * C)
    assert np.allclose(got, _patch_merge_torch(x, I, gamma, beta, W, 1e-5), rtol=1e-12, atol=1e-12)


def test_patch_merge_gathers_each_token_once():
    """Tokens carrying their own raster index: every input token lands in exactly one output
    token, in the slot its (row, column) parity names."""
    I, C = 6, 1
    x = np.arange(I * I, dtype=np.float64).reshape(1, I * I, 1)
    # W = identity (4C -> 4C here) exposes the normalised concatenation itself
    got = oracle.patch_merge(x, I, np.ones(4), np.zeros(4), np.eye(4), 0.0)[0]   # [9, 4]
    for py in range(I // 2):
        for px in range(I // 2):
            src = [(2 * py + dy) * I + (2 * px + dx) for dy, dx in ((0, 0), (1, 0), (0, 1), (1, 1))]
            v = np.array(src, np.float64)
            ref = (v - v.mean()) / np.sqrt(v.var())
            assert np.allclose(got[py * (I // 2) + px], ref, atol=1e-12)
