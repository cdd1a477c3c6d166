"""GPU parity of the Swin path: the preprocessed relative-position bias (exact), the
fused shifted-window attention (its gather/scatter index map exact, values within
tolerance, with and without shift) and the whole pre-LN block, small and at the
full Swin-T stage-1 size on sampled images."""
import numpy as np
import pytest
import torch

import oracle
import remove_padding_prefix_gb300 as rpp
from workloads import make_swin_workload, round_to_dtype, config_by_name
from gpu_util import dev, up, down, assert_close, check_err

pytestmark = pytest.mark.gpu
SWIN = config_by_name("swin_t_stage1_fp16")


def _cfg(I=56, s=3, dtype="fp16"):
    return rpp.swin_cfg(I, 96, 3, 7, s, 384, 1e-5, dtype)


def test_relative_position_bias_exact():
    rng = np.random.default_rng(0)
    table = round_to_dtype(0.02 * rng.standard_normal((169, 3), dtype=np.float32), "fp16")
    bias = rpp.swin_prepare_bias(_cfg(), up(table, "fp16"))
    assert np.array_equal(bias.cpu().numpy(), oracle.relative_position_bias(table, 7).astype(np.float32))


@pytest.mark.parametrize("I,s,dtype,B", [(14, 3, "fp16", 2), (14, 0, "fp16", 2), (56, 3, "bf16", 2), (21, 2, "fp16", 2),
                                         (56, 3, "fp16", 9)])
def test_window_attention(I, s, dtype, B):
    """B = 9 at 56 x 56 gives more windows than the kernel's CTAs per head, so each CTA
    walks several windows (with the next one's rows prefetched)."""
    rng = np.random.default_rng(I + s)
    C = 96
    qkv = round_to_dtype(rng.standard_normal((B, I * I, 3 * C), dtype=np.float32), dtype)
    table = round_to_dtype(0.5 * rng.standard_normal((169, 3), dtype=np.float32), dtype)
    cfg = _cfg(I, s, dtype)
    bias = rpp.swin_prepare_bias(cfg, up(table, dtype))
    err = rpp.new_error_word()
    out = rpp.window_attention_forward(cfg, B, up(qkv.reshape(-1, 3 * C), dtype), bias, err=err)
    check_err(err)
    ref = oracle.window_attention(qkv, I, 7, s, 3, oracle.relative_position_bias(table, 7))
    assert_close(down(out).reshape(B, I * I, C), ref, dtype, f"window attention I={I} s={s}")


def test_window_attention_index_map_exact():
    """Q = K = large random vectors: each token's softmax saturates to itself, so the
    output row must equal the same raster row of V exactly -- the shifted gather and
    the reverse/unshift scatter are inverse index maps."""
    rng = np.random.default_rng(1)
    B, I, C = 2, 56, 96
    qk = rng.standard_normal((B, I * I, 3, 32)).astype(np.float32)
    qk = 16.0 * qk / np.linalg.norm(qk, axis=-1, keepdims=True)
    v = rng.standard_normal((B, I * I, C)).astype(np.float32)
    qkv = np.concatenate([qk.reshape(B, I * I, C), qk.reshape(B, I * I, C), v], axis=-1)
    qkv = round_to_dtype(qkv, "fp16")
    cfg = _cfg(I, 3)
    bias = torch.zeros(3, 49, 49, device=dev())
    out = rpp.window_attention_forward(cfg, B, up(qkv.reshape(-1, 3 * C), "fp16"), bias)
    assert np.array_equal(out.float().cpu().numpy().reshape(B, I * I, C), qkv[..., 2 * C:])


@pytest.mark.parametrize("affine,dtype", [(True, "fp16"), (False, "bf16")])
def test_swin_block_small(affine, dtype):
    wl = make_swin_workload(SWIN, B=3, I=14, affine=affine)
    c = wl["cfg"]
    cfg = rpp.swin_cfg(c.I, c.C, c.nh, c.w, c.s, c.F, c.eps, dtype)
    w = {k: round_to_dtype(v, dtype) for k, v in wl["weights"].items()}
    x = round_to_dtype(wl["x"], dtype)
    block = rpp.SwinBlock(cfg, w)
    err = rpp.new_error_word()
    y = rpp.swin_block_forward(block, up(x.reshape(-1, c.C), dtype), c.B, err=err)
    check_err(err)
    ref = oracle.swin_block(x, w, c.I, c.w, c.s, c.nh, c.eps)
    assert_close(down(y).reshape(ref.shape), ref, dtype, "swin block small")


def test_swin_block_multi_tile_ragged():
    """13 images of 56 x 56 (40 768 tokens = 318.5 tiles of 128): the fused MLP's CTAs each
    run two or three tiles through the cross-tile pipeline, and the last tile is half
    full.  Images are independent; the oracle checks the first, a middle and the last.
    Run in fp16: at this size the block's outputs reach |y| ~ 5, where one bf16 step is
    0.031, so the bf16 rounding of y (and of the residual stream before it) alone exceeds
    the 2e-2 max-abs bound (measured 2.6e-2, mean-abs 1.5e-3); the kernel code is the same
    for both types, and bf16 is checked on the smaller block."""
    dtype = "fp16"
    wl = make_swin_workload(SWIN, B=13, affine=True)
    c = wl["cfg"]
    cfg = rpp.swin_cfg(c.I, c.C, c.nh, c.w, c.s, c.F, c.eps, dtype)
    w = {k: round_to_dtype(v, dtype) for k, v in wl["weights"].items()}
    x = round_to_dtype(wl["x"], dtype)
    block = rpp.SwinBlock(cfg, w)
    err = rpp.new_error_word()
    y = rpp.swin_block_forward(block, up(x.reshape(-1, c.C), dtype), c.B, err=err)
    check_err(err)
    got = down(y).reshape(c.B, c.I * c.I, c.C)
    for b in (0, 6, c.B - 1):
        ref = oracle.swin_block(x[b:b + 1], w, c.I, c.w, c.s, c.nh, c.eps)
        assert_close(got[b:b + 1], ref, dtype, f"swin block {dtype} image {b} of {c.B}")


def test_swin_block_full_config_sampled_images():
    """The Swin-T stage-1 block (B=64, 56x56, C=96) at full size; images are independent, so the oracle
    checks three of them, the first and the last included."""
    wl = make_swin_workload(SWIN)
    c = wl["cfg"]
    cfg = rpp.swin_cfg(c.I, c.C, c.nh, c.w, c.s, c.F, c.eps, "fp16")
    block = rpp.SwinBlock(cfg, wl["weights"])
    err = rpp.new_error_word()
    y = rpp.swin_block_forward(block, up(wl["x"].reshape(-1, c.C), "fp16"), c.B, err=err)
    check_err(err)
    got = down(y).reshape(c.B, c.I * c.I, c.C)
    for b in (0, 17, c.B - 1):
        ref = oracle.swin_block(wl["x"][b:b + 1], wl["weights"], c.I, c.w, c.s, c.nh, c.eps)
        assert_close(got[b:b + 1], ref, "fp16", f"swin block image {b}")


@pytest.mark.parametrize("C,nh,I,s", [(192, 6, 28, 3), (384, 12, 14, 3), (768, 24, 7, 0)])
def test_swin_block_later_stages(C, nh, I, s):
    """Swin-T stages 2-4 (C = 192 / 384 / 768 at 28 / 14 / 7 tokens a side; the last stage's
    single window is unshifted) through the same kernels."""
    from dataclasses import replace
    wl = make_swin_workload(replace(SWIN, C=C, nh=nh), B=1, I=I, s=s, affine=True)
    c = wl["cfg"]
    cfg = rpp.swin_cfg(c.I, c.C, c.nh, c.w, c.s, c.F, c.eps, "fp16")
    block = rpp.SwinBlock(cfg, wl["weights"])
    err = rpp.new_error_word()
    y = rpp.swin_block_forward(block, up(wl["x"].reshape(-1, c.C), "fp16"), c.B, err=err)
    check_err(err)
    ref = oracle.swin_block(wl["x"], wl["weights"], c.I, c.w, c.s, c.nh, c.eps)
    assert_close(down(y).reshape(ref.shape), ref, "fp16", f"swin stage C={C}")


@pytest.mark.parametrize("I,C,dtype,B", [(56, 96, "fp16", 3), (28, 192, "bf16", 2), (14, 384, "fp16", 2),
                                         (8, 768, "fp16", 1), (4, 8, "fp16", 2)])
def test_patch_merge(I, C, dtype, B):
    """At C = 768 (K = 3072) the outputs have magnitude ~1, where the bf16 output rounding
    alone averages ~2e-3 (a quarter of a bf16 step), the mean-abs bound itself; that
    size runs in fp16."""
    rng = np.random.default_rng(I + C)
    x = round_to_dtype(rng.standard_normal((B, I * I, C), dtype=np.float32), dtype)
    gamma = round_to_dtype(1 + 0.1 * rng.standard_normal(4 * C, dtype=np.float32), dtype)
    beta = round_to_dtype(0.1 * rng.standard_normal(4 * C, dtype=np.float32), dtype)
    W = round_to_dtype(0.02 * rng.standard_normal((4 * C, 2 * C), dtype=np.float32), dtype)
    pm = rpp.PatchMerge(rpp.merge_cfg(I, C, 1e-5, dtype), gamma, beta, W)
    err = rpp.new_error_word()
    y = rpp.patch_merge_forward(pm, up(x.reshape(-1, C), dtype), B, err=err)
    check_err(err)
    ref = oracle.patch_merge(x, I, gamma, beta, W, 1e-5)
    assert_close(down(y).reshape(ref.shape), ref, dtype, f"patch merge I={I} C={C}")
