"""Seeded synthetic workloads shared by the CUDA path's tests/bench and the CPU oracle.

This module holds only the configurations and the random draws: no step of the
encoder-layer arithmetic lives here, so the oracle and the CUDA path stay
independent of each other and meet only on identical inputs.

Every draw happens in fp32 on the host from ``numpy.random.Generator(PCG64(seed))``
and is rounded once (round-to-nearest-even) to the configuration's storage dtype.
Arrays are returned as float32 holding exactly the rounded values, so both sides
consume bit-identical inputs.

Draw order (fixed; changing it changes every workload):
  BERT-shaped:  lengths, padded input [B, L, H] (pad slots hold random junk), then
                per layer Wqkv [H, 3H], bqkv [3H], Wo [H, H], bo [H], W1 [H, F], b1 [F],
                W2 [F, H], b2 [H].  gamma = 1, beta = 0 unless ``affine`` is requested,
                in which case gamma1, beta1, gamma2, beta2 follow b2.
  Swin-shaped:  input [B, I*I, C], Wqkv [C, 3C], bqkv, relative-position table
                [(2w-1)^2, nh], Wo, bo, W1, b1, W2, b2 (then optional affine LN params).
Weights are stored [in, out] (y = x @ W + b).  The int8 calibration batch of a
configuration uses seed + 500.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

__all__ = [
    "EncoderConfig", "SwinConfig", "CONFIGS", "config_by_name",
    "round_to_dtype", "draw_lengths", "make_bert_workload", "make_swin_workload",
    "make_calibration_batch", "make_patch_merge_workload",
]


@dataclass(frozen=True)
class EncoderConfig:
    """A BERT-shaped (post-LayerNorm) encoder configuration."""
    name: str
    dtype: str                      # "fp32" | "fp16" | "bf16" | "int8" (int8 GEMMs, fp16 elsewhere)
    B: int
    L: int
    H: int
    nh: int
    F: int
    layers: int = 1
    eps: float = 1e-12
    len_lo: int = 1
    len_hi: int = 0                 # 0 -> L
    bimodal: Optional[tuple] = None  # ((lo1, hi1), (lo2, hi2)): half of the batch from each range
    bias_std: float = 0.02
    weight_std: float = 0.02
    seed: int = 1000
    kind: str = "bert"

    @property
    def d(self) -> int:
        return self.H // self.nh

    @property
    def storage_dtype(self) -> str:
        """dtype of activations and float weights in HBM (int8 configs keep fp16 there)."""
        return "fp16" if self.dtype == "int8" else self.dtype


@dataclass(frozen=True)
class SwinConfig:
    """A Swin-T-stage-shaped (pre-LayerNorm, shifted-window) block configuration."""
    name: str
    dtype: str
    B: int
    I: int                          # image side in tokens
    C: int
    nh: int
    w: int                          # window side
    s: int                          # cyclic shift
    mlp_ratio: int = 4
    eps: float = 1e-5
    weight_std: float = 0.02
    bias_std: float = 0.02
    table_std: float = 0.02
    seed: int = 1004
    kind: str = "swin"

    @property
    def d(self) -> int:
        return self.C // self.nh

    @property
    def F(self) -> int:
        return self.C * self.mlp_ratio

    @property
    def T(self) -> int:
        return self.B * self.I * self.I

    @property
    def storage_dtype(self) -> str:
        return self.dtype


CONFIGS = [
    EncoderConfig("tiny_fp32", "fp32", B=4, L=64, H=256, nh=4, F=1024, eps=1e-12,
                  len_lo=8, len_hi=64, bias_std=0.01, seed=1000),
    EncoderConfig("bert_base_fp16", "fp16", B=32, L=128, H=768, nh=12, F=3072,
                  len_lo=16, len_hi=128, seed=1001),
    EncoderConfig("bert_large_bf16_x24", "bf16", B=64, L=384, H=1024, nh=16, F=4096,
                  layers=24, bimodal=((32, 128), (256, 384)), seed=1002),
    EncoderConfig("bert_large_int8", "int8", B=64, L=256, H=1024, nh=16, F=4096,
                  len_lo=64, len_hi=256, seed=1003),
    SwinConfig("swin_t_stage1_fp16", "fp16", B=64, I=56, C=96, nh=3, w=7, s=3, seed=1004),
]


def config_by_name(name: str):
    for c in CONFIGS:
        if c.name == name:
            return c
    raise KeyError(name)


def round_to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 data once, RNE, to the storage dtype; return float32 holding the result."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "fp32":
        return x.copy()
    if dtype in ("fp16", "int8"):
        return x.astype(np.float16).astype(np.float32)
    if dtype == "bf16":
        u = x.view(np.uint32).astype(np.uint64)
        # round-to-nearest-even on the low 16 bits (inputs here are finite)
        lsb = (u >> 16) & 1
        u = (u + 0x7FFF + lsb) & 0xFFFF0000
        return u.astype(np.uint32).view(np.float32)
    raise ValueError(dtype)


def draw_lengths(cfg: EncoderConfig, rng: np.random.Generator) -> np.ndarray:
    """Per-sequence valid lengths, int32[B]."""
    if cfg.bimodal is not None:
        (a1, b1), (a2, b2) = cfg.bimodal
        half = cfg.B // 2
        short = rng.integers(a1, b1 + 1, size=half)
        long_ = rng.integers(a2, b2 + 1, size=cfg.B - half)
        lens = np.concatenate([short, long_])
        lens = lens[rng.permutation(cfg.B)]
    else:
        hi = cfg.len_hi if cfg.len_hi else cfg.L
        lens = rng.integers(cfg.len_lo, hi + 1, size=cfg.B)
    return lens.astype(np.int32)


def _normal(rng, shape, std, dtype):
    return round_to_dtype(rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std), dtype)


def _draw_layer(rng, H, F, cfg, dtype, affine):
    w = cfg.weight_std
    b = cfg.bias_std
    layer = {
        "Wqkv": _normal(rng, (H, 3 * H), w, dtype),
        "bqkv": _normal(rng, (3 * H,), b, dtype),
        "Wo": _normal(rng, (H, H), w, dtype),
        "bo": _normal(rng, (H,), b, dtype),
        "W1": _normal(rng, (H, F), w, dtype),
        "b1": _normal(rng, (F,), b, dtype),
        "W2": _normal(rng, (F, H), w, dtype),
        "b2": _normal(rng, (H,), b, dtype),
    }
    if affine:
        layer["gamma1"] = round_to_dtype(1.0 + 0.1 * rng.standard_normal(H, dtype=np.float32), dtype)
        layer["beta1"] = _normal(rng, (H,), 0.1, dtype)
        layer["gamma2"] = round_to_dtype(1.0 + 0.1 * rng.standard_normal(H, dtype=np.float32), dtype)
        layer["beta2"] = _normal(rng, (H,), 0.1, dtype)
    else:
        layer["gamma1"] = np.ones(H, np.float32)
        layer["beta1"] = np.zeros(H, np.float32)
        layer["gamma2"] = np.ones(H, np.float32)
        layer["beta2"] = np.zeros(H, np.float32)
    return layer


def make_bert_workload(cfg: EncoderConfig, *, seed: Optional[int] = None, B: Optional[int] = None,
                       L: Optional[int] = None, layers: Optional[int] = None,
                       lengths: Optional[np.ndarray] = None, affine: bool = False) -> dict:
    """Seeded BERT-shaped workload.

    Returns dict(cfg, lengths int32[B], x_padded float32[B, L, H], layers=[dict...]).
    ``B``, ``L``, ``layers`` override the configuration (small parity cases);
    ``lengths`` overrides the drawn lengths (edge cases) but the draw still happens
    so the remaining stream is unchanged.
    """
    if B is not None or L is not None or layers is not None:
        cfg = replace(cfg, B=B or cfg.B, L=L or cfg.L, layers=layers or cfg.layers,
                      len_hi=min(cfg.len_hi or cfg.L, L or cfg.L),
                      len_lo=min(cfg.len_lo, L or cfg.L),
                      bimodal=None if (L is not None and cfg.bimodal is not None) else cfg.bimodal)
    rng = np.random.Generator(np.random.PCG64(cfg.seed if seed is None else seed))
    lens = draw_lengths(cfg, rng)
    if lengths is not None:
        lens = np.asarray(lengths, dtype=np.int32).copy()
        assert lens.shape == (cfg.B,)
    dt = cfg.storage_dtype
    x = _normal(rng, (cfg.B, cfg.L, cfg.H), 1.0, dt)
    layers_ = [_draw_layer(rng, cfg.H, cfg.F, cfg, dt, affine) for _ in range(cfg.layers)]
    return {"cfg": cfg, "lengths": lens, "x_padded": x, "layers": layers_}


def make_calibration_batch(cfg: EncoderConfig) -> dict:
    """The int8 calibration batch: same shape, seed + 500, inputs only (weights are the model's)."""
    rng = np.random.Generator(np.random.PCG64(cfg.seed + 500))
    lens = draw_lengths(cfg, rng)
    x = _normal(rng, (cfg.B, cfg.L, cfg.H), 1.0, cfg.storage_dtype)
    return {"lengths": lens, "x_padded": x}


def make_swin_workload(cfg: SwinConfig, *, seed: Optional[int] = None, B: Optional[int] = None,
                       I: Optional[int] = None, s: Optional[int] = None, affine: bool = False) -> dict:
    """Seeded Swin-block workload: dict(cfg, x [B, I*I, C], weights dict)."""
    if B is not None or I is not None or s is not None:
        cfg = replace(cfg, B=B or cfg.B, I=I or cfg.I, s=cfg.s if s is None else s)
    rng = np.random.Generator(np.random.PCG64(cfg.seed if seed is None else seed))
    dt = cfg.storage_dtype
    C, F, nh, w = cfg.C, cfg.F, cfg.nh, cfg.w
    x = _normal(rng, (cfg.B, cfg.I * cfg.I, C), 1.0, dt)
    wt = {
        "Wqkv": _normal(rng, (C, 3 * C), cfg.weight_std, dt),
        "bqkv": _normal(rng, (3 * C,), cfg.bias_std, dt),
        "table": _normal(rng, ((2 * w - 1) ** 2, nh), cfg.table_std, dt),
        "Wo": _normal(rng, (C, C), cfg.weight_std, dt),
        "bo": _normal(rng, (C,), cfg.bias_std, dt),
        "W1": _normal(rng, (C, F), cfg.weight_std, dt),
        "b1": _normal(rng, (F,), cfg.bias_std, dt),
        "W2": _normal(rng, (F, C), cfg.weight_std, dt),
        "b2": _normal(rng, (C,), cfg.bias_std, dt),
    }
    if affine:
        for k in ("1", "2"):
            wt["gamma" + k] = round_to_dtype(1.0 + 0.1 * rng.standard_normal(C, dtype=np.float32), dt)
            wt["beta" + k] = _normal(rng, (C,), 0.1, dt)
    else:
        for k in ("1", "2"):
            wt["gamma" + k] = np.ones(C, np.float32)
            wt["beta" + k] = np.zeros(C, np.float32)
    return {"cfg": cfg, "x": x, "weights": wt}


def make_patch_merge_workload(cfg: SwinConfig, *, seed: Optional[int] = None, B: Optional[int] = None,
                              I: Optional[int] = None) -> dict:
    """Seeded input and weights of the stage downsampling after a Swin stage of `cfg`'s
    shape (seed + 300 unless given): dict(cfg, x [B, I*I, C], gamma [4C], beta [4C],
    W [4C, 2C]).  Draw order: x, gamma, beta, W."""
    if B is not None or I is not None:
        cfg = replace(cfg, B=B or cfg.B, I=I or cfg.I)
    rng = np.random.default_rng(np.random.PCG64(cfg.seed + 300 if seed is None else seed))
    dt = cfg.storage_dtype
    C = cfg.C
    x = _normal(rng, (cfg.B, cfg.I * cfg.I, C), 1.0, dt)
    gamma = round_to_dtype(1.0 + 0.1 * rng.standard_normal(4 * C, dtype=np.float32), dt)
    beta = _normal(rng, (4 * C,), 0.1, dt)
    W = _normal(rng, (4 * C, 2 * C), cfg.weight_std, dt)
    return {"cfg": cfg, "x": x, "gamma": gamma, "beta": beta, "W": W}
