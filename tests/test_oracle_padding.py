"""Pins for the oracle's offset mask, padding removal and rebuild.

What fixes these functions ('GPU底層優化 | 如何讓Transformer在GPU上跑得更快？' Fig. 9): the
padded and the packed forms convert into each other exactly.  The pins below check a
hand-worked example, a brute-force derivation from the boolean validity mask (a
different route from the prefix sum), the round-trip identities and special cases.
"""
import json
import os

import numpy as np
import pytest

import oracle
from workloads import CONFIGS, make_bert_workload, draw_lengths, config_by_name

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_offsets_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "offsets_small.json")))
    cu, po, T = oracle.build_offsets(g["lengths"], g["L"])
    assert cu.tolist() == g["cu_seqlens"]
    assert po.tolist() == g["padding_offset"]
    assert T == g["T"]


def _offsets_from_mask(lengths, L):
    # brute force: enumerate padded slots in order, keep the valid ones
    valid = np.arange(L)[None, :] < np.asarray(lengths)[:, None]
    flat = np.nonzero(valid.reshape(-1))[0]
    return flat - np.arange(len(flat))


@pytest.mark.parametrize("seed", range(20))
def test_offsets_match_mask_enumeration(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 70))
    L = int(rng.integers(1, 400))
    lengths = rng.integers(0, L + 1, size=B)
    cu, po, T = oracle.build_offsets(lengths, L)
    assert T == int(np.sum(lengths))
    assert cu[0] == 0 and np.all(np.diff(cu) == lengths)
    assert np.array_equal(po, _offsets_from_mask(lengths, L))


def test_offsets_special_cases():
    cu, po, T = oracle.build_offsets([7, 7, 7], 7)          # no padding at all
    assert T == 21 and np.all(po == 0)
    cu, po, T = oracle.build_offsets([0, 0], 5)             # everything is padding
    assert T == 0 and cu.tolist() == [0, 0, 0] and len(po) == 0
    cu, po, T = oracle.build_offsets([1, 1, 1], 4)          # one token per sequence
    assert po.tolist() == [0, 3, 6]
    with pytest.raises(ValueError):
        oracle.build_offsets([3, 9], 8)
    with pytest.raises(ValueError):
        oracle.build_offsets([-1], 8)


@pytest.mark.parametrize("cfg", [c for c in CONFIGS if c.kind == "bert"], ids=lambda c: c.name)
def test_lengths_of_configs_are_in_range(cfg):
    rng = np.random.Generator(np.random.PCG64(cfg.seed))
    lens = draw_lengths(cfg, rng)
    assert lens.min() >= 1 and lens.max() <= cfg.L
    cu, po, T = oracle.build_offsets(lens, cfg.L)
    assert np.array_equal(po, _offsets_from_mask(lens, cfg.L))


def test_remove_rebuild_round_trips():
    rng = np.random.default_rng(3)
    B, L, H = 5, 9, 6
    lengths = np.array([9, 0, 4, 1, 7])
    x = rng.standard_normal((B, L, H))
    valid = np.arange(L)[None, :] < lengths[:, None]
    x_pad_nan = x.copy()
    x_pad_nan[~valid] = np.nan                      # junk in the pad slots must never be read
    cu, po, T = oracle.build_offsets(lengths, L)
    packed = oracle.remove_padding(x_pad_nan, po)
    assert packed.shape == (T, H) and np.isfinite(packed).all()
    # packed order = the valid rows in padded order
    assert np.array_equal(packed, x[valid])
    rebuilt = oracle.rebuild_padding(packed, cu, B, L)
    expect = np.where(valid[..., None], x, 0.0)
    assert np.array_equal(rebuilt, expect)          # rebuild . remove = identity on valid, 0 on pads
    assert np.array_equal(oracle.remove_padding(rebuilt, po), packed)   # remove . rebuild = identity


def test_remove_padding_on_a_config_workload():
    wl = make_bert_workload(config_by_name("tiny_fp32"))
    cfg = wl["cfg"]
    cu, po, T = oracle.build_offsets(wl["lengths"], cfg.L)
    packed = oracle.remove_padding(wl["x_padded"], po)
    for b in range(cfg.B):
        n = wl["lengths"][b]
        assert np.array_equal(packed[cu[b]:cu[b] + n], wl["x_padded"][b, :n])
