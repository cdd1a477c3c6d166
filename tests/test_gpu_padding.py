"""GPU parity: offset builder, padding removal and rebuild -- bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import remove_padding_prefix_gb300 as rpp
from workloads import CONFIGS, draw_lengths, make_bert_workload, config_by_name
from gpu_util import dev, up, check_err, TDT

pytestmark = pytest.mark.gpu
BERT = [c for c in CONFIGS if c.kind == "bert"]


def _offsets(lengths, L):
    lt = torch.as_tensor(np.asarray(lengths, np.int32), device=dev())
    err = rpp.new_error_word()
    cu, po = rpp.build_offsets(lt, L, err=err)
    return cu, po, err


@pytest.mark.parametrize("cfg", BERT, ids=lambda c: c.name)
def test_offsets_bit_exact_on_config_lengths(cfg):
    lens = draw_lengths(cfg, np.random.Generator(np.random.PCG64(cfg.seed)))
    cu, po, err = _offsets(lens, cfg.L)
    check_err(err)
    cu_ref, po_ref, T = oracle.build_offsets(lens, cfg.L)
    assert np.array_equal(cu.cpu().numpy(), cu_ref)
    assert np.array_equal(po.cpu().numpy()[:T], po_ref)


@pytest.mark.parametrize("lens,L", [([0], 5), ([0, 0, 0], 3), ([1] * 7, 1), ([3, 0, 5, 1], 5),
                                    (list(range(1, 1100)), 1100), ([384] * 64, 384)])
def test_offsets_edge_cases(lens, L):
    cu, po, err = _offsets(lens, L)
    check_err(err)
    cu_ref, po_ref, T = oracle.build_offsets(lens, L)
    assert np.array_equal(cu.cpu().numpy(), cu_ref)
    assert np.array_equal(po.cpu().numpy()[:T], po_ref)


def test_offsets_report_bad_length_and_stay_in_bounds():
    cu, po, err = _offsets([3, 9, 2], 8)
    assert rpp.get_device_error(err) == rpp.RPP_DERR_LENGTH
    # clamped to L, so later kernels stay in bounds
    assert cu.cpu().numpy().tolist() == [0, 3, 11, 13]
    cu, po, err = _offsets([3, -2, 2], 8)
    assert rpp.get_device_error(err) == rpp.RPP_DERR_LENGTH
    assert cu.cpu().numpy().tolist() == [0, 3, 3, 5]


@pytest.mark.parametrize("dtype,H", [("fp32", 256), ("fp16", 768), ("bf16", 1024), ("fp16", 96), ("bf16", 8)])
def test_remove_rebuild_bit_exact(dtype, H):
    rng = np.random.default_rng(H)
    B, L = 9, 37
    lens = rng.integers(0, L + 1, size=B).astype(np.int32)
    lens[0], lens[1] = L, 0
    x = rng.standard_normal((B, L, H)).astype(np.float32)
    xt = up(x.reshape(B * L, H), dtype)
    xr = xt.float().cpu().numpy().reshape(B, L, H)          # the exact values on the device
    cu, po, err = _offsets(lens, L)
    packed = rpp.remove_padding(xt, po, cu, B, L, err=err)
    padded = rpp.rebuild_padding(packed, cu, B, L, err=err)
    check_err(err)
    cu_ref, po_ref, T = oracle.build_offsets(lens, L)
    ref_packed = oracle.remove_padding(xr, po_ref)
    assert np.array_equal(packed[:T].float().cpu().numpy(), ref_packed)
    ref_padded = oracle.rebuild_padding(ref_packed, cu_ref, B, L)
    assert np.array_equal(padded.float().cpu().numpy().reshape(B, L, H), ref_padded)


def test_remove_padding_full_size_config():
    cfg = config_by_name("bert_large_bf16_x24")   # B=64, L=384, H=1024, bf16: the largest padded batch
    wl = make_bert_workload(cfg, layers=1)
    cu, po, err = _offsets(wl["lengths"], cfg.L)
    x = up(wl["x_padded"].reshape(-1, cfg.H), "bf16")
    packed = rpp.remove_padding(x, po, cu, cfg.B, cfg.L, err=err)
    back = rpp.rebuild_padding(packed, cu, cfg.B, cfg.L, err=err)
    check_err(err)
    cu_ref, po_ref, T = oracle.build_offsets(wl["lengths"], cfg.L)
    # sampled rows: the oracle's gather row by row
    rows = np.random.default_rng(0).integers(0, T, size=200)
    got = packed[torch.as_tensor(rows, device=dev())].float().cpu().numpy()
    flat = wl["x_padded"].reshape(-1, cfg.H)
    assert np.array_equal(got, flat[rows + po_ref[rows]])
    # property at full size: rebuild . remove keeps valid rows and zeroes pads
    valid = torch.as_tensor((np.arange(cfg.L)[None, :] < wl["lengths"][:, None]).reshape(-1), device=dev())
    assert torch.equal(back[valid], x[valid])
    assert not back[~valid].any()
