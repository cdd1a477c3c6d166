"""GPU parity of the whole encoder path (offsets -> remove padding -> layer(s) ->
rebuild padding) through the C ABI against the oracle.

Small cases span several tiles and ragged tails; the full-size configurations are
checked on sequences sampled from the real batch (per-sequence independence lets
the oracle run a sequence alone), at the sizes and launch configuration the bench
times."""
import numpy as np
import pytest
import torch

import oracle
import remove_padding_prefix_gb300 as rpp
from workloads import CONFIGS, make_bert_workload
from gpu_util import dev, up, down, assert_close, check_err, TOL

pytestmark = pytest.mark.gpu


def _run_path(wl, dtype, layers=None, hint=False, poison=None):
    """hint=True passes the true token count as the tile-shape hint (the bench's launch
    configuration: exact-size tiles and split-K with LayerNorm-side reduction).
    poison: a byte every workspace byte is set to before the call (the capacity past the
    token count is never written and must never reach a valid output)."""
    cfg = wl["cfg"]
    layers = layers if layers is not None else wl["layers"]
    T = int(wl["lengths"].sum())
    ecfg = rpp.encoder_cfg(cfg.H, cfg.nh, cfg.F, cfg.eps, dtype, tokens_hint=T if hint else 0)
    prepared = [rpp.EncoderLayer(ecfg, l) for l in layers]
    lengths = torch.as_tensor(wl["lengths"], device=dev())
    x = up(wl["x_padded"].reshape(-1, cfg.H), dtype)
    err = rpp.new_error_word()
    ws = None
    if poison is not None:
        ws = prepared[0].workspace(cfg.B * cfg.L, dev())
        ws.view(torch.uint8).fill_(poison)
    y, cu, po = rpp.encoder_forward(prepared, lengths, x, cfg.L, workspace=ws, err=err)
    check_err(err)
    # the fused offsets + removal of the whole-path call: offsets bit-exact
    cu_ref, po_ref, T = oracle.build_offsets(wl["lengths"], cfg.L)
    assert np.array_equal(cu.cpu().numpy(), cu_ref)
    assert np.array_equal(po.cpu().numpy()[:T], po_ref)
    return down(y).reshape(cfg.B, cfg.L, cfg.H), prepared


@pytest.mark.parametrize("hint", [False, True])
@pytest.mark.parametrize("idx,B,L,lens", [
    (0, 4, 64, None),                                  # tiny fp32 config as drawn
    (1, 6, 128, [128, 1, 17, 64, 65, 100]),           # BERT-base shapes, fp16
    (2, 3, 384, [384, 129, 33]),                       # BERT-large shapes, bf16
])
def test_layer_small(idx, B, L, lens, hint):
    cfg = CONFIGS[idx]
    wl = make_bert_workload(cfg, B=B, L=L, layers=1, lengths=None if lens is None else np.array(lens, np.int32),
                            affine=True)
    got, _ = _run_path(wl, cfg.dtype, hint=hint)
    ref, _, _ = oracle.bert_forward(wl["x_padded"], wl["lengths"], wl["layers"], cfg.nh, cfg.eps)
    assert_close(got, ref, cfg.dtype, cfg.name)


@pytest.mark.parametrize("hint", [False, True])
@pytest.mark.parametrize("idx,lens", [(1, [128, 1, 17, 64, 65, 100]), (2, [384, 129, 33])])
def test_layer_poisoned_workspace(idx, lens, hint):
    """Workspace bytes 0x47 (7.3 in fp16, 5.1e4 in bf16 and fp32) before the call: the
    unwritten capacity rows past the token count feed the attention's out-of-sequence
    query rows large values; the valid outputs match the oracle all the same."""
    cfg = CONFIGS[idx]
    wl = make_bert_workload(cfg, B=len(lens), L=max(lens) if idx == 1 else 384, layers=1,
                            lengths=np.array(lens, np.int32), affine=True)
    got, _ = _run_path(wl, cfg.dtype, hint=hint, poison=0x47)
    ref, _, _ = oracle.bert_forward(wl["x_padded"], wl["lengths"], wl["layers"], cfg.nh, cfg.eps)
    assert_close(got, ref, cfg.dtype, f"{cfg.name} poisoned workspace")


@pytest.mark.parametrize("mode", [1, 2])
def test_layer_gemm_cluster_modes(mode):
    """The BERT-base layer with its GEMMs unpaired and always paired into clusters."""
    cfg = CONFIGS[1]
    wl = make_bert_workload(cfg, B=6, L=128, layers=1, lengths=np.array([128, 1, 17, 64, 65, 100], np.int32),
                            affine=True)
    assert rpp.lib().rpp_set_gemm_cluster_mode(mode) == 0
    try:
        got, _ = _run_path(wl, cfg.dtype, hint=True)
    finally:
        rpp.lib().rpp_set_gemm_cluster_mode(0)
    ref, _, _ = oracle.bert_forward(wl["x_padded"], wl["lengths"], wl["layers"], cfg.nh, cfg.eps)
    assert_close(got, ref, cfg.dtype, f"{cfg.name} cluster mode {mode}")


def test_layer_all_lengths_zero_gives_zero_output():
    cfg = CONFIGS[1]
    wl = make_bert_workload(cfg, B=3, L=16, layers=1, lengths=np.zeros(3, np.int32))
    got, _ = _run_path(wl, "fp16")
    assert np.all(got == 0)


def test_bert_base_full_config():
    """The BERT-base-shaped fp16 layer (B=32, L=128) at full size (the bench workload), every
    output against the oracle."""
    cfg = CONFIGS[1]
    wl = make_bert_workload(cfg)
    ref, _, _ = oracle.bert_forward(wl["x_padded"], wl["lengths"], wl["layers"], cfg.nh, cfg.eps)
    for hint in (True, False):
        got, _ = _run_path(wl, "fp16", hint=hint)
        assert_close(got, ref, "fp16", f"{cfg.name} hint={hint}")


def test_tiny_fp32_full_config():
    cfg = CONFIGS[0]
    wl = make_bert_workload(cfg)
    got, _ = _run_path(wl, "fp32")
    ref, _, _ = oracle.bert_forward(wl["x_padded"], wl["lengths"], wl["layers"], cfg.nh, cfg.eps)
    assert_close(got, ref, "fp32", cfg.name)


def _teacher_forced_stack(wl, dtype, n_layers, sample):
    """Run each layer on the GPU and check it against the oracle applied to the exact
    (rounded) input the GPU layer saw, on sampled sequences."""
    cfg = wl["cfg"]
    ecfg = rpp.encoder_cfg(cfg.H, cfg.nh, cfg.F, cfg.eps, dtype, tokens_hint=int(wl["lengths"].sum()))
    lengths = torch.as_tensor(wl["lengths"], device=dev())
    err = rpp.new_error_word()
    cu, po = rpp.build_offsets(lengths, cfg.L, err=err)
    x = rpp.remove_padding(up(wl["x_padded"].reshape(-1, cfg.H), dtype), po, cu, cfg.B, cfg.L, err=err)
    ws = None
    cu_h = cu.cpu().numpy()
    worst = (0.0, 0.0)
    for i in range(n_layers):
        layer = rpp.EncoderLayer(ecfg, wl["layers"][i])
        ws = ws if ws is not None else layer.workspace(x.shape[0])
        x_in = x.clone()
        rpp.encoder_layer_forward(layer, x, cu, cfg.B, cfg.L, y=x, workspace=ws, err=err)
        check_err(err)
        xin_h = down(x_in)
        y_h = down(x)
        for b in sample:
            lo, hi = cu_h[b], cu_h[b + 1]
            ref = oracle.bert_layer(xin_h[lo:hi], np.array([0, hi - lo]), wl["layers"][i], cfg.nh, cfg.eps)
            m = assert_close(y_h[lo:hi], ref, dtype, f"{cfg.name} layer {i} seq {b}")
            worst = (max(worst[0], m[0]), max(worst[1], m[1]))
        del layer
    return x, worst


def test_bert_large_stack_sampled_sequences():
    """The BERT-large-shaped bf16 stack (B=64, L=384): 24 layers at full size; each layer
    checked (teacher-forced) on four sequences, longest and shortest included."""
    cfg = CONFIGS[2]
    wl = make_bert_workload(cfg)
    lens = wl["lengths"]
    sample = sorted({int(np.argmax(lens)), int(np.argmin(lens)), 5, 40})
    _teacher_forced_stack(wl, "bf16", cfg.layers, sample)


def test_bert_large_stack_end_to_end_drift_bounded():
    """The 24-layer bf16 stack end to end vs the fp64 oracle on one sequence: errors
    compound through 24 roundings of every intermediate, so this uses a looser bound
    (max-abs 0.25, mean-abs 2e-2) than the per-layer tolerance."""
    cfg = CONFIGS[2]
    wl = make_bert_workload(cfg)
    got, _ = _run_path(wl, "bf16")
    b = int(np.argmin(wl["lengths"]))
    n = int(wl["lengths"][b])
    ref = oracle.bert_stack_packed(wl["x_padded"][b, :n].astype(np.float64), np.array([0, n]), wl["layers"],
                                   cfg.nh, cfg.eps)
    d = np.abs(got[b, :n] - ref)
    assert d.max() < 0.25 and d.mean() < 2e-2, (d.max(), d.mean())
