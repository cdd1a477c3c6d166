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
from workloads import make_bert_workload, round_to_dtype, config_by_name
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
@pytest.mark.parametrize("name,B,L,lens", [
    ("tiny_fp32", 4, 64, None),                                  # tiny fp32 config as drawn
    ("bert_base_fp16", 6, 128, [128, 1, 17, 64, 65, 100]),           # BERT-base shapes, fp16
    ("bert_large_bf16_x24", 3, 384, [384, 129, 33]),                       # BERT-large shapes, bf16
])
def test_layer_small(name, B, L, lens, hint):
    cfg = config_by_name(name)
    wl = make_bert_workload(cfg, B=B, L=L, layers=1, lengths=None if lens is None else np.array(lens, np.int32),
                            affine=True)
    got, _ = _run_path(wl, cfg.dtype, hint=hint)
    ref, _, _ = oracle.bert_forward(wl["x_padded"], wl["lengths"], wl["layers"], cfg.nh, cfg.eps)
    assert_close(got, ref, cfg.dtype, cfg.name)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_layer_hidden_not_multiple_of_256(dtype):
    """H = 384 (six heads of 64): a hidden size that is not a multiple of the widest GEMM
    tile, so proj and FC2 (bias + residual epilogue, fp16 pre-LayerNorm sums) take
    narrower column tiles than the BERT shapes."""
    from dataclasses import replace
    cfg = replace(config_by_name("bert_large_bf16_x24"), H=384, nh=6, F=1536, dtype=dtype, layers=1)
    wl = make_bert_workload(cfg, B=4, L=200, lengths=np.array([200, 3, 77, 130], np.int32), affine=True)
    for hint in (False, True):
        got, _ = _run_path(wl, dtype, hint=hint)
        ref, _, _ = oracle.bert_forward(wl["x_padded"], wl["lengths"], wl["layers"], cfg.nh, cfg.eps)
        assert_close(got, ref, dtype, f"H=384 {dtype} hint={hint}")


@pytest.mark.parametrize("hint", [False, True])
@pytest.mark.parametrize("name,lens", [("bert_base_fp16", [128, 1, 17, 64, 65, 100]),
                                       ("bert_large_bf16_x24", [384, 129, 33])])
def test_layer_poisoned_workspace(name, lens, hint):
    """Workspace bytes 0x47 (7.3 in fp16, 5.1e4 in bf16 and fp32) before the call: the
    unwritten capacity rows past the token count feed the attention's out-of-sequence
    query rows large values; the valid outputs match the oracle all the same."""
    cfg = config_by_name(name)
    wl = make_bert_workload(cfg, B=len(lens), L=max(lens) if name == "bert_base_fp16" else 384, layers=1,
                            lengths=np.array(lens, np.int32), affine=True)
    got, _ = _run_path(wl, cfg.dtype, hint=hint, poison=0x47)
    ref, _, _ = oracle.bert_forward(wl["x_padded"], wl["lengths"], wl["layers"], cfg.nh, cfg.eps)
    assert_close(got, ref, cfg.dtype, f"{cfg.name} poisoned workspace")


@pytest.mark.parametrize("mode", [1, 2])
def test_layer_gemm_cluster_modes(mode):
    """The BERT-base layer with its GEMMs unpaired and always paired into clusters."""
    cfg = config_by_name("bert_base_fp16")
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
    cfg = config_by_name("bert_base_fp16")
    wl = make_bert_workload(cfg, B=3, L=16, layers=1, lengths=np.zeros(3, np.int32))
    got, _ = _run_path(wl, "fp16")
    assert np.all(got == 0)


def test_bert_base_full_config():
    """The BERT-base-shaped fp16 layer (B=32, L=128) at full size (the bench workload), every
    output against the oracle."""
    cfg = config_by_name("bert_base_fp16")
    wl = make_bert_workload(cfg)
    ref, _, _ = oracle.bert_forward(wl["x_padded"], wl["lengths"], wl["layers"], cfg.nh, cfg.eps)
    for hint in (True, False):
        got, _ = _run_path(wl, "fp16", hint=hint)
        assert_close(got, ref, "fp16", f"{cfg.name} hint={hint}")


def test_tiny_fp32_full_config():
    cfg = config_by_name("tiny_fp32")
    wl = make_bert_workload(cfg)
    got, _ = _run_path(wl, "fp32")
    ref, _, _ = oracle.bert_forward(wl["x_padded"], wl["lengths"], wl["layers"], cfg.nh, cfg.eps)
    assert_close(got, ref, "fp32", cfg.name)


def _layer_gain(x, cu, layer, nh, eps, rel, seed):
    """How much one layer of the oracle amplifies a small input perturbation: eta =
    x * rel * U(-1, 1) (the size of a rounding error), returns the ratios of the output
    change to eta in max-abs and in mean-abs."""
    rng = np.random.default_rng(seed)
    eta = x * rel * rng.uniform(-1.0, 1.0, size=x.shape)
    y0 = oracle.bert_layer(x, cu, layer, nh, eps)
    y1 = oracle.bert_layer(x + eta, cu, layer, nh, eps)
    d = np.abs(y1 - y0)
    return d.max() / np.abs(eta).max(), d.mean() / np.abs(eta).mean()


def test_bert_large_stack_all_sequences():
    """The BERT-large-shaped bf16 stack (B=64, L=384, 24 layers) at full size, every
    sequence of the batch.

    Per layer: the GPU layer against the oracle run on the exact bf16 input that GPU
    layer saw (teacher forced), at the stated tolerance, max-abs 2e-2 / mean-abs 2e-3.

    End to end: the chained GPU stack against the oracle's own 24-layer chain from the
    same input.  Its bound is derived, not picked: with delta_l the per-layer error just
    measured and G_l the oracle layer's measured gain on a perturbation of rounding
    size (max-abs and mean-abs ratios), a first-order bound on the final error is
    E = sum_l delta_l * prod_{k > l} G_k, taken separately for max-abs and mean-abs;
    the test allows 1.25 E for the terms beyond first order."""
    cfg = config_by_name("bert_large_bf16_x24")
    wl = make_bert_workload(cfg)
    dtype = "bf16"
    ecfg = rpp.encoder_cfg(cfg.H, cfg.nh, cfg.F, cfg.eps, dtype, tokens_hint=int(wl["lengths"].sum()))
    lengths = torch.as_tensor(wl["lengths"], device=dev())
    err = rpp.new_error_word()
    cu, po = rpp.build_offsets(lengths, cfg.L, err=err)
    x = rpp.remove_padding(up(wl["x_padded"].reshape(-1, cfg.H), dtype), po, cu, cfg.B, cfg.L, err=err)
    cu_h = cu.cpu().numpy()
    T = int(cu_h[-1])
    x0 = down(x)[:T]
    ws = None
    deltas, gains = [], []
    for i in range(cfg.layers):
        layer = rpp.EncoderLayer(ecfg, wl["layers"][i])
        ws = ws if ws is not None else layer.workspace(x.shape[0])
        xin = down(x)[:T]
        rpp.encoder_layer_forward(layer, x, cu, cfg.B, cfg.L, y=x, workspace=ws, err=err)
        check_err(err)
        ref = oracle.bert_layer(xin, cu_h, wl["layers"][i], cfg.nh, cfg.eps)
        deltas.append(assert_close(down(x)[:T], ref, dtype, f"{cfg.name} layer {i}, all sequences"))
        # gain measured on eight sequences (a rounding-size perturbation of the GPU's input)
        lo, hi = cu_h[0], cu_h[8]
        gains.append(_layer_gain(xin[lo:hi], cu_h[:9] - lo, wl["layers"][i], cfg.nh, cfg.eps, 2.0 ** -9, i))
        del layer
    got = down(x)[:T]
    ref = oracle.bert_stack_packed(x0, cu_h, wl["layers"], cfg.nh, cfg.eps)
    d = np.abs(got - ref)
    bound = [0.0, 0.0]
    for j in (0, 1):
        for l in range(cfg.layers):
            bound[j] += deltas[l][j] * float(np.prod([gains[k][j] for k in range(l + 1, cfg.layers)]))
    print(f"24-layer bf16 stack: end-to-end max-abs {d.max():.3e} mean-abs {d.mean():.3e}; derived bound "
          f"{bound[0]:.3e} / {bound[1]:.3e}; per-layer delta max {max(t[0] for t in deltas):.3e} "
          f"mean {max(t[1] for t in deltas):.3e}; gains max {max(g[0] for g in gains):.3f} "
          f"mean {max(g[1] for g in gains):.3f}")
    assert d.max() <= 1.25 * bound[0] and d.mean() <= 1.25 * bound[1], (d.max(), d.mean(), bound)


def test_captured_graph_replays_with_new_lengths():
    """One CUDA graph of the whole path (offsets, removal, two BERT-base-shaped fp16
    layers, rebuild) captured once and replayed with new lengths and new inputs written
    into the captured buffers: the token count lives in device memory, so every replay
    must match the oracle for its own lengths, with zero pad slots."""
    cfg = config_by_name("bert_base_fp16")
    B, L = 6, 128
    wl = make_bert_workload(cfg, B=B, L=L, layers=2, affine=True)
    ecfg = rpp.encoder_cfg(cfg.H, cfg.nh, cfg.F, cfg.eps, "fp16", tokens_hint=B * L // 2)
    prepared = [rpp.EncoderLayer(ecfg, l) for l in wl["layers"]]
    lengths = torch.as_tensor(wl["lengths"], device=dev())
    x = up(wl["x_padded"].reshape(-1, cfg.H), "fp16")
    y = torch.empty_like(x)
    cu = torch.empty(B + 1, dtype=torch.int32, device=dev())
    po = torch.zeros(B * L, dtype=torch.int32, device=dev())
    packed = torch.empty_like(x)
    ws = prepared[0].workspace(B * L, dev())
    err = rpp.new_error_word()

    def step():
        rpp.encoder_forward(prepared, lengths, x, L, y_padded=y, cu_seqlens=cu, padding_offset=po, packed=packed,
                            workspace=ws, err=err)

    step()                                # eager warm-up (module load, attributes) before capture
    torch.cuda.synchronize()
    check_err(err)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    sets = [[128, 1, 17, 64, 65, 100], [0, 128, 128, 3, 0, 77], [5, 5, 5, 5, 5, 5], [128] * 6, [0] * 6]
    for i, lens in enumerate(sets):
        lens = np.array(lens, np.int32)
        xp = round_to_dtype(rng.standard_normal((B, L, cfg.H), dtype=np.float32), "fp16")
        lengths.copy_(torch.as_tensor(lens))
        x.copy_(up(xp.reshape(-1, cfg.H), "fp16"))
        y.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        check_err(err)
        got = down(y).reshape(B, L, cfg.H)
        ref, cu_ref, _ = oracle.bert_forward(xp, lens, wl["layers"], cfg.nh, cfg.eps)
        assert np.array_equal(cu.cpu().numpy(), cu_ref), f"replay {i}: cu_seqlens"
        assert_close(got, ref, "fp16", f"graph replay {i}, lengths {lens.tolist()}")
