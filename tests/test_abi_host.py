"""Host-side checks of the C ABI (no GPU needed).

The library loads and exports every entry point include/rpp.h declares; size
queries and argument validation are pure host logic and return without touching the
device.
"""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rpp.h")


@pytest.fixture(scope="module")
def lib():
    from remove_padding_prefix_gb300 import _abi, build
    if not os.path.exists(_abi.LIB_PATH):
        build.build()
    return _abi.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^RPP_API\s+[\w\s\*]+?\b(rpp_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for must in ("rpp_build_offsets", "rpp_remove_padding", "rpp_rebuild_padding", "rpp_encoder_layer_forward",
                 "rpp_window_attention_forward", "rpp_swin_block_forward", "rpp_gemm_i8_i32"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    from remove_padding_prefix_gb300 import _abi
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
        assert n in _abi.SIGNATURES, f"binding lacks {n}"
    assert set(_abi.SIGNATURES) == set(names)


def test_status_strings_and_version(lib):
    assert lib.rpp_status_string(0) == b"ok"
    assert lib.rpp_status_string(-4) == b"workspace too small"
    assert lib.rpp_version() >= 100


def test_argument_validation_returns_without_launching(lib):
    # null pointers and bad sizes are rejected on the host
    assert lib.rpp_build_offsets(None, 4, 8, None, None, None, None) == -1
    assert lib.rpp_remove_padding(None, None, None, 1, 1, 8, 1, None, None, None) == -1
    assert lib.rpp_rebuild_padding(None, None, 1, 1, 8, 1, None, None, None) == -1
    assert lib.rpp_linear(None, None, None, None, None, 1, None, 16, 16, 1, 0, None, None) == -1
    assert lib.rpp_attention_varlen(None, None, 1, 1, 1, 1, 64, 1, None, None, None) == -1
    assert lib.rpp_gemm_i8_i32(None, None, None, 1, 16, 16, None, 0, None, None) == -1
    # misaligned activation pointer (odd address) is rejected before any launch
    assert lib.rpp_remove_padding(1, 16, 16, 1, 1, 8, 1, 32, None, None) == -1
    # the exact int8 GEMM: K beyond four 1024-K chunks, or K / N off the 16 grid, is
    # unsupported (checked before the pointers are used; these never reach the device)
    unsupported = -2
    assert lib.rpp_gemm_i8_i32(256, 256, 256, 1, 16, 4112, 256, 1 << 30, None, None) == unsupported
    assert lib.rpp_gemm_i8_i32(256, 256, 256, 1, 16, 24, 256, 1 << 30, None, None) == unsupported
    assert lib.rpp_gemm_i8_i32(256, 256, 256, 1, 24, 16, 256, 1 << 30, None, None) == unsupported


def test_size_queries(lib):
    from remove_padding_prefix_gb300 import _abi
    cfg = _abi.EncoderCfg(768, 12, 64, 3072, 1e-12, _abi.RPP_F16, 0)
    wbytes = lib.rpp_layer_bytes(C.byref(cfg))
    H, F = 768, 3072
    assert wbytes >= (4 * H * H + 2 * H * F) * 2 + (3 * H + 2 * H + F + 4 * H) * 4
    ws = lib.rpp_encoder_workspace_bytes(C.byref(cfg), 4096)
    assert ws >= 4096 * (3 * H + 3 * H + F) * 2 + 4096 * H * 4
    cfg8 = _abi.EncoderCfg(1024, 16, 64, 4096, 1e-12, _abi.RPP_F16, 1)
    assert lib.rpp_encoder_workspace_bytes(C.byref(cfg8), 100) > lib.rpp_encoder_workspace_bytes(
        C.byref(_abi.EncoderCfg(1024, 16, 64, 4096, 1e-12, _abi.RPP_F16, 0)), 100)
    bad = _abi.EncoderCfg(768, 12, 60, 3072, 1e-12, _abi.RPP_F16, 0)   # heads * head_dim != hidden
    assert lib.rpp_layer_bytes(C.byref(bad)) == 0
    int8_bf16 = _abi.EncoderCfg(768, 12, 64, 3072, 1e-12, _abi.RPP_BF16, 1)   # int8 needs fp16 activations
    assert lib.rpp_layer_bytes(C.byref(int8_bf16)) == 0
    assert lib.rpp_gemm_i8_workspace_bytes(128, 64, 256) >= (128 + 64) * 256 * 2
    sw = _abi.SwinCfg(56, 96, 3, 7, 3, 384, 1e-5, _abi.RPP_F16)
    assert lib.rpp_swin_block_bytes(C.byref(sw)) > 0
    # C = 96 with MLP 384 runs the fused MLP, which keeps a second copy of W1 ([C, mlp], read
    # N-major); other widths hold the K-major copy only
    Cs, F = 96, 384
    kmajor = (3 * Cs * Cs + Cs * Cs + 2 * F * Cs) * 2
    assert lib.rpp_swin_block_bytes(C.byref(sw)) >= kmajor + F * Cs * 2
    sw192 = _abi.SwinCfg(28, 192, 6, 7, 3, 768, 1e-5, _abi.RPP_F16)
    b192 = lib.rpp_swin_block_bytes(C.byref(sw192))
    assert (3 * 192 * 192 + 192 * 192 + 2 * 768 * 192) * 2 <= b192 < (3 * 192 * 192 + 192 * 192 + 3 * 768 * 192) * 2
    assert lib.rpp_swin_workspace_bytes(C.byref(sw), 2) >= 2 * 56 * 56 * (96 * 5 + 384) * 2
    # workspace too small is reported before any launch
    assert lib.rpp_encoder_layer_forward(C.byref(cfg), 256, None, 256, 256, 4, 512, 128, 256, 256, 16, None,
                                         None) == -4


def test_tuning_and_profiling_knobs_validate_on_the_host(lib):
    assert lib.rpp_set_gemm_cluster_mode(3) == -1
    assert lib.rpp_set_gemm_cluster_mode(-1) == -1
    for m in (1, 2, 0):
        assert lib.rpp_set_gemm_cluster_mode(m) == 0
    assert lib.rpp_set_launch_event_filter(b"") == -1
    assert lib.rpp_set_launch_event_filter(b"x" * 64) == -1
    assert lib.rpp_set_launch_event_filter(b"gemm_fc1") == 0
    assert lib.rpp_set_launch_event_filter(None) == 0
    assert lib.rpp_launch_event_count() == 0


def test_patch_merge_size_queries_and_validation(lib):
    from remove_padding_prefix_gb300 import _abi
    ok = _abi.MergeCfg(56, 96, 1e-5, _abi.RPP_F16)
    assert lib.rpp_patch_merge_bytes(C.byref(ok)) >= 8 * 96 * 96 * 2 + 10 * 96 * 4
    assert lib.rpp_patch_merge_workspace_bytes(C.byref(ok), 2) >= 2 * 28 * 28 * 4 * 96 * 2
    assert lib.rpp_patch_merge_bytes(C.byref(_abi.MergeCfg(7, 96, 1e-5, _abi.RPP_F16))) == 0     # odd side
    assert lib.rpp_patch_merge_bytes(C.byref(_abi.MergeCfg(56, 100, 1e-5, _abi.RPP_F16))) == 0   # C % 8
    assert lib.rpp_patch_merge_bytes(C.byref(_abi.MergeCfg(56, 96, 1e-5, _abi.RPP_F32))) == 0    # 16-bit only
    assert lib.rpp_patch_merge_forward(C.byref(ok), None, 1, None, None, None, 0, None, None) == -1


def test_tile_width_hook_rejects_other_values(lib):
    """The tuning hook takes 0 or a tile width the GEMM instantiates (no launch here)."""
    for bad in (-1, 1, 100, 512):
        assert lib.rpp_set_gemm_tile_width(bad) != 0
    for ok in (0, 64, 256, 0):
        assert lib.rpp_set_gemm_tile_width(ok) == 0


def test_stall_hook_rejects_out_of_range_limits(lib):
    """The test-only stall hook takes 1 us .. 1 s and nothing else (no launch here)."""
    assert lib.rpp_test_stall_next_gemm(0) == -1
    assert lib.rpp_test_stall_next_gemm(1000001) == -1
