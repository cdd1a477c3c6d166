"""ctypes declarations of the C ABI in include/rpp.h (argument marshalling only).

Loading fails loudly when the library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "librpp.so")

RPP_OK, RPP_EINVAL, RPP_EUNSUPPORTED, RPP_ECUDA, RPP_EWORKSPACE, RPP_EDEVICE = 0, -1, -2, -3, -4, -5
RPP_F32, RPP_F16, RPP_BF16, RPP_I8 = 0, 1, 2, 3
RPP_EPI_BIAS, RPP_EPI_BIAS_GELU, RPP_EPI_BIAS_RESIDUAL = 0, 1, 2
RPP_DERR_LENGTH, RPP_DERR_TIMEOUT, RPP_DERR_ROWS, RPP_DERR_TMEM = 1, 2, 3, 4

vp = C.c_void_p
i32 = C.c_int
f32 = C.c_float
sz = C.c_size_t


class EncoderCfg(C.Structure):
    _fields_ = [("hidden", i32), ("heads", i32), ("head_dim", i32), ("ffn", i32), ("eps", f32),
                ("dtype", i32), ("int8", i32), ("tokens_hint", i32)]


class LayerSrc(C.Structure):
    _fields_ = [(n, vp) for n in ("Wq", "Wk", "Wv", "bq", "bk", "bv", "Wo", "bo", "W1", "b1", "W2", "b2",
                                  "gamma1", "beta1", "gamma2", "beta2")]


class SwinCfg(C.Structure):
    _fields_ = [("img", i32), ("channels", i32), ("heads", i32), ("window", i32), ("shift", i32),
                ("mlp", i32), ("eps", f32), ("dtype", i32)]


class MergeCfg(C.Structure):
    _fields_ = [("img", i32), ("channels", i32), ("eps", f32), ("dtype", i32)]


class SwinSrc(C.Structure):
    _fields_ = [(n, vp) for n in ("gamma1", "beta1", "Wqkv", "bqkv", "table", "Wo", "bo", "gamma2", "beta2",
                                  "W1", "b1", "W2", "b2")]


# name -> (restype, argtypes); mirrors include/rpp.h
SIGNATURES = {
    "rpp_status_string": (C.c_char_p, [i32]),
    "rpp_version": (i32, []),
    "rpp_set_launch_events": (i32, [C.POINTER(vp), i32]),
    "rpp_set_launch_event_filter": (i32, [C.c_char_p]),
    "rpp_set_gemm_cluster_mode": (i32, [i32]),
    "rpp_set_gemm_tile_width": (i32, [i32]),
    "rpp_test_stall_next_gemm": (i32, [C.c_uint]),
    "rpp_launch_event_count": (i32, []),
    "rpp_launch_event_label": (C.c_char_p, [i32]),
    "rpp_get_device_error": (i32, [vp, C.POINTER(C.c_int32), vp]),
    "rpp_build_offsets": (i32, [vp, i32, i32, vp, vp, vp, vp]),
    "rpp_remove_padding": (i32, [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp]),
    "rpp_rebuild_padding": (i32, [vp, vp, i32, i32, i32, i32, vp, vp, vp]),
    "rpp_linear": (i32, [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, vp, vp]),
    "rpp_layernorm": (i32, [vp, vp, vp, vp, i32, vp, i32, f32, i32, vp, vp]),
    "rpp_attention_varlen": (i32, [vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp]),
    "rpp_attention_varlen_i8": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]),
    "rpp_layer_bytes": (sz, [C.POINTER(EncoderCfg)]),
    "rpp_prepare_layer": (i32, [C.POINTER(EncoderCfg), C.POINTER(LayerSrc), vp, vp]),
    "rpp_encoder_workspace_bytes": (sz, [C.POINTER(EncoderCfg), i32]),
    "rpp_encoder_layer_forward": (i32, [C.POINTER(EncoderCfg), vp, vp, vp, vp, i32, i32, i32, vp, vp, sz, vp, vp]),
    "rpp_encoder_layer_calibrate": (i32, [C.POINTER(EncoderCfg), vp, vp, vp, i32, i32, i32, vp, vp, sz, vp, vp]),
    "rpp_encoder_forward": (i32, [C.POINTER(EncoderCfg), C.POINTER(vp), C.POINTER(vp), i32, vp, i32, i32, vp, vp,
                                  vp, vp, vp, vp, sz, vp, vp]),
    "rpp_quantize_weight": (i32, [vp, i32, i32, i32, vp, vp, vp]),
    "rpp_quantize_activation": (i32, [vp, vp, vp, i32, vp, i32, i32, vp, vp]),
    "rpp_gemm_i8_workspace_bytes": (sz, [i32, i32, i32]),
    "rpp_gemm_i8_i32": (i32, [vp, vp, vp, i32, i32, i32, vp, sz, vp, vp]),
    "rpp_gemm_i8_i32_noalloc": (i32, [vp, vp, vp, i32, i32, i32, vp, vp]),
    "rpp_swin_prepare_bias": (i32, [C.POINTER(SwinCfg), vp, vp, vp]),
    "rpp_window_attention_forward": (i32, [C.POINTER(SwinCfg), i32, vp, vp, vp, vp, vp]),
    "rpp_swin_block_bytes": (sz, [C.POINTER(SwinCfg)]),
    "rpp_swin_prepare_block": (i32, [C.POINTER(SwinCfg), C.POINTER(SwinSrc), vp, vp]),
    "rpp_swin_workspace_bytes": (sz, [C.POINTER(SwinCfg), i32]),
    "rpp_swin_block_forward": (i32, [C.POINTER(SwinCfg), vp, i32, vp, vp, vp, sz, vp, vp]),
    "rpp_patch_merge_bytes": (sz, [C.POINTER(MergeCfg)]),
    "rpp_patch_merge_prepare": (i32, [C.POINTER(MergeCfg), vp, vp, vp, vp, vp]),
    "rpp_patch_merge_workspace_bytes": (sz, [C.POINTER(MergeCfg), i32]),
    "rpp_patch_merge_forward": (i32, [C.POINTER(MergeCfg), vp, i32, vp, vp, vp, sz, vp, vp]),
}

_lib = None


def load():
    """Load librpp.so (built by remove_padding_prefix_gb300.build) and declare every entry point."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: run `python -m remove_padding_prefix_gb300.build` "
                           "(the CUDA library is required; there is no CPU fallback)")
    lib = C.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
