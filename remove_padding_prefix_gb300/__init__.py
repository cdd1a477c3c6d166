"""Python binding of the padding-removed encoder-layer library (include/rpp.h).

Each function here marshals torch CUDA tensors into the C ABI call of the same name
(``remove_padding`` -> ``rpp_remove_padding`` ...) on the current CUDA stream and
raises :class:`RppError` on a negative status.  Every step of the path runs in the
library's CUDA kernels; PyTorch only provides device memory and the stream.  The
library must have been built (``python -m remove_padding_prefix_gb300.build``); there
is no CPU fallback.
"""
from __future__ import annotations

import ctypes as C
from typing import Optional, Sequence

import numpy as np
import torch

from . import _abi
from ._abi import (RPP_F32, RPP_F16, RPP_BF16, RPP_I8, RPP_EPI_BIAS, RPP_EPI_BIAS_GELU,  # noqa: F401
                   RPP_EPI_BIAS_RESIDUAL, RPP_DERR_LENGTH, RPP_DERR_TIMEOUT, RPP_DERR_ROWS, RPP_DERR_TMEM, EncoderCfg, LayerSrc,
                   SwinCfg, SwinSrc, MergeCfg)

__all__ = [
    "RppError", "lib", "torch_dtype", "dtype_code", "build_offsets", "remove_padding", "rebuild_padding", "linear",
    "layernorm", "attention_varlen", "attention_varlen_i8", "encoder_cfg", "EncoderLayer", "encoder_layer_forward",
    "encoder_layer_calibrate", "encoder_forward", "quantize_weight", "quantize_activation", "gemm_i8_i32",
    "swin_cfg", "SwinBlock", "swin_prepare_bias", "window_attention_forward", "swin_block_forward",
    "merge_cfg", "PatchMerge", "patch_merge_forward",
    "get_device_error", "new_error_word",
]

_DT = {"fp32": RPP_F32, "fp16": RPP_F16, "bf16": RPP_BF16, "int8": RPP_F16}
_TORCH = {RPP_F32: torch.float32, RPP_F16: torch.float16, RPP_BF16: torch.bfloat16, RPP_I8: torch.int8}


class RppError(RuntimeError):
    def __init__(self, name, status):
        msg = lib().rpp_status_string(status).decode()
        super().__init__(f"{name} failed: {msg} ({status})")
        self.status = status


def lib():
    return _abi.load()


def dtype_code(dt) -> int:
    if isinstance(dt, str):
        return _DT[dt]
    for code, t in _TORCH.items():
        if t == dt:
            return code
    raise ValueError(dt)


def torch_dtype(dt) -> torch.dtype:
    return _TORCH[dtype_code(dt) if not isinstance(dt, int) else dt]


def _p(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return t.data_ptr()


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(name, status):
    if status != 0:
        raise RppError(name, status)


def new_error_word(device="cuda") -> torch.Tensor:
    """A zeroed int32 device error word."""
    return torch.zeros(1, dtype=torch.int32, device=device)


def get_device_error(err: torch.Tensor, stream=None) -> int:
    code = C.c_int32(0)
    st = lib().rpp_get_device_error(_p(err), C.byref(code), _stream(stream))
    if st not in (0, _abi.RPP_EDEVICE):
        raise RppError("rpp_get_device_error", st)
    return code.value


# ---------------------------------------------------------------- padding removal
def build_offsets(lengths: torch.Tensor, L: int, cu_seqlens=None, padding_offset=None, err=None, stream=None):
    B = lengths.numel()
    dev = lengths.device
    cu = cu_seqlens if cu_seqlens is not None else torch.empty(B + 1, dtype=torch.int32, device=dev)
    po = padding_offset if padding_offset is not None else torch.zeros(B * L, dtype=torch.int32, device=dev)
    _check("rpp_build_offsets", lib().rpp_build_offsets(_p(lengths), B, L, _p(cu), _p(po), _p(err), _stream(stream)))
    return cu, po


def remove_padding(padded: torch.Tensor, padding_offset, cu_seqlens, B: int, L: int, packed=None, err=None,
                   stream=None):
    H = padded.shape[-1]
    out = packed if packed is not None else torch.empty(B * L, H, dtype=padded.dtype, device=padded.device)
    _check("rpp_remove_padding", lib().rpp_remove_padding(_p(padded), _p(padding_offset), _p(cu_seqlens), B, L, H,
                                                          dtype_code(padded.dtype), _p(out), _p(err),
                                                          _stream(stream)))
    return out


def rebuild_padding(packed: torch.Tensor, cu_seqlens, B: int, L: int, padded=None, err=None, stream=None):
    H = packed.shape[-1]
    out = padded if padded is not None else torch.empty(B * L, H, dtype=packed.dtype, device=packed.device)
    _check("rpp_rebuild_padding", lib().rpp_rebuild_padding(_p(packed), _p(cu_seqlens), B, L, H,
                                                            dtype_code(packed.dtype), _p(out), _p(err),
                                                            _stream(stream)))
    return out


# ---------------------------------------------------------------- building blocks
def linear(a, w_t, bias, epilogue=RPP_EPI_BIAS, residual=None, out=None, rows=None, err=None, stream=None):
    M, K = a.shape
    N = w_t.shape[0]
    o = out if out is not None else torch.empty(M, N, dtype=a.dtype, device=a.device)
    _check("rpp_linear", lib().rpp_linear(_p(a), _p(w_t), _p(bias), _p(residual), _p(o), M, _p(rows), N, K,
                                          dtype_code(a.dtype), epilogue, _p(err), _stream(stream)))
    return o


def layernorm(x, gamma, beta, eps, out=None, rows=None, err=None, stream=None):
    M, H = x.shape
    o = out if out is not None else torch.empty_like(x)
    _check("rpp_layernorm", lib().rpp_layernorm(_p(x), _p(gamma), _p(beta), _p(o), M, _p(rows), H, float(eps),
                                                dtype_code(x.dtype), _p(err), _stream(stream)))
    return o


def attention_varlen(qkv, cu_seqlens, B: int, max_len: int, nh: int, d: int = 64, out=None, err=None, stream=None):
    T_max = qkv.shape[0]
    o = out if out is not None else torch.empty(T_max, nh * d, dtype=qkv.dtype, device=qkv.device)
    _check("rpp_attention_varlen", lib().rpp_attention_varlen(_p(qkv), _p(cu_seqlens), B, T_max, max_len, nh, d,
                                                              dtype_code(qkv.dtype), _p(o), _p(err),
                                                              _stream(stream)))
    return o


def attention_varlen_i8(qkv_codes, qkv_scales, cu_seqlens, B: int, max_len: int, nh: int, d: int = 64, out=None,
                        err=None, stream=None):
    """Attention on int8 codes held in a bf16 [T_max, 3*nh*d] tensor; qkv_scales: device
    float32[3] (s_q, s_k, s_v); returns the fp16 [T_max, nh*d] output."""
    T_max = qkv_codes.shape[0]
    o = out if out is not None else torch.empty(T_max, nh * d, dtype=torch.float16, device=qkv_codes.device)
    _check("rpp_attention_varlen_i8", lib().rpp_attention_varlen_i8(_p(qkv_codes), _p(qkv_scales), _p(cu_seqlens), B,
                                                                    T_max, max_len, nh, d, _p(o), _p(err),
                                                                    _stream(stream)))
    return o


# ---------------------------------------------------------------- encoder layer
def encoder_cfg(H, nh, F, eps, dtype, int8=False, tokens_hint=0) -> EncoderCfg:
    code = dtype_code(dtype) if not isinstance(dtype, int) else dtype
    return EncoderCfg(H, nh, H // nh, F, float(eps), code, int(int8), int(tokens_hint))


class EncoderLayer:
    """One prepared layer: the library-private weight block in device memory."""

    def __init__(self, cfg: EncoderCfg, weights: dict, device="cuda", stream=None):
        self.cfg = cfg
        nbytes = lib().rpp_layer_bytes(C.byref(cfg))
        if nbytes == 0:
            raise RppError("rpp_layer_bytes", _abi.RPP_EINVAL)
        self.block = torch.empty(nbytes, dtype=torch.uint8, device=device)
        tdt = _TORCH[cfg.dtype]
        H = cfg.hidden
        up = lambda a: torch.as_tensor(np.ascontiguousarray(a)).to(device=device, dtype=tdt).contiguous()
        W = weights["Wqkv"]
        b = weights["bqkv"]
        tens = {
            "Wq": up(W[:, :H]), "Wk": up(W[:, H:2 * H]), "Wv": up(W[:, 2 * H:]),
            "bq": up(b[:H]), "bk": up(b[H:2 * H]), "bv": up(b[2 * H:]),
            "Wo": up(weights["Wo"]), "bo": up(weights["bo"]), "W1": up(weights["W1"]), "b1": up(weights["b1"]),
            "W2": up(weights["W2"]), "b2": up(weights["b2"]),
            "gamma1": up(weights["gamma1"]), "beta1": up(weights["beta1"]),
            "gamma2": up(weights["gamma2"]), "beta2": up(weights["beta2"]),
        }
        src = LayerSrc(**{k: v.data_ptr() for k, v in tens.items()})
        _check("rpp_prepare_layer", lib().rpp_prepare_layer(C.byref(cfg), C.byref(src), _p(self.block),
                                                            _stream(stream)))
        (stream or torch.cuda.current_stream()).synchronize()   # the source tensors die here
        del tens

    def workspace_bytes(self, T_max: int) -> int:
        return lib().rpp_encoder_workspace_bytes(C.byref(self.cfg), T_max)

    def workspace(self, T_max: int, device="cuda") -> torch.Tensor:
        return torch.empty(self.workspace_bytes(T_max), dtype=torch.uint8, device=device)


def encoder_layer_forward(layer: EncoderLayer, x, cu_seqlens, B: int, max_len: int, y=None, workspace=None,
                          act_scales=None, err=None, stream=None):
    T_max = x.shape[0]
    out = y if y is not None else torch.empty_like(x)
    ws = workspace if workspace is not None else layer.workspace(T_max, x.device)
    _check("rpp_encoder_layer_forward",
           lib().rpp_encoder_layer_forward(C.byref(layer.cfg), _p(layer.block), _p(act_scales), _p(x),
                                           _p(cu_seqlens), B, T_max, max_len, _p(out), _p(ws), ws.numel(), _p(err),
                                           _stream(stream)))
    return out


def encoder_layer_calibrate(layer: EncoderLayer, x, cu_seqlens, B: int, max_len: int, workspace=None, err=None,
                            stream=None):
    T_max = x.shape[0]
    amax = torch.empty(7, dtype=torch.float32, device=x.device)
    ws = workspace if workspace is not None else layer.workspace(T_max, x.device)
    _check("rpp_encoder_layer_calibrate",
           lib().rpp_encoder_layer_calibrate(C.byref(layer.cfg), _p(layer.block), _p(x), _p(cu_seqlens), B, T_max,
                                             max_len, _p(amax), _p(ws), ws.numel(), _p(err), _stream(stream)))
    return amax


def encoder_forward(layers: Sequence[EncoderLayer], lengths, x_padded, L: int, act_scales=None, y_padded=None,
                    cu_seqlens=None, padding_offset=None, packed=None, workspace=None, err=None, stream=None):
    """Offsets -> remove padding -> layers -> rebuild padding, one C ABI call."""
    B = lengths.numel()
    H = x_padded.shape[-1]
    dev = x_padded.device
    cfg = layers[0].cfg
    y = y_padded if y_padded is not None else torch.empty(B * L, H, dtype=x_padded.dtype, device=dev)
    cu = cu_seqlens if cu_seqlens is not None else torch.empty(B + 1, dtype=torch.int32, device=dev)
    po = padding_offset if padding_offset is not None else torch.zeros(B * L, dtype=torch.int32, device=dev)
    pk = packed if packed is not None else torch.empty(B * L, H, dtype=x_padded.dtype, device=dev)
    ws = workspace if workspace is not None else layers[0].workspace(B * L, dev)
    lp = (C.c_void_p * len(layers))(*[l.block.data_ptr() for l in layers])
    sp = None
    if act_scales is not None:
        sp = (C.c_void_p * len(layers))(*[s.data_ptr() for s in act_scales])
    _check("rpp_encoder_forward",
           lib().rpp_encoder_forward(C.byref(cfg), lp, sp, len(layers), _p(lengths), B, L, _p(x_padded), _p(y),
                                     _p(cu), _p(po), _p(pk), _p(ws), ws.numel(), _p(err), _stream(stream)))
    return y, cu, po


# ---------------------------------------------------------------- int8 pieces
def quantize_weight(w, stream=None):
    """w [K, N] (in, out) -> (codes int8 [N, K], s_w float32 [N])."""
    K, N = w.shape
    q = torch.empty(N, K, dtype=torch.int8, device=w.device)
    s = torch.empty(N, dtype=torch.float32, device=w.device)
    _check("rpp_quantize_weight", lib().rpp_quantize_weight(_p(w), K, N, dtype_code(w.dtype), _p(q), _p(s),
                                                            _stream(stream)))
    return q, s


def quantize_activation(x, scale, rows=None, err=None, stream=None):
    M, H = x.shape
    q = torch.empty(M, H, dtype=torch.int8, device=x.device)
    _check("rpp_quantize_activation", lib().rpp_quantize_activation(_p(x), _p(scale), _p(q), M, _p(rows), H,
                                                                    dtype_code(x.dtype), _p(err), _stream(stream)))
    return q


def gemm_i8_i32(aq, wq_t, workspace=None, err=None, stream=None):
    M, K = aq.shape
    N = wq_t.shape[0]
    acc = torch.empty(M, N, dtype=torch.int32, device=aq.device)
    nbytes = lib().rpp_gemm_i8_workspace_bytes(M, N, K)
    ws = workspace if workspace is not None else torch.empty(nbytes, dtype=torch.uint8, device=aq.device)
    _check("rpp_gemm_i8_i32", lib().rpp_gemm_i8_i32(_p(aq), _p(wq_t), _p(acc), M, N, K, _p(ws), ws.numel(), _p(err),
                                                    _stream(stream)))
    return acc


# ---------------------------------------------------------------- Swin
def swin_cfg(I, C_, nh, w, s, mlp, eps, dtype) -> SwinCfg:
    code = dtype_code(dtype) if not isinstance(dtype, int) else dtype
    return SwinCfg(I, C_, nh, w, s, mlp, float(eps), code)


def swin_prepare_bias(cfg: SwinCfg, table, stream=None):
    N = cfg.window * cfg.window
    bias = torch.empty(cfg.heads, N, N, dtype=torch.float32, device=table.device)
    _check("rpp_swin_prepare_bias", lib().rpp_swin_prepare_bias(C.byref(cfg), _p(table), _p(bias), _stream(stream)))
    return bias


def window_attention_forward(cfg: SwinCfg, B: int, qkv, bias, out=None, err=None, stream=None):
    o = out if out is not None else torch.empty(qkv.shape[0], cfg.channels, dtype=qkv.dtype, device=qkv.device)
    _check("rpp_window_attention_forward",
           lib().rpp_window_attention_forward(C.byref(cfg), B, _p(qkv), _p(bias), _p(o), _p(err), _stream(stream)))
    return o


class SwinBlock:
    """One prepared Swin block (library-private weight block in device memory)."""

    def __init__(self, cfg: SwinCfg, weights: dict, device="cuda", stream=None):
        self.cfg = cfg
        nbytes = lib().rpp_swin_block_bytes(C.byref(cfg))
        if nbytes == 0:
            raise RppError("rpp_swin_block_bytes", _abi.RPP_EINVAL)
        self.block = torch.empty(nbytes, dtype=torch.uint8, device=device)
        tdt = _TORCH[cfg.dtype]
        up = lambda a: torch.as_tensor(np.ascontiguousarray(a)).to(device=device, dtype=tdt).contiguous()
        tens = {k: up(weights[k]) for k in ("gamma1", "beta1", "Wqkv", "bqkv", "table", "Wo", "bo", "gamma2",
                                            "beta2", "W1", "b1", "W2", "b2")}
        src = SwinSrc(**{k: v.data_ptr() for k, v in tens.items()})
        _check("rpp_swin_prepare_block", lib().rpp_swin_prepare_block(C.byref(cfg), C.byref(src), _p(self.block),
                                                                      _stream(stream)))
        (stream or torch.cuda.current_stream()).synchronize()
        del tens

    def workspace_bytes(self, B: int) -> int:
        return lib().rpp_swin_workspace_bytes(C.byref(self.cfg), B)

    def workspace(self, B: int, device="cuda") -> torch.Tensor:
        return torch.empty(self.workspace_bytes(B), dtype=torch.uint8, device=device)


def swin_block_forward(block: SwinBlock, x, B: int, y=None, workspace=None, err=None, stream=None):
    out = y if y is not None else torch.empty_like(x)
    ws = workspace if workspace is not None else block.workspace(B, x.device)
    _check("rpp_swin_block_forward",
           lib().rpp_swin_block_forward(C.byref(block.cfg), _p(block.block), B, _p(x), _p(out), _p(ws), ws.numel(),
                                        _p(err), _stream(stream)))
    return out


# ---------------------------------------------------------------- Swin patch merging
def merge_cfg(I, C_, eps, dtype) -> MergeCfg:
    code = dtype_code(dtype) if not isinstance(dtype, int) else dtype
    return MergeCfg(I, C_, float(eps), code)


class PatchMerge:
    """Prepared patch-merging weights (K-major reduction map, fp32 LayerNorm parameters)."""

    def __init__(self, cfg: MergeCfg, gamma, beta, W, device="cuda", stream=None):
        self.cfg = cfg
        nbytes = lib().rpp_patch_merge_bytes(C.byref(cfg))
        if nbytes == 0:
            raise RppError("rpp_patch_merge_bytes", _abi.RPP_EUNSUPPORTED)
        self.block = torch.empty(nbytes, dtype=torch.uint8, device=device)
        tdt = _TORCH[cfg.dtype]
        up = lambda a: torch.as_tensor(np.ascontiguousarray(a)).to(device=device, dtype=tdt).contiguous()
        g, b, w = up(gamma), up(beta), up(W)
        _check("rpp_patch_merge_prepare", lib().rpp_patch_merge_prepare(C.byref(cfg), _p(g), _p(b), _p(w),
                                                                        _p(self.block), _stream(stream)))
        (stream or torch.cuda.current_stream()).synchronize()

    def workspace(self, B: int, device="cuda") -> torch.Tensor:
        return torch.empty(lib().rpp_patch_merge_workspace_bytes(C.byref(self.cfg), B), dtype=torch.uint8,
                           device=device)


def patch_merge_forward(pm: PatchMerge, x, B: int, y=None, workspace=None, err=None, stream=None):
    I, C_ = pm.cfg.img, pm.cfg.channels
    out = y if y is not None else torch.empty(B * (I // 2) * (I // 2), 2 * C_, dtype=x.dtype, device=x.device)
    ws = workspace if workspace is not None else pm.workspace(B, x.device)
    _check("rpp_patch_merge_forward",
           lib().rpp_patch_merge_forward(C.byref(pm.cfg), _p(pm.block), B, _p(x), _p(out), _p(ws), ws.numel(),
                                         _p(err), _stream(stream)))
    return out
