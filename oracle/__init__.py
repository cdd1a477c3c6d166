"""CPU oracle for the padding-removed encoder-layer forward pass (TEST INFRASTRUCTURE ONLY).

This package is the plain, slow, obviously-correct statement of what the GPU path
computes.  It is test infrastructure: only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it.  It shares no code with the
CUDA library (no kernels, headers, helpers or constant tables); the two meet only on
the seeded inputs produced by ``workloads``.

Arithmetic is fp64 unless a step is an integer decision (int8 quantisation), where
the oracle takes the decision in IEEE fp32 exactly as the kernel does.

Sources cited in the docstrings (by page title and figure/section):

* [KS] "GPU底層優化 | 如何讓Transformer在GPU上跑得更快？" (Kuaishou heterogeneous
  computing team).  Fig. 9: padding removal through an Offset Mask, packed and padded
  sequences convert into each other.  Fig. 10: kernels classified by whether they can
  run on the packed tokens.  Fig. 6: fusion of the self-attention and FFN blocks.
* [SW] NVIDIA talk "Swin Transformer training and inference optimisation" (Japanese
  transcript, m.sbmmt.com/ja/faq/533025).  §1: window attention, cyclic window shift
  and relative position bias; §2: window shift/partition/merge are index mappings,
  fMHA with mask and bias tensors; §3 (inference): relative-position-bias lookup moved
  to preprocessing, fMHA = batch GEMM + softmax + batch GEMM with the transposes in its
  I/O, QKV GEMM+bias with reformatted weights, the INT8 flow (int8 GEMM with int32
  accumulation, dequantise, bias/residual/LayerNorm kept in floating point).

Pins (tests/test_oracle_*.py) check every function here against closed forms,
library routines that reduce to the same definition, invariants and brute force.
"""
from .padding import build_offsets, remove_padding, rebuild_padding
from .encoder import (linear, gelu, layernorm, attention_varlen, bert_layer,
                      bert_forward, bert_stack_packed)
from .swin import (shift, unshift, window_partition, window_reverse, window_coords,
                   relative_position_bias, shift_attend_mask, window_attention,
                   swin_block, patch_merge)
from .int8 import (quantize_weight_per_channel, quantize_activation, int8_gemm,
                   int8_linear, bert_layer_int8, calibrate_int8, prepare_int8_layer,
                   attention_varlen_int8, calibrate_int8_qkv)

__all__ = [
    "build_offsets", "remove_padding", "rebuild_padding",
    "linear", "gelu", "layernorm", "attention_varlen", "bert_layer", "bert_forward",
    "bert_stack_packed",
    "shift", "unshift", "window_partition", "window_reverse", "window_coords",
    "relative_position_bias", "shift_attend_mask", "window_attention", "swin_block", "patch_merge",
    "quantize_weight_per_channel", "quantize_activation", "int8_gemm", "int8_linear",
    "bert_layer_int8", "calibrate_int8", "prepare_int8_layer",
    "attention_varlen_int8", "calibrate_int8_qkv",
]
