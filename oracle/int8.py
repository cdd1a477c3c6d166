"""Oracle: the INT8 encoder-layer flow (test infrastructure only).

[SW] §3 (INT8 quantisation): floating-point inputs and weights are quantised to
int8, the int8 matrix product accumulates in int32, and a dequantisation gives
floating-point results again; in the flow used for the transformer every matrix
product is int8 with quantise / dequantise nodes around it, while bias, residual and
LayerNorm stay in floating point (their I/O may be int8).  The int8-output variant
(requantise inside the GEMM epilogue) is used for the FC1 -> FC2 hand-off.

Readings (the talk gives no formulas):

* Weights: symmetric per output channel.  s_w[n] = fp32(max_k |W[k, n]| / 127)
  (one IEEE fp32 division); Wq = clamp(rne(fp32(W / s_w[n])), -127, 127); a column of
  zeros gets s_w = 1.
* Activations: symmetric per tensor, one scale per GEMM input (QKV input, attention
  output, FC1 input, FC2 input).  q = clamp(rne(fp32(fp32(x) * fp32(1 / s_a))), -127, 127):
  the multiply is one IEEE fp32 operation and ties round to even.  These are integer
  decisions, so the oracle takes them in fp32 exactly as the kernels do.
* Scales come from calibration: s_a = fp32(max|x| / 127) over the valid tokens of a
  seeded calibration batch run through the fp64 float layer.
* Accumulation is exact (int64 here; the products fit int32 at these sizes).
* Dequantisation: acc * s_a * s_w[n] + b (fp64 here).
* Attention stays in floating point in the four-GEMM flow (`bert_layer_int8` with four
  scales).  The all-int8 flow (seven scales) also runs both attention products on int8
  codes, `attention_varlen_int8`:
  - Q, K and V are quantised per tensor (scales s_q, s_k, s_v from calibration: the
    max |.| of each over the valid tokens, / 127);
  - the scores are the exact integer product Qc Kc^T, dequantised by s_q s_k / sqrt(d);
  - the softmax runs in floating point over the sequence's keys;
  - P, which lies in [0, 1], is quantised with the fixed scale 1/127: codes
    clamp(rne(127 P), 0, 127).  P is the normalised softmax, so the row maximum and
    sum are known before any code is taken (a two-pass reading of the flow);
  - O = (Pc Vc) s_v / 127, the product again exact in integers.
  The codes of P are decided here in fp64; a kernel deciding them in fp32 can differ by
  one where 127 P lies within rounding distance of a half-integer.
"""
import numpy as np

from .encoder import linear, gelu, layernorm, attention_varlen, _softmax_rows
from .padding import build_offsets, remove_padding

QMAX = 127


def _rne_clamp(v32):
    # np.rint rounds half to even; v32 is float32
    return np.clip(np.rint(v32), -QMAX, QMAX).astype(np.int8)


def quantize_weight_per_channel(W):
    """Per-output-channel symmetric int8 weights: returns (Wq int8 [in, out], s_w float32 [out])."""
    W32 = np.asarray(W, np.float32)
    amax = np.abs(W32).max(axis=0)
    s_w = np.where(amax > 0, amax / np.float32(QMAX), np.float32(1.0)).astype(np.float32)
    q = W32 / s_w[None, :]                      # IEEE fp32 division, element by element
    return _rne_clamp(q.astype(np.float32)), s_w


def quantize_activation(x, s_a):
    """Per-tensor symmetric int8: clamp(rne(fp32(x) * fp32(1/s_a)), -127, 127)."""
    inv = np.float32(1.0) / np.float32(s_a)
    v = np.asarray(x).astype(np.float32) * inv  # one fp32 multiply
    return _rne_clamp(v.astype(np.float32))


def int8_gemm(aq, bq):
    """Exact integer product of int8 matrices aq [M, K] and bq [K, N]; int64 result.

    Computed as a float64 matrix product: every product is an integer of magnitude at
    most 127^2 and every partial sum stays below 2^53 for K < 2^38, so float64
    represents all of them exactly whatever the summation order.
    """
    aq = np.asarray(aq)
    bq = np.asarray(bq)
    assert aq.shape[1] < 2 ** 38
    return (aq.astype(np.float64) @ bq.astype(np.float64)).astype(np.int64)


def int8_linear(x, s_a, Wq, s_w, b):
    """Quantise -> int8 GEMM with integer accumulation -> dequantise + bias ([SW] §3 INT8 flow)."""
    acc = int8_gemm(quantize_activation(x, s_a), Wq)
    return acc.astype(np.float64) * (np.float64(s_a) * np.asarray(s_w, np.float64))[None, :] \
        + np.asarray(b, np.float64)


def prepare_int8_layer(layer):
    """Quantise the four weight matrices of a float layer; biases and LN params stay float."""
    q = {}
    for name in ("Wqkv", "Wo", "W1", "W2"):
        q[name + "_q"], q[name + "_s"] = quantize_weight_per_channel(layer[name])
    for name in ("bqkv", "bo", "b1", "b2", "gamma1", "beta1", "gamma2", "beta2"):
        q[name] = layer[name]
    return q


def attention_varlen_int8(qc, kc, vc, s_q, s_k, s_v, cu_seqlens, nh):
    """fMHA on int8 codes ([SW] §3 INT8 flow: the matrix products int8, Q / DQ around them).

    qc, kc, vc: int8 codes [T, nh*d] (token-major, head h in columns [h*d, (h+1)*d)),
    per-tensor scales s_q, s_k, s_v.  For sequence b and head h:
      S  = Qc Kc^T                       exact integers
      P  = softmax_j(S s_q s_k / sqrt d)  over the sequence's keys, fp64
      Pc = clamp(rne(127 P), 0, 127)
      O  = (Pc Vc) s_v / 127             exact integer product, then fp64
    Returns [T, nh*d] float64.
    """
    qc, kc, vc = (np.asarray(t) for t in (qc, kc, vc))
    T, Hd = qc.shape
    d = Hd // nh
    sc = float(np.float32(s_q)) * float(np.float32(s_k)) / np.sqrt(d)
    dq = float(np.float32(s_v)) / QMAX
    out = np.zeros((T, Hd), np.float64)
    for b in range(len(cu_seqlens) - 1):
        lo, hi = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        if hi == lo:
            continue
        for h in range(nh):
            cs = slice(h * d, (h + 1) * d)
            S = int8_gemm(qc[lo:hi, cs], kc[lo:hi, cs].T)
            P = _softmax_rows(S.astype(np.float64) * sc)
            Pc = np.clip(np.rint(P * QMAX), 0, QMAX).astype(np.int8)
            out[lo:hi, cs] = int8_gemm(Pc, vc[lo:hi, cs]).astype(np.float64) * dq
    return out


def bert_layer_int8(x, cu_seqlens, qlayer, scales, nh, eps):
    """Post-LN layer with the four linear GEMMs in int8 ([SW] §3 INT8 flow).

    scales = (s_qkv_in, s_attn_out, s_fc1_in, s_fc2_in), float32, or those four
    followed by (s_q, s_k, s_v) for the all-int8 flow, where the QKV GEMM's output is
    quantised and the attention runs on codes (`attention_varlen_int8`).
    """
    x = np.asarray(x, np.float64)
    H = x.shape[1]
    s0, s1, s2, s3 = [np.float32(v) for v in scales[:4]]
    qkv = int8_linear(x, s0, qlayer["Wqkv_q"], qlayer["Wqkv_s"], qlayer["bqkv"])
    if len(scales) == 7:
        sq, sk, sv = [np.float32(v) for v in scales[4:]]
        attn = attention_varlen_int8(quantize_activation(qkv[:, :H], sq), quantize_activation(qkv[:, H:2 * H], sk),
                                     quantize_activation(qkv[:, 2 * H:], sv), sq, sk, sv, cu_seqlens, nh)
    else:
        attn = attention_varlen(qkv[:, :H], qkv[:, H:2 * H], qkv[:, 2 * H:], cu_seqlens, nh)
    y = int8_linear(attn, s1, qlayer["Wo_q"], qlayer["Wo_s"], qlayer["bo"]) + x
    x1 = layernorm(y, qlayer["gamma1"], qlayer["beta1"], eps)
    g = gelu(int8_linear(x1, s2, qlayer["W1_q"], qlayer["W1_s"], qlayer["b1"]))
    z = int8_linear(g, s3, qlayer["W2_q"], qlayer["W2_s"], qlayer["b2"]) + x1
    return layernorm(z, qlayer["gamma2"], qlayer["beta2"], eps)


def calibrate_int8(x_padded, lengths, layer, nh, eps):
    """Per-tensor activation scales from a calibration batch through the fp64 float layer.

    Returns float32[4]: max|.| / 127 of the QKV input, the attention output, the FC1
    input (LN1 output) and the FC2 input (GELU output), over valid tokens only.
    """
    x_padded = np.asarray(x_padded)
    _, L, H = x_padded.shape
    cu, po, _ = build_offsets(lengths, L)
    x = remove_padding(x_padded, po).astype(np.float64)
    qkv = linear(x, layer["Wqkv"], layer["bqkv"])
    attn = attention_varlen(qkv[:, :H], qkv[:, H:2 * H], qkv[:, 2 * H:], cu, nh)
    x1 = layernorm(x + linear(attn, layer["Wo"], layer["bo"]), layer["gamma1"], layer["beta1"], eps)
    g = gelu(linear(x1, layer["W1"], layer["b1"]))
    amax = [np.abs(t).max() for t in (x, attn, x1, g)]
    return np.asarray([np.float32(a / QMAX) for a in amax], np.float32)


def calibrate_int8_qkv(x_padded, lengths, layer, nh):
    """Per-tensor scales (s_q, s_k, s_v) of the all-int8 flow: max |.| / 127 of Q, K and V
    (the float QKV projection) over the valid tokens of the calibration batch."""
    x_padded = np.asarray(x_padded)
    _, L, H = x_padded.shape
    _, po, _ = build_offsets(lengths, L)
    qkv = linear(remove_padding(x_padded, po).astype(np.float64), layer["Wqkv"], layer["bqkv"])
    amax = [np.abs(qkv[:, i * H:(i + 1) * H]).max() for i in range(3)]
    return np.asarray([np.float32(a / QMAX) for a in amax], np.float32)
