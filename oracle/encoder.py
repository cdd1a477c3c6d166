"""Oracle: the BERT-shaped (post-LayerNorm) encoder layer on packed tokens, fp64.

Test infrastructure only.  Passages followed:

* [KS] Fig. 6 (self-attention and feed-forward blocks fused and restructured) and
  Fig. 10 (row-wise kernels run on the packed tokens; attention needs the sequence
  boundaries), with the encoder structure of Fig. 3 (attention + FFN).
* [SW] §3: fMHA is batch GEMM -> softmax -> batch GEMM; GEMM + bias (+ activation)
  epilogues; bias split from the GEMM and fused into the following op (residual,
  LayerNorm).

Readings where the pages are silent:

* Linear weights are stored [in, out]: y = x @ W + b.
* GELU is the exact erf form x * Phi(x).
* LayerNorm uses the biased variance over the hidden dimension, eps inside the
  square root.
* Keys past a sequence's length are excluded from its softmax (equivalent to an
  additive -inf); there are no fully-masked query rows because only valid queries
  produce outputs.
* Post-LN layer: X1 = LN1(X + Attn(X) Wo + bo); Y = LN2(X1 + GELU(X1 W1 + b1) W2 + b2).
"""
import numpy as np
from scipy.special import erf

from .padding import build_offsets, remove_padding, rebuild_padding


def linear(x, W, b=None):
    """y = x @ W (+ b), W stored [in, out] ([SW] §3 GEMM + bias)."""
    y = np.asarray(x, np.float64) @ np.asarray(W, np.float64)
    if b is not None:
        y = y + np.asarray(b, np.float64)
    return y


def gelu(x):
    """Exact GELU, x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)) ([SW] §3 GEMM + bias + activation)."""
    x = np.asarray(x, np.float64)
    return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))


def layernorm(x, gamma, beta, eps):
    """Row LayerNorm: (x - mean) / sqrt(var + eps) * gamma + beta, biased variance ([SW] §2-3)."""
    x = np.asarray(x, np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)


def _softmax_rows(s):
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=-1, keepdims=True)


def attention_varlen(q, k, v, cu_seqlens, nh):
    """Multi-head attention over packed variable-length sequences ([SW] §3 fMHA; [KS] Fig. 10).

    q, k, v: [T, nh*d] token-major, head h in columns [h*d, (h+1)*d).  For sequence b
    (packed rows cu[b]..cu[b+1]) and head h: o_i = sum_j softmax_j(q_i . k_j / sqrt d) v_j,
    with j running over the same sequence only.  Returns [T, nh*d].
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    T, Hd = q.shape
    d = Hd // nh
    scale = 1.0 / np.sqrt(d)
    out = np.zeros((T, Hd), np.float64)
    B = len(cu_seqlens) - 1
    for b in range(B):
        lo, hi = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        if hi == lo:
            continue
        for h in range(nh):
            cs = slice(h * d, (h + 1) * d)
            s = (q[lo:hi, cs] @ k[lo:hi, cs].T) * scale
            p = _softmax_rows(s)
            out[lo:hi, cs] = p @ v[lo:hi, cs]
    return out


def bert_layer(x, cu_seqlens, layer, nh, eps):
    """One post-LN encoder layer on packed tokens x [T, H] ([KS] Fig. 6, [SW] §3).

    ``layer`` holds Wqkv [H, 3H] (columns Q | K | V, head-contiguous), bqkv, Wo, bo,
    W1, b1, W2, b2, gamma1, beta1, gamma2, beta2.
    """
    x = np.asarray(x, np.float64)
    H = x.shape[1]
    qkv = linear(x, layer["Wqkv"], layer["bqkv"])
    q, k, v = qkv[:, :H], qkv[:, H:2 * H], qkv[:, 2 * H:]
    attn = attention_varlen(q, k, v, cu_seqlens, nh)
    x1 = layernorm(x + linear(attn, layer["Wo"], layer["bo"]), layer["gamma1"], layer["beta1"], eps)
    g = gelu(linear(x1, layer["W1"], layer["b1"]))
    y = layernorm(x1 + linear(g, layer["W2"], layer["b2"]), layer["gamma2"], layer["beta2"], eps)
    return y


def bert_stack_packed(x, cu_seqlens, layers, nh, eps):
    """Apply the layers in order to packed tokens."""
    for layer in layers:
        x = bert_layer(x, cu_seqlens, layer, nh, eps)
    return x


def bert_forward(x_padded, lengths, layers, nh, eps):
    """Whole path of [KS] Fig. 9/10: offsets -> remove padding -> layers -> rebuild padding.

    Returns (y_padded [B, L, H] with zero pads, cu_seqlens, padding_offset).
    """
    x_padded = np.asarray(x_padded)
    B, L, _ = x_padded.shape
    cu, po, T = build_offsets(lengths, L)
    x = remove_padding(x_padded, po).astype(np.float64)
    y = bert_stack_packed(x, cu, layers, nh, eps)
    return rebuild_padding(y, cu, B, L), cu, po
