"""Oracle: the Swin shifted-window block, fp64 (test infrastructure only).

Passages followed ([SW]): §1 describes window attention (attention only among the
patches of one window), the cyclic window shift that links neighbouring windows, and
the relative position bias; §2 treats shift / partition / merge as pure index
mappings and runs fMHA with the mask and bias given as tensors; §3 moves the
relative-position-bias lookup into preprocessing.  The block is pre-LayerNorm
(attention and MLP each wrapped as x + f(LN(x))).

Readings (the talk names these pieces without formulas; the standard Swin
definitions are taken):

* Shift: roll by -s on both image axes, x'[y, x] = x[(y+s) mod I, (x+s) mod I];
  unshift rolls by +s.
* Windows are numbered row-major inside an image, win = (y // w) * (I // w) + x // w,
  token t = (y % w) * w + x % w.
* Relative position bias: B[h, t, u] = table[(ty - uy + w - 1) * (2w - 1)
  + (tx - ux + w - 1), h] with (ty, tx), (uy, ux) the in-window coordinates.
* Shift mask: in the shifted frame each axis coordinate c has region r(c) = 0 if
  c < I - w, 1 if c < I - s, 2 otherwise; tokens of one window attend to each other
  only when 3 r(y) + r(x) agrees.  Excluded pairs are dropped from the softmax (the
  usual additive -100 differs from exclusion by e^-100).
* Attention scale 1 / sqrt(d); LayerNorm eps 1e-5.
* Downsampling between stages (the talk shows stages at falling resolution with a
  downsampling step between them, without its formula): the standard patch merging is
  taken.  Output token (py, px) concatenates the four input tokens (2py, 2px),
  (2py+1, 2px), (2py, 2px+1), (2py+1, 2px+1) in that order (4C channels), applies
  LayerNorm over the 4C channels and a bias-free linear map 4C -> 2C.
"""
import numpy as np

from .encoder import linear, gelu, layernorm


def shift(img, s):
    """Cyclic shift by -s on both axes: out[y, x] = img[(y+s) % I, (x+s) % I].  img [I, I, ...]."""
    I = img.shape[0]
    out = np.empty_like(img)
    for y in range(I):
        for x in range(I):
            out[y, x] = img[(y + s) % I, (x + s) % I]
    return out


def unshift(img, s):
    """Inverse of :func:`shift`: out[(y+s) % I, (x+s) % I] = img[y, x]."""
    I = img.shape[0]
    out = np.empty_like(img)
    for y in range(I):
        for x in range(I):
            out[(y + s) % I, (x + s) % I] = img[y, x]
    return out


def window_coords(I, w):
    """For each (window, token) the shifted-frame coordinates: int arrays yy, xx of shape [nW, w*w]."""
    nWs = I // w
    yy = np.empty((nWs * nWs, w * w), np.int64)
    xx = np.empty((nWs * nWs, w * w), np.int64)
    for wy in range(nWs):
        for wx in range(nWs):
            for t in range(w * w):
                yy[wy * nWs + wx, t] = wy * w + t // w
                xx[wy * nWs + wx, t] = wx * w + t % w
    return yy, xx


def window_partition(img, w):
    """[I, I, C] -> [nW, w*w, C] with the row-major window / token numbering."""
    yy, xx = window_coords(img.shape[0], w)
    return img[yy, xx]


def window_reverse(win, I, w):
    """[nW, w*w, C] -> [I, I, C], inverse of :func:`window_partition`."""
    yy, xx = window_coords(I, w)
    out = np.empty((I, I) + win.shape[2:], dtype=win.dtype)
    out[yy, xx] = win
    return out


def relative_position_bias(table, w):
    """Bias lookup of [SW] §1/§3 done once in preprocessing: [nh, w*w, w*w] from table [(2w-1)^2, nh]."""
    table = np.asarray(table, np.float64)
    nh = table.shape[1]
    N = w * w
    out = np.empty((nh, N, N), np.float64)
    for t in range(N):
        ty, tx = divmod(t, w)
        for u in range(N):
            uy, ux = divmod(u, w)
            idx = (ty - uy + w - 1) * (2 * w - 1) + (tx - ux + w - 1)
            out[:, t, u] = table[idx, :]
    return out


def shift_attend_mask(I, w, s):
    """Boolean [nW, w*w, w*w]: True where token t may attend to token u (shifted-window mask)."""
    yy, xx = window_coords(I, w)
    nW, N = yy.shape
    if s == 0:
        return np.ones((nW, N, N), bool)

    def region(c):
        return np.where(c < I - w, 0, np.where(c < I - s, 1, 2))

    label = 3 * region(yy) + region(xx)
    return label[:, :, None] == label[:, None, :]


def _window_attention_windows(qw, kw, vw, bias, allow, nh):
    """Attention inside each window: qw/kw/vw [nW, N, C]; returns [nW, N, C]."""
    nW, N, C = qw.shape
    d = C // nh
    scale = 1.0 / np.sqrt(d)
    out = np.zeros((nW, N, C), np.float64)
    for h in range(nh):
        cs = slice(h * d, (h + 1) * d)
        s = np.einsum("wtd,wud->wtu", qw[:, :, cs], kw[:, :, cs]) * scale + bias[h][None]
        s = np.where(allow, s, -np.inf)
        m = s.max(axis=-1, keepdims=True)
        e = np.exp(s - m)
        p = e / e.sum(axis=-1, keepdims=True)
        out[:, :, cs] = np.einsum("wtu,wud->wtd", p, vw[:, :, cs])
    return out


def window_attention(qkv, I, w, s, nh, bias):
    """Shifted-window attention on raster-order projected tokens ([SW] §1-§3).

    qkv: [B, I*I, 3C] in raster order (columns Q | K | V, head-contiguous).
    bias: [nh, w*w, w*w] from :func:`relative_position_bias`.
    Returns the attention output [B, I*I, C] in raster order (before the output
    projection): shift -> partition -> attention with bias and mask -> reverse -> unshift.
    """
    qkv = np.asarray(qkv, np.float64)
    B, T_img, C3 = qkv.shape
    C = C3 // 3
    allow = shift_attend_mask(I, w, s)
    out = np.empty((B, T_img, C), np.float64)
    for b in range(B):
        img = qkv[b].reshape(I, I, C3)
        win = window_partition(shift(img, s), w)
        o = _window_attention_windows(win[..., :C], win[..., C:2 * C], win[..., 2 * C:], bias, allow, nh)
        out[b] = unshift(window_reverse(o, I, w), s).reshape(T_img, C)
    return out


def swin_block(x, wt, I, w, s, nh, eps):
    """Pre-LN shifted-window block on x [B, I*I, C] ([SW] §1 structure, §3 fused path).

    x' = x + unshift(reverse(proj(WAttn(partition(shift(LN1 x))))));  y = x' + MLP(LN2 x').
    The QKV projection and the output projection are applied to window-partitioned
    tokens here, as in the block's definition.
    """
    x = np.asarray(x, np.float64)
    B, T_img, C = x.shape
    bias = relative_position_bias(wt["table"], w)
    allow = shift_attend_mask(I, w, s)
    out = np.empty_like(x)
    for b in range(B):
        h = layernorm(x[b], wt["gamma1"], wt["beta1"], eps).reshape(I, I, C)
        win = window_partition(shift(h, s), w)                      # [nW, N, C]
        qkv = linear(win, wt["Wqkv"], wt["bqkv"])
        o = _window_attention_windows(qkv[..., :C], qkv[..., C:2 * C], qkv[..., 2 * C:], bias, allow, nh)
        o = linear(o, wt["Wo"], wt["bo"])
        xa = x[b] + unshift(window_reverse(o, I, w), s).reshape(T_img, C)
        m = linear(gelu(linear(layernorm(xa, wt["gamma2"], wt["beta2"], eps), wt["W1"], wt["b1"])),
                   wt["W2"], wt["b2"])
        out[b] = xa + m
    return out


def patch_merge(x, I, gamma, beta, W, eps):
    """Stage downsampling of x [B, I*I, C] (raster) into [B, (I/2)^2, 2C]: the 2 x 2
    neighbourhood of each output token concatenated in the order (0,0), (1,0), (0,1),
    (1,1) of (row offset, column offset), LayerNorm over 4C, then x @ W with W [4C, 2C]
    and no bias."""
    x = np.asarray(x, np.float64)
    B, T_img, C = x.shape
    assert T_img == I * I and I % 2 == 0
    Ih = I // 2
    out = np.empty((B, Ih * Ih, W.shape[1]), np.float64)
    for b in range(B):
        img = x[b].reshape(I, I, C)
        cat = np.empty((Ih, Ih, 4 * C), np.float64)
        for k, (dy, dx) in enumerate(((0, 0), (1, 0), (0, 1), (1, 1))):
            cat[:, :, k * C:(k + 1) * C] = img[dy::2, dx::2, :]
        h = layernorm(cat.reshape(Ih * Ih, 4 * C), gamma, beta, eps)
        out[b] = linear(h, W)
    return out
