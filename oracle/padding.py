"""Oracle: the offset mask, padding removal and padding rebuild (test infrastructure only).

[KS] Fig. 9 states that introducing an Offset Mask lets the padding-removed sequence
and the original padded sequence be converted into each other.  The figure itself is
not reproduced on the page, so the content of the mask is a reading:

* ``cu_seqlens[b]`` is the exclusive prefix sum of the valid lengths (the packed row
  where sequence b starts), ``cu_seqlens[B] = T``;
* ``padding_offset[i]`` is the number of pad slots that precede packed token i in the
  padded [B, L] layout, so that packed token i lives at padded flat row
  ``i + padding_offset[i]`` (for token p of sequence b: ``b*L - cu_seqlens[b]``).

Pad slots are filled with zeros on rebuild (the page is silent on the fill value).
"""
import numpy as np


def build_offsets(lengths, L):
    """Offset mask of [KS] Fig. 9: returns (cu_seqlens int32[B+1], padding_offset int32[T], T).

    A length outside [0, L] is an error (ValueError); a length of 0 makes the
    sequence vanish from the packed batch.
    """
    lengths = [int(v) for v in np.asarray(lengths).reshape(-1)]
    for v in lengths:
        if v < 0 or v > L:
            raise ValueError(f"sequence length {v} outside [0, {L}]")
    B = len(lengths)
    cu = [0] * (B + 1)
    for b in range(B):
        cu[b + 1] = cu[b] + lengths[b]
    T = cu[B]
    offs = [0] * T
    for b in range(B):
        for i in range(cu[b], cu[b + 1]):
            offs[i] = b * L - cu[b]
    return np.asarray(cu, np.int32), np.asarray(offs, np.int32), T


def remove_padding(padded, padding_offset):
    """Gather the valid tokens ([KS] Fig. 9): packed[i] = padded_rows[i + padding_offset[i]].

    ``padded`` is [B, L, ...]; the result is [T, ...] with T = len(padding_offset).
    """
    padded = np.asarray(padded)
    rows = padded.reshape((-1,) + padded.shape[2:])
    T = len(padding_offset)
    out = np.empty((T,) + padded.shape[2:], dtype=padded.dtype)
    for i in range(T):
        out[i] = rows[i + int(padding_offset[i])]
    return out


def rebuild_padding(packed, cu_seqlens, B, L):
    """Scatter packed tokens back to [B, L, ...] ([KS] Fig. 9); pad slots become 0."""
    packed = np.asarray(packed)
    out = np.zeros((B, L) + packed.shape[1:], dtype=packed.dtype)
    for b in range(B):
        n = int(cu_seqlens[b + 1]) - int(cu_seqlens[b])
        for p in range(n):
            out[b, p] = packed[int(cu_seqlens[b]) + p]
    return out
