"""Padded packed rows <-> compact THD, written out plainly - TEST
INFRASTRUCTURE (used by the tests and the benchmark's checks only).

Definition (NeMo-Automodel PR "feat(minimax-m3): add SM100 MSA sparse
attention with custom backward", section "Design": the padding tokens of
packed rows are dropped before the flat attention call, its output scattered
back): row b of a [B, S, ...] array holds row_len[b] real tokens followed by
padding; the compact array lists the real tokens of row 0, then row 1, ...;
unpacking puts them back and zero-fills the padding.  Lengths are clamped
into [0, S].
"""
from __future__ import annotations

import numpy as np


def clamp_lengths(row_len, S: int) -> np.ndarray:
    return np.clip(np.asarray(row_len, dtype=np.int64), 0, S)


def row_offsets(row_len, S: int) -> np.ndarray:
    """Exclusive prefix sum of the clamped lengths, [B + 1]."""
    lens = clamp_lengths(row_len, S)
    out = np.zeros(lens.size + 1, dtype=np.int64)
    for b, n in enumerate(lens):
        out[b + 1] = out[b] + n
    return out


def pack_thd(x: np.ndarray, row_len) -> np.ndarray:
    """[B, S, ...] -> [T, ...]: the real tokens of each row, rows in order."""
    B, S = x.shape[0], x.shape[1]
    lens = clamp_lengths(row_len, S)
    rows = []
    for b in range(B):
        for s in range(int(lens[b])):
            rows.append(x[b, s])
    if not rows:
        return np.zeros((0,) + x.shape[2:], dtype=x.dtype)
    return np.stack(rows)


def unpack_bshd(y: np.ndarray, row_len, S: int) -> np.ndarray:
    """[T, ...] -> [B, S, ...] with zero padding rows."""
    lens = clamp_lengths(row_len, S)
    x = np.zeros((lens.size, S) + y.shape[1:], dtype=y.dtype)
    t = 0
    for b in range(lens.size):
        for s in range(int(lens[b])):
            x[b, s] = y[t]
            t += 1
    return x
