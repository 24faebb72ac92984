"""3D rotary position embedding over (t, h, w) token positions.

The pages only say that ConvKV resets the memory's RoPE positions
("SoulX-LiveAct", 技术内核); the video DiT's 3D RoPE itself is not printed.
Reading taken (a standard 3D RoPE):
  * the head dim D splits into contiguous parts [t | h | w] of sizes
    D - 4*floor(D/6), 2*floor(D/6), 2*floor(D/6) (44/42/42 for D = 128,
    24/20/20 for D = 64);
  * inside each part, dims (2i, 2i+1) form a pair rotated by the angle
    pos_axis * theta**(-2i / d_axis), theta = 10000;
  * (x0, x1) -> (x0 cos a - x1 sin a, x0 sin a + x1 cos a).
Tokens of a block are in raster order (frame, row, column).
"""
from __future__ import annotations

import numpy as np


def split(D: int) -> tuple[int, int, int]:
    hw = 2 * (D // 6)
    return D - 2 * hw, hw, hw


def freqs(d_axis: int, theta: float = 10000.0) -> np.ndarray:
    i = np.arange(d_axis // 2, dtype=np.float64)
    return theta ** (-2.0 * i / d_axis)


def block_positions(F: int, GH: int, GW: int):
    """(frame, row, column) of each token of one block, raster order."""
    f, h, w = np.meshgrid(np.arange(F), np.arange(GH), np.arange(GW), indexing="ij")
    return f.reshape(-1), h.reshape(-1), w.reshape(-1)


def rotate(x: np.ndarray, t, h, w, theta: float = 10000.0, parts=None) -> np.ndarray:
    """Rotate x [N, ..., D] by per-token positions t, h, w (each [N]); fp64.
    parts: the (t, h, w) dims of the head dim, default split(D)."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    parts = split(D) if parts is None else tuple(parts)
    assert sum(parts) == D and all(d % 2 == 0 for d in parts)
    out = x.copy()
    base = 0
    for pos, d in zip((t, h, w), parts):
        pos = np.asarray(pos, dtype=np.float64).reshape(-1)
        ang = pos[:, None] * freqs(d, theta)[None, :]          # [N, d/2]
        shape = (x.shape[0],) + (1,) * (x.ndim - 2) + (d // 2,)
        c = np.cos(ang).reshape(shape)
        s = np.sin(ang).reshape(shape)
        x0 = x[..., base:base + d:2]
        x1 = x[..., base + 1:base + d:2]
        out[..., base:base + d:2] = x0 * c - x1 * s
        out[..., base + 1:base + d:2] = x0 * s + x1 * c
        base += d
    return out
