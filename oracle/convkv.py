"""ConvKV memory: strided depthwise Conv1d compression into a fixed FIFO.

"Soul App开源实时数字人生成框架SoulX-LiveAct详解" (youleyou.com), 技术内核:
recent frames keep exact K/V; older K/V are compressed by a 1D convolution,
compression ratio up to 5:1, into fixed-length memory whose RoPE positions
are reset.

Readings taken:
  * depthwise over the H*D channels, kernel 5, stride 5, no padding, no bias,
    cross-correlation order (output j reads tokens 5j .. 5j+4), separate
    weights for K and V, applied to the raw (un-rotated) K;
  * output rounded to bf16 (the cache's storage type);
  * the memory is token-granular FIFO: it keeps the newest `cap` compressed
    tokens in chronological order;
  * reset positions: memory token j (0 = oldest kept) has t = j, h = w = 0.
"""
from __future__ import annotations

import numpy as np


def compress(x: np.ndarray, w: np.ndarray, stride: int) -> np.ndarray:
    """x [T, H, D], w [H, D, R] -> [(T - R) // stride + 1, H, D] in fp64."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T = x.shape[0]
    R = w.shape[-1]
    n_out = (T - R) // stride + 1
    out = np.zeros((n_out,) + x.shape[1:], dtype=np.float64)
    for r in range(R):
        out += w[None, :, :, r] * x[r: r + stride * (n_out - 1) + 1: stride]
    return out


def fifo_append(mem: np.ndarray | None, new: np.ndarray, cap: int) -> np.ndarray:
    """Append `new` [m, H, D] after `mem` [n, H, D]; keep the newest cap tokens."""
    cat = new if mem is None or mem.shape[0] == 0 else np.concatenate([mem, new], axis=0)
    return cat[-cap:] if cat.shape[0] > cap else cat
