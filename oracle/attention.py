"""Dense softmax attention, fp64.

"LiveAnimate" (ai-feeds.com), 方法: the DiT is block-causal, each time block
depending only on the reference and on earlier generated blocks.  Reading
taken: inside a block there is no mask; the context holds only earlier
blocks plus the current one, so there is nothing to mask at all.  The
output is the plain definition O = softmax(scale * Q K^T) V, with no online
softmax or blocking.
"""
from __future__ import annotations

import numpy as np


def softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """q [N, D], k [M, D], v [M, Dv] -> [N, Dv] in fp64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = (q @ k.T) * scale
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    return (p @ v) / p.sum(axis=1, keepdims=True)
