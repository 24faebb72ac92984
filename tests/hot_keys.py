"""Inputs that move the attention's running max at every slot.

Every query row gets 16 in dim dt-2 and 0 in dim dt-1 (the lowest-frequency
temporal pair of the 3D RoPE: it turns by under 0.01 rad over short
streams).  The "hot" key of block b is beta_b * e_{dt-2}, so its score is
scale * log2(e) * 16 * beta_b, about 3 + 9.5 * b in log2 units, whatever
the row.  Along a context in ascending block order the row max therefore
grows by more than 8 (log2 units) at every slot.  Every block's V gets one
element of 8, larger than any other, so an e4m3 cache gives every block the
same V scale.  All values set are bf16-exact, so the device and the oracle
see the same numbers.
"""
from __future__ import annotations

import numpy as np

from oracle import stream as ostream

ALPHA = 16.0
V_PIN = 8.0


def _bf16(x: float) -> float:
    """x rounded to bf16 (round to nearest even), as a Python float."""
    u = np.array([x], np.float32).view(np.uint32)[0]
    u = (int(u) + 0x7FFF + ((int(u) >> 16) & 1)) & 0xFFFF0000
    return float(np.array([u], np.uint32).view(np.float32)[0])


class HotKeys:
    def __init__(self, sc):
        self.T = sc.tokens_per_block
        self.slow = ostream.rope_parts(sc)[0] - 2
        self.c = sc.softmax_scale / np.log(2.0)            # score -> log2 units

    def hot_token(self, b: int) -> int:
        return (97 * b + 11) % self.T

    def beta(self, b: int) -> float:
        return _bf16((3.0 + 9.5 * b) / (self.c * ALPHA))

    def modify(self, b: int, q, k, v):
        """The change, in place, on torch (device, bf16) or NumPy arrays [T, H, D]."""
        q[:, :, self.slow] = ALPHA
        q[:, :, self.slow + 1] = 0.0
        t = self.hot_token(b)
        k[t] = 0.0
        k[t, :, self.slow] = self.beta(b)
        v[(t + 1) % self.T, :, 0] = V_PIN
        return q, k, v

    def kv_of(self, vals, layer=0, step=0):
        """Oracle-side (k, v) of a block: the seeded values, changed."""
        def f(blk):
            z = np.zeros_like(vals.get(layer, blk, step, "q"))
            _, k, v = self.modify(blk, z, vals.get(layer, blk, step, "k").copy(),
                                  vals.get(layer, blk, step, "v").copy())
            return k, v
        return f

    def q_of(self, vals, b, layer=0, step=0):
        q = vals.get(layer, b, step, "q").copy()
        z = np.zeros_like(q)
        return self.modify(b, q, z, z.copy())[0]
