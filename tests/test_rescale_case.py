"""The hot-key stream of the GPU rescale test has the power it claims.

An online softmax in fp64 with the tensor-core kernel's lazy running max
(128-key tiles per slot, the max moved only when a tile's row sum passes
2^8 and its max grew by more than 8 in log2 units, then O and the row sum
rescaled) matches the oracle's one-pass softmax on that stream.  The same
loop with either rescale left out misses it by far more than the bf16
bounds the GPU test applies, so a kernel with such a mistake fails there.
"""
import numpy as np
import pytest

from oracle import rope
from oracle import stream as ostream
from synth import C2_MID, gen

from . import harness as H
from .hot_keys import HotKeys


def _lazy_softmax(qr, K, V, scale, T, n_slots, rescale_o=True, rescale_l=True):
    """Rows of qr [R, D] against K, V [n_slots * T, D]; fp64."""
    x_all = (qr @ K.T) * (scale / np.log(2.0))               # log2 units
    R = qr.shape[0]
    m = np.full(R, -np.inf)
    l = np.zeros(R)
    O = np.zeros((R, V.shape[1]))
    first = True
    for s in range(n_slots):
        for a in range(s * T, (s + 1) * T, 128):
            b = min(a + 128, (s + 1) * T)
            x = x_all[:, a:b]
            p = np.exp2(x - m[:, None])
            move = np.ones(R, bool) if first else (p.sum(1) > 256.0)
            mx = x.max(1)
            move &= mx > m + 8.0
            alpha = np.where(move, np.exp2(m - np.where(move, mx, m)), 1.0)
            if not first:
                if rescale_o:
                    O *= alpha[:, None]
                if rescale_l:
                    l *= alpha
            m = np.where(move, mx, m)
            p = np.exp2(x - m[:, None])
            O += p @ V[a:b]
            l += p.sum(1)
            first = False
    return O / l[:, None]


@pytest.mark.parametrize("b", [9, 11])
def test_hot_key_stream_needs_both_rescales(b):
    sc = C2_MID.with_(grid_h=13, grid_w=15, num_heads=2)
    hk = HotKeys(sc)
    ctx = ostream.plan_stream(sc, gen.poses(sc, n_blocks=b + 1), b + 1)[b]
    assert list(ctx.blocks) == sorted(ctx.blocks)
    vals = H.Values(sc)
    q = hk.q_of(vals, b)
    ref = ostream.chunk_attention(sc, ctx, q, hk.kv_of(vals))
    f, hh, ww = rope.block_positions(sc.frames_per_block, sc.grid_h, sc.grid_w)
    qr = rope.rotate(q, ctx.t0[-1] + f, hh, ww, sc.rope_theta, ostream.rope_parts(sc))
    K, V = ostream.context_kv(sc, ctx, hk.kv_of(vals))
    T, n = sc.tokens_per_block, len(ctx.blocks)
    moved = 0
    for h in range(sc.num_heads):
        args = (qr[:, h], K[:, h], V[:, h], sc.softmax_scale, T, n)
        good = _lazy_softmax(*args)
        H.compare(good[:, None], ref[:, h:h + 1], "f32", f"head {h} lazy max")
        for kw in (dict(rescale_o=False), dict(rescale_l=False)):
            bad = _lazy_softmax(*args, **kw)
            d = np.abs(bad - ref[:, h])
            assert d.mean() > 10 * H.TOL["bf16"]["mean_abs"], (h, kw, d.mean())
            moved += 1
    assert moved == 2 * sc.num_heads
