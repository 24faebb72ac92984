"""The decomposition behind the tensor-core attention's split query tiles.

When a head has an odd number of 128-row query tiles, the kernel runs that
tile once per context slot and a merge pass combines the pieces: each piece
keeps, per row, its running max m_s (log2 units), its sum l_s of
2^(x - m_s) and its unnormalised output O_s = sum 2^(x - m_s) v, and the
merge forms O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s with
M = max_s m_s.  Here that formula, applied to per-slot pieces computed in
fp64 on the CPU, must reproduce the oracle's one-pass softmax over the
whole context ("LiveAnimate" (ai-feeds.com), 方法: one softmax over the
bounded context), including rows whose scores differ by far more than the
fp32 exponent range between slots, and a piece whose keys are all masked.
"""
import numpy as np

from oracle import attention, rope
from oracle import stream as ostream
from synth import C2_MID, gen

from . import harness as H


def _piece(qr, K, V, scale):
    """(m, l, O) of one slot: base-2 running max, sum and unnormalised output."""
    x = (qr @ K.T) * (scale / np.log(2.0))
    m = x.max(axis=1)
    p = np.exp2(x - m[:, None])
    return m, p.sum(axis=1), p @ V


def _merge(pieces):
    M = np.max([m for m, _, _ in pieces], axis=0)
    num = sum(np.exp2(m - M)[:, None] * o for m, _, o in pieces)
    den = sum(np.exp2(m - M) * l for m, l, _ in pieces)
    return num / den[:, None]


def test_per_slot_pieces_merge_to_the_oracle():
    sc = C2_MID.with_(grid_h=13, grid_w=15, num_heads=2)        # 390 tokens: an odd 4th tile
    b = 11
    ctx = ostream.plan_stream(sc, gen.poses(sc, n_blocks=b + 1), b + 1)[b]
    vals = H.Values(sc)
    kv_of = vals.kv_of(0, lambda blk: 0)
    q = vals.get(0, b, 0, "q")
    T = sc.tokens_per_block
    rows = np.arange(384, T)                                    # the odd tile's rows
    ref = ostream.chunk_attention(sc, ctx, q, kv_of, rows=rows)
    f, hh, ww = rope.block_positions(sc.frames_per_block, sc.grid_h, sc.grid_w)
    qr = rope.rotate(np.asarray(q)[rows], ctx.t0[-1] + f[rows], hh[rows], ww[rows], sc.rope_theta,
                     ostream.rope_parts(sc))
    K, V = ostream.context_kv(sc, ctx, kv_of)
    for h in range(sc.num_heads):
        pieces = [_piece(qr[:, h], K[s * T:(s + 1) * T, h], V[s * T:(s + 1) * T, h], sc.softmax_scale)
                  for s in range(len(ctx.blocks))]
        got = _merge(pieces)
        assert np.abs(got - ref[:, h]).max() < 1e-12
        # a single piece is not the answer: the merge matters
        assert np.abs(pieces[-1][2] / pieces[-1][1][:, None] - ref[:, h]).max() > 1e-2


def test_merge_far_apart_maxima_and_an_empty_piece():
    rng = np.random.default_rng(3)
    D = 64
    q = rng.standard_normal((5, D))
    ks = [rng.standard_normal((40, D)) * a for a in (0.1, 1.0, 30.0)]   # scores 0.1x .. 30x apart
    vs = [rng.standard_normal((40, D)) for _ in ks]
    scale = D ** -0.5
    ref = attention.softmax_attention(q, np.concatenate(ks), np.concatenate(vs), scale)
    pieces = [_piece(q, k, v, scale) for k, v in zip(ks, vs)]
    # an empty piece (every key past its slot's end) carries m = -inf, l = 0, O = 0
    pieces.append((np.full(5, -np.inf), np.zeros(5), np.zeros((5, D))))
    with np.errstate(invalid="ignore"):
        got = _merge(pieces)
    assert np.abs(got - ref).max() < 1e-12
