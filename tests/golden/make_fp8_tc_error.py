"""Expected error of the e4m3 tensor-core attention against the oracle, by
simulation; writes fp8_tc_error.txt next to this file.

The oracle attends over the dequantised e4m3 cache with exact queries and
exact probabilities.  The tensor-core path ("SoulX-LiveAct", 技术内核 and
上手实践指南: FP8 attention over an FP8 KV cache) also rounds the rotated
queries and the probabilities to e4m3 before its two products.  This script
models only those two extra roundings, in fp64 NumPy on top of the oracle's
own storage functions (oracle.stream.fp8_store, rotate_within_block_f32,
oracle.rope), and reports how far that moves the output from the oracle's:
the relative-L2, max-abs and mean-abs figures that set the e4m3 tensor-core
tolerance of the GPU parity tests.

Model of the kernel's arithmetic (the reading of the FP8 attention):
  * query row of a token: one scale per (head, token), the largest norm of
    its rotation pairs / 448 (a turn keeps pair norms, so no slot's rotated
    copy saturates); codes = e4m3(turned q * 448 / that norm);
  * scores = codes_q . codes_k * q_scale * k_scale(slot) (exact products);
  * base-2 online softmax over 128-key tiles in slot order with a lazy
    running max m: set from the first tile; raised to a tile's max only when
    the tile's probabilities sum above 2^8 and the max grew by more than 8
    (then the accumulated output and sum are rescaled);
  * P = e4m3(2^(x - m) * v_scale(slot) / v_max) per element (<= 256, no
    saturation); O accumulates P . codes_v; the row sum takes the unrounded
    2^(x - m); O = v_max * O / sum.

Usage: python tests/golden/make_fp8_tc_error.py   (about a minute)
"""
from __future__ import annotations

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import e4m3, rope, stream  # noqa: E402
from synth import C5_FP8, gen  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "fp8_tc_error.txt")
TILE = 128


def _values(sc, block, which, heads):
    T, H, D = sc.tokens_per_block, sc.num_heads, sc.head_dim
    idx = ((np.arange(T)[:, None, None] * H + np.asarray(heads)[None, :, None]) * D
           + np.arange(D)[None, None, :]).reshape(-1).astype(np.uint64)
    key = gen.qkv_key(sc, 0, block, 0, which)
    return gen.tensor_np(key, None, "bf16", index_map=idx).reshape(T, len(heads), D)


def simulate(sc=C5_FP8, block=40, heads=(0, 21), n_rows=64, rounding=True):
    """(oracle O, simulated tensor-core O) for `heads` x n_rows query rows of
    one steady-state call of the stream `sc`.  rounding=False keeps the
    queries and probabilities exact (the simulation must then reproduce the
    oracle)."""
    heads = list(heads)
    kps = gen.poses(sc, n_blocks=block + 1)
    ctx = stream.plan_stream(sc, kps, block + 1)[block]
    kv = {b: (_values(sc, b, "k", heads), _values(sc, b, "v", heads)) for b in ctx.blocks}
    q = _values(sc, block, "q", heads)
    T, D = sc.tokens_per_block, sc.head_dim
    rows = np.linspace(0, T - 1, n_rows).astype(int)
    o_ref = stream.chunk_attention(sc, ctx, q, lambda b: kv[b], rows=rows)

    parts = stream.rope_parts(sc)
    f, h, w = rope.block_positions(sc.frames_per_block, sc.grid_h, sc.grid_w)
    stored = {}
    for b in ctx.blocks:
        kc, ks, _, _ = stream.fp8_store(stream.rotate_within_block_f32(kv[b][0], sc))
        vc, vs, _, _ = stream.fp8_store(np.asarray(kv[b][1], np.float32))
        stored[b] = (e4m3.decode(kc), ks.astype(np.float64), e4m3.decode(vc), vs.astype(np.float64))
    t0c = ctx.t0[-1]
    log2e = 1.0 / np.log(2.0)
    o_sim = np.zeros_like(o_ref)
    for hi in range(len(heads)):
        qr = np.asarray(q[rows, hi, :], np.float64)                     # [R, D]
        pair_norm = np.sqrt(qr[:, 0::2] ** 2 + qr[:, 1::2] ** 2).max(axis=1)
        q_scale = np.where(pair_norm > 0, pair_norm / 448.0, 1.0)
        v_max = max(stored[b][3][hi] for b in ctx.blocks)
        m = None
        acc = np.zeros((len(rows), D))
        l = np.zeros(len(rows))
        for b, t0 in zip(ctx.blocks, ctx.t0):
            kcode, ks, vcode, vs = stored[b]
            turned = rope.rotate(qr, t0c - t0 + f[rows], h[rows], w[rows], sc.rope_theta, parts)
            qcode = turned / q_scale[:, None]
            if rounding:
                qcode = e4m3.decode(e4m3.encode(qcode))
            c = sc.softmax_scale * log2e * q_scale * ks[hi]
            r = vs[hi] / v_max
            for a in range(0, T, TILE):
                x = (qcode @ kcode[a:a + TILE, hi, :].T) * c[:, None]   # log2 units
                tmax = x.max(axis=1)
                if m is None:
                    m = tmax.copy()
                else:
                    over = (np.exp2(x - m[:, None]) * r).sum(axis=1) > 256.0
                    grow = over & (tmax > m + 8.0)
                    alpha = np.where(grow, np.exp2(m - tmax), 1.0)
                    acc *= alpha[:, None]
                    l *= alpha
                    m = np.where(grow, tmax, m)
                p = np.exp2(x - m[:, None])
                pq = e4m3.decode(e4m3.encode(p * r)) if rounding else p * r
                acc += pq @ vcode[a:a + TILE, hi, :]
                l += p.sum(axis=1)
        o_sim[:, hi, :] = v_max * acc / l[:, None]
    return o_ref, o_sim


def errors(o_ref, o_sim):
    d = np.abs(o_sim - o_ref)
    return {"rel_l2": float(np.linalg.norm(d) / np.linalg.norm(o_ref)),
            "max_abs": float(d.max()), "mean_abs": float(d.mean())}


def main():
    heads, n_rows = (0, 13, 26, 39), 256
    e = errors(*simulate(heads=heads, n_rows=n_rows))
    with open(OUT, "w") as fh:
        fh.write("# e4m3 tensor-core attention vs the oracle, simulated: FP8 stress stream\n"
                 "# (40 heads x 128, 4680 tokens, top-4 dynamic sink, 42120 keys), block 40,\n"
                 f"# heads {list(heads)}, {n_rows} query rows spread over the block.\n"
                 "# Written by tests/golden/make_fp8_tc_error.py (oracle/ and synth/ only).\n")
        for k, v in e.items():
            fh.write(f"{k} {v:.6e}\n")
    print(e)


if __name__ == "__main__":
    main()
