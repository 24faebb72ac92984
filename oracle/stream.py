"""Per-block context of the bounded cache, and the chunk attention over it.

PR-Sink ("LiveAnimate", ai-feeds.com, 方法): when block b is generated its
context is the static sink (block 0, kept forever), the dynamic sink (top-k
history blocks by pose similarity to block b's driving pose), the rolling
window (the 3 most recent blocks) and block b itself.

ConvKV ("SoulX-LiveAct", youleyou.com, 技术内核): the context is the
compressed memory (older blocks, conv-compressed, FIFO of fixed length) plus
the exact recent blocks (the window) and the current block.

Readings taken:
  * slot order [sink, dynamic (ascending id), window (oldest first),
    current]; empty slots are dropped;
  * RoPE temporal positions are slot-relative: the s-th exact slot starts at
    t0 = s * F (F latent frames per block), so positions stay bounded however
    long the stream (the page says cache size and per-block latency stay
    constant); ConvKV memory token j sits at (j, 0, 0) and the exact slots
    follow at t0 = n_mem + s * F;
  * a token of a slot at t0 has position (t0 + frame, row, column);
  * FP8 cache: the stored key is the key rotated by its within-block
    position (frame, row, column) in fp32 single roundings, quantised per
    (head, block); the slot's temporal offset t0 is applied after
    dequantisation.  The current block is read through the same format.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import attention, convkv, e4m3, pose, rope


@dataclass
class Context:
    block: int
    blocks: list[int]                 # exact blocks in slot order; last is current
    t0: list[int]                     # temporal base of each exact slot
    mem_tokens: int = 0               # ConvKV memory tokens in front of the exact slots
    dyn_ids: list[int] = field(default_factory=list)
    dyn_scores: list[float] = field(default_factory=list)
    gap: float = np.inf
    tokens_per_block: int = 0

    @property
    def kv_len(self) -> int:
        return self.mem_tokens + len(self.blocks) * self.tokens_per_block


def plan_prsink(cfg, b: int, descs: np.ndarray, query_desc: np.ndarray) -> Context:
    """Context of block b given the descriptors of blocks 0..b-1."""
    F, T, W = cfg.frames_per_block, cfg.tokens_per_block, cfg.window
    sink = [0] if (cfg.static_sink and b >= 1) else []
    window = [j for j in range(max(0, b - W), b) if j not in sink]
    cand = pose.candidates(b, W, cfg.static_sink)
    dyn, dyn_s, gap = [], [], np.inf
    if cand and cfg.dyn_topk > 0:
        sc = pose.cosine_scores(query_desc, descs[cand])
        dyn, dyn_s, gap = pose.select_topk(sc, cand, cfg.dyn_topk)
    blocks = sink + dyn + window + [b]
    return Context(block=b, blocks=blocks, t0=[s * F for s in range(len(blocks))],
                   dyn_ids=dyn, dyn_scores=dyn_s, gap=gap, tokens_per_block=T)


def plan_convkv(cfg, b: int) -> Context:
    F, T, W = cfg.frames_per_block, cfg.tokens_per_block, cfg.window
    blocks = list(range(max(0, b - W), b)) + [b]
    n_evicted = max(0, b - W)
    per = (T - cfg.conv_kernel) // cfg.conv_stride + 1
    n_mem = min(cfg.mem_slots, per * n_evicted)
    return Context(block=b, blocks=blocks,
                   t0=[n_mem + s * F for s in range(len(blocks))],
                   mem_tokens=n_mem, tokens_per_block=T)


def plan_stream(cfg, kps: np.ndarray, n_blocks: int | None = None) -> list[Context]:
    """Contexts of blocks 0..n-1 of a stream with driving poses kps [n, 17, 2]."""
    n = len(kps) if n_blocks is None else n_blocks
    out = []
    if cfg.policy == "convkv":
        return [plan_convkv(cfg, b) for b in range(n)]
    descs = np.stack([pose.descriptor(k) for k in kps[:n]]) if n else np.zeros((0, 34))
    for b in range(n):
        out.append(plan_prsink(cfg, b, descs[:b], descs[b]))
    return out


# ------------------------------------------------------------ value handling
def rope_parts(cfg) -> tuple[int, int, int]:
    """(t, h, w) dims of the head dim: the config's explicit split when it
    gives one (the C ABI takes any even split), else rope.split(D)."""
    dims = getattr(cfg, "rope_dims", None)
    return tuple(dims) if dims else rope.split(cfg.head_dim)


def rotate_within_block_f32(x: np.ndarray, cfg) -> np.ndarray:
    """Key rotated by its within-block (frame, row, column) position using
    fp32 single roundings: each product and the sum/difference rounded once,
    cos/sin rounded to fp32 from fp64.  x [T, H, D] fp32 -> fp32."""
    x = np.asarray(x, dtype=np.float32)
    f, h, w = rope.block_positions(cfg.frames_per_block, cfg.grid_h, cfg.grid_w)
    out = x.copy()
    base = 0
    for pos, d in zip((f, h, w), rope_parts(cfg)):
        ang = pos.astype(np.float64)[:, None] * rope.freqs(d, cfg.rope_theta)[None, :]
        c = np.cos(ang).astype(np.float32)[:, None, :]
        s = np.sin(ang).astype(np.float32)[:, None, :]
        x0 = x[..., base:base + d:2]
        x1 = x[..., base + 1:base + d:2]
        out[..., base:base + d:2] = (x0 * c).astype(np.float32) - (x1 * s).astype(np.float32)
        out[..., base + 1:base + d:2] = (x0 * s).astype(np.float32) + (x1 * c).astype(np.float32)
        base += d
    return out


def fp8_store(x_thd: np.ndarray):
    """Quantise [T, H, D] fp32 per head.  Returns (codes [T,H,D] uint8,
    scales [H] fp32, dequantised fp64 [T, H, D], scaled fp32 values)."""
    T, H, D = x_thd.shape
    codes = np.zeros((T, H, D), np.uint8)
    scaled = np.zeros((T, H, D), np.float32)
    scales = np.zeros(H, np.float32)
    for hh in range(H):
        c, s, y = e4m3.quantize(x_thd[:, hh, :])
        codes[:, hh, :] = c
        scales[hh] = s
        scaled[:, hh, :] = y
    deq = e4m3.decode(codes) * scales[None, :, None].astype(np.float64)
    return codes, scales, deq, scaled


def context_kv(cfg, ctx: Context, kv_of, mem=None):
    """Keys rotated at their full positions and values, over the context.

    kv_of(block) -> (k, v) raw values [T, H', D] (any head subset H').
    mem: (k_mem, v_mem) raw compressed memory [n, H', D] (ConvKV), or None.
    Returns (K [M, H', D], V [M, H', D]) in fp64."""
    f, h, w = rope.block_positions(cfg.frames_per_block, cfg.grid_h, cfg.grid_w)
    ks, vs = [], []
    if ctx.mem_tokens:
        km, vm = mem
        assert km.shape[0] == ctx.mem_tokens
        j = np.arange(ctx.mem_tokens)
        z = np.zeros_like(j)
        ks.append(rope.rotate(km, j, z, z, cfg.rope_theta, rope_parts(cfg)))
        vs.append(np.asarray(vm, dtype=np.float64))
    for blk, t0 in zip(ctx.blocks, ctx.t0):
        k, v = kv_of(blk)
        if cfg.kv_dtype == "e4m3":
            _, _, kd, _ = fp8_store(rotate_within_block_f32(k, cfg))
            _, _, vd, _ = fp8_store(np.asarray(v, dtype=np.float32))
            zero = np.zeros_like(f)
            ks.append(rope.rotate(kd, t0 + zero, zero, zero, cfg.rope_theta, rope_parts(cfg)))
            vs.append(vd)
        else:
            ks.append(rope.rotate(k, t0 + f, h, w, cfg.rope_theta, rope_parts(cfg)))
            vs.append(np.asarray(v, dtype=np.float64))
    return np.concatenate(ks, axis=0), np.concatenate(vs, axis=0)


def chunk_attention(cfg, ctx: Context, q: np.ndarray, kv_of, mem=None, rows=None):
    """Output of the current block's chunk attention.

    q: raw queries [T, H', D] of the current block; rows: optional subset of
    query tokens.  Returns O [len(rows) or T, H', D] in fp64."""
    f, h, w = rope.block_positions(cfg.frames_per_block, cfg.grid_h, cfg.grid_w)
    t0c = ctx.t0[-1]
    if rows is None:
        rows = np.arange(q.shape[0])
    rows = np.asarray(rows)
    qr = rope.rotate(np.asarray(q)[rows], t0c + f[rows], h[rows], w[rows], cfg.rope_theta,
                     rope_parts(cfg))
    K, V = context_kv(cfg, ctx, kv_of, mem)
    out = np.zeros((len(rows), q.shape[1], V.shape[2]))
    for hh in range(q.shape[1]):
        out[:, hh, :] = attention.softmax_attention(qr[:, hh, :], K[:, hh, :], V[:, hh, :],
                                                    cfg.softmax_scale)
    return out


def convkv_memory(cfg, b: int, kv_of, w_kv: np.ndarray):
    """Raw memory (k_mem, v_mem) present when block b is generated.

    kv_of(block) -> raw (k, v) [T, H', D]; w_kv [2, H', D, R] conv weights.
    Only the evicted blocks whose tokens can still be in the FIFO are read."""
    ctx = plan_convkv(cfg, b)
    n_evicted = max(0, b - cfg.window)
    T = cfg.tokens_per_block
    per = (T - cfg.conv_kernel) // cfg.conv_stride + 1
    need = -(-cfg.mem_slots // per) if per else 0
    first = max(0, n_evicted - need)
    km = vm = None
    for e in range(first, n_evicted):
        k, v = kv_of(e)
        ck = bf16_round(convkv.compress(k, w_kv[0], cfg.conv_stride))
        cv = bf16_round(convkv.compress(v, w_kv[1], cfg.conv_stride))
        km = convkv.fifo_append(km, ck, cfg.mem_slots)
        vm = convkv.fifo_append(vm, cv, cfg.mem_slots)
    if km is None:
        return None
    assert km.shape[0] == ctx.mem_tokens
    return km, vm


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 (ties to even) of the fp64 values, via their fp32 value."""
    x32 = np.asarray(x, dtype=np.float64)
    # exact fp64 -> bf16 rounding: round the fp64 significand directly
    b = x32.view(np.uint64) if x32.flags.c_contiguous else np.ascontiguousarray(x32).view(np.uint64)
    # fp64 has 52 fraction bits, bf16 has 7: drop 45 bits with RNE
    drop = np.uint64(45)
    half = np.uint64(1) << np.uint64(44)
    lsb = (b >> drop) & np.uint64(1)
    r = ((b + (half - np.uint64(1)) + lsb) >> drop) << drop
    return r.view(np.float64).reshape(np.shape(x))
