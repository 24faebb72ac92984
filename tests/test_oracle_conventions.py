"""Pins for the oracle's position and storage conventions, each against a
hand-written expectation rather than the oracle's own helpers.

* Raster token order inside a block ("LiveAnimate", 方法: blocks of latent
  frames; reading: token = frame * rows * cols + row * cols + col).
* PR-Sink slot positions: the s-th slot starts at t0 = s * F.
* ConvKV memory positions ("SoulX-LiveAct", 技术内核: the compressed memory's
  RoPE positions are reset): memory token j at (j, 0, 0), the exact slots
  after it at t0 = n_mem + s * F.
* The e4m3 cache ("SoulX-LiveAct", 上手实践指南: FP8 KV cache): the key is
  turned by its within-block position, quantised, and turned by the slot's
  temporal base after dequantisation.  When every stored value is exactly
  representable the e4m3 branch must reduce to the bf16 branch.

The rotations here are written as complex multiplications at positions typed
out by hand, so a wrong index order, a memory token placed at (j, j, j), or a
key turned twice by its within-block position fails.
"""
import numpy as np

from oracle import e4m3, rope, stream
from synth import C2_MID, C4_CONVKV, C5_FP8


def _turn(x, positions, parts, theta=10000.0):
    """x [N, D] turned token by token: pair (2i, 2i+1) of an axis part of
    size d is the complex number x_2i + i x_2i+1 times exp(i pos theta^(-2i/d))."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    for n, pos in enumerate(positions):
        base = 0
        for p, d in zip(pos, parts):
            for i in range(d // 2):
                z = complex(x[n, base + 2 * i], x[n, base + 2 * i + 1])
                z *= np.exp(1j * p * theta ** (-2.0 * i / d))
                out[n, base + 2 * i], out[n, base + 2 * i + 1] = z.real, z.imag
            base += d
    return out


def _attend(q, k, v, scale):
    s = np.array([[np.dot(a, b) * scale for b in k] for a in q])
    p = np.exp(s - s.max(axis=1, keepdims=True))
    return (p @ v) / p.sum(axis=1, keepdims=True)


def test_block_positions_raster_order():
    f, h, w = rope.block_positions(2, 2, 3)
    hand = [(0, 0, 0), (0, 0, 1), (0, 0, 2), (0, 1, 0), (0, 1, 1), (0, 1, 2),
            (1, 0, 0), (1, 0, 1), (1, 0, 2), (1, 1, 0), (1, 1, 1), (1, 1, 2)]
    assert list(zip(f.tolist(), h.tolist(), w.tolist())) == hand


def test_prsink_context_positions_hand_listed():
    """Context keys and the output of a tiny PR-Sink call, positions typed out:
    2 frames of 1 x 2 tokens per block, slots [0, 2, 4, 5, 6, 7] at
    t0 = 0, 2, 4, 6, 8, 10."""
    cfg = C2_MID.with_(num_heads=1, head_dim=12, frames_per_block=2, grid_h=1, grid_w=2,
                       rope_dims=(4, 4, 4))
    ctx = stream.Context(block=7, blocks=[0, 2, 4, 5, 6, 7], t0=[0, 2, 4, 6, 8, 10],
                         tokens_per_block=4)
    rng = np.random.default_rng(0)
    kv = {b: (rng.normal(size=(4, 1, 12)), rng.normal(size=(4, 1, 12))) for b in ctx.blocks}
    q = rng.normal(size=(4, 1, 12))
    # token order in a block: (f, row, col) = (0,0,0), (0,0,1), (1,0,0), (1,0,1)
    within = [(0, 0, 0), (0, 0, 1), (1, 0, 0), (1, 0, 1)]
    pos = [(t0 + a, b, c) for t0 in (0, 2, 4, 6, 8, 10) for (a, b, c) in within]
    K_hand = _turn(np.concatenate([kv[b][0][:, 0] for b in ctx.blocks]), pos, (4, 4, 4))
    V_hand = np.concatenate([kv[b][1][:, 0] for b in ctx.blocks])
    K, V = stream.context_kv(cfg, ctx, lambda b: kv[b])
    np.testing.assert_allclose(K[:, 0], K_hand, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(V[:, 0], V_hand)
    q_hand = _turn(q[:, 0], [(10 + a, b, c) for (a, b, c) in within], (4, 4, 4))
    o_hand = _attend(q_hand, K_hand, V_hand, cfg.softmax_scale)
    o = stream.chunk_attention(cfg, ctx, q, lambda b: kv[b])
    np.testing.assert_allclose(o[:, 0], o_hand, rtol=0, atol=1e-12)


def test_convkv_memory_positions_hand_listed():
    """ConvKV with 3 memory tokens: memory at (0,0,0), (1,0,0), (2,0,0); the
    exact blocks 2..5 (1 frame of 2 x 2 tokens) at t0 = 3, 4, 5, 6."""
    cfg = C4_CONVKV.with_(num_heads=1, head_dim=12, frames_per_block=1, grid_h=2, grid_w=2,
                          conv_kernel=2, conv_stride=2, mem_slots=3, rope_dims=(4, 4, 4))
    ctx = stream.plan_convkv(cfg, 5)
    assert ctx.blocks == [2, 3, 4, 5] and ctx.mem_tokens == 3 and ctx.t0 == [3, 4, 5, 6]
    rng = np.random.default_rng(1)
    kv = {b: (rng.normal(size=(4, 1, 12)), rng.normal(size=(4, 1, 12))) for b in ctx.blocks}
    km, vm = rng.normal(size=(3, 1, 12)), rng.normal(size=(3, 1, 12))
    q = rng.normal(size=(4, 1, 12))
    within = [(0, 0, 0), (0, 0, 1), (0, 1, 0), (0, 1, 1)]
    pos = [(0, 0, 0), (1, 0, 0), (2, 0, 0)] + \
          [(t0 + a, b, c) for t0 in (3, 4, 5, 6) for (a, b, c) in within]
    keys = np.concatenate([km[:, 0]] + [kv[b][0][:, 0] for b in ctx.blocks])
    K_hand = _turn(keys, pos, (4, 4, 4))
    V_hand = np.concatenate([vm[:, 0]] + [kv[b][1][:, 0] for b in ctx.blocks])
    K, V = stream.context_kv(cfg, ctx, lambda b: kv[b], mem=(km, vm))
    np.testing.assert_allclose(K[:, 0], K_hand, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(V[:, 0], V_hand)
    q_hand = _turn(q[:, 0], [(6 + a, b, c) for (a, b, c) in within], (4, 4, 4))
    o = stream.chunk_attention(cfg, ctx, q, lambda b: kv[b], mem=(km, vm))
    np.testing.assert_allclose(o[:, 0], _attend(q_hand, K_hand, V_hand, cfg.softmax_scale),
                               rtol=0, atol=1e-12)


def _representable_block(rng, T, H, D, s, cfg):
    """Raw K (fp32) whose within-block turn lands on e4m3 codes x s, with a
    code of 448 in every head (so amax / 448 = s), and V = codes x s exactly."""
    finite = np.array([c for c in range(0x7F)] + [c | 0x80 for c in range(0x7F)], np.uint8)

    def codes():
        c = rng.choice(finite, size=(T, H, D))
        c[0, :, 5] = 0x7E                      # 448 in every head
        return c

    k_turned = e4m3.decode(codes()) * s                                   # target K'
    f, h, w = rope.block_positions(cfg.frames_per_block, cfg.grid_h, cfg.grid_w)
    k_raw = rope.rotate(k_turned, -f, -h, -w, cfg.rope_theta, stream.rope_parts(cfg))
    v = (e4m3.decode(codes()) * s).astype(np.float32)
    return k_raw.astype(np.float32), v, k_turned


def _e4m3_and_bf16_branches():
    """Context keys and outputs of both branches over representable blocks."""
    cfg8 = C5_FP8.with_(num_heads=2, frames_per_block=2, grid_h=3, grid_w=4)   # T = 24
    cfg16 = cfg8.with_(kv_dtype="bf16")
    T, H, D = cfg8.tokens_per_block, 2, 128
    rng = np.random.default_rng(2)
    ctx = stream.Context(block=9, blocks=[0, 3, 5, 6, 7, 8, 9],
                         t0=[0, 2, 4, 6, 8, 10, 12], tokens_per_block=T)
    kv, turned = {}, {}
    for b in ctx.blocks:
        k, v, turned[b] = _representable_block(rng, T, H, D, np.float64(2.0 ** -5), cfg8)
        kv[b] = (k, v)
    q = rng.normal(size=(T, H, D)).astype(np.float32)
    out = {}
    for name, cfg in (("e4m3", cfg8), ("bf16", cfg16)):
        K, V = stream.context_kv(cfg, ctx, lambda b: kv[b])
        out[name] = (K, V, stream.chunk_attention(cfg, ctx, q, lambda b: kv[b]))
    return cfg8, kv, turned, out


def test_e4m3_branch_reduces_to_bf16_branch_when_representable():
    cfg8, kv, turned, out = _e4m3_and_bf16_branches()
    for b, (k, _) in kv.items():
        # the stored form is exact: within-block turn, quantise, dequantise
        _, _, deq, _ = stream.fp8_store(stream.rotate_within_block_f32(k, cfg8))
        np.testing.assert_allclose(deq, turned[b], rtol=0, atol=1e-6 * np.abs(turned[b]).max())
    (K8, V8, o8), (K16, V16, o16) = out["e4m3"], out["bf16"]
    np.testing.assert_array_equal(V8, V16)
    np.testing.assert_allclose(K8, K16, rtol=0, atol=1e-6 * np.abs(K16).max())
    np.testing.assert_allclose(o8, o16, rtol=0, atol=1e-5)


def test_e4m3_pin_catches_a_key_turned_twice(monkeypatch):
    """Plant the mistake in the oracle: the e4m3 branch turns the key by its
    within-block position twice.  The pin above must then fail by far."""
    once = stream.rotate_within_block_f32
    monkeypatch.setattr(stream, "rotate_within_block_f32", lambda x, cfg: once(once(x, cfg), cfg))
    _, _, _, out = _e4m3_and_bf16_branches()
    assert np.abs(out["e4m3"][2] - out["bf16"][2]).max() > 1e-2
