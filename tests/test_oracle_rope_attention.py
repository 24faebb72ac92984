"""Pins for the oracle's 3D RoPE and dense attention."""
import numpy as np
import pytest
import torch
from scipy.special import softmax as sp_softmax

from oracle import attention, rope, stream
from synth import C1_TINY, C2_MID, gen


def test_split_sizes():
    # t/h/w splits of the head dim used by the workloads: t24/h20/w20 (D=64),
    # t44/h42/w42 (D=128)
    assert rope.split(64) == (24, 20, 20)
    assert rope.split(128) == (44, 42, 42)


def _rotate_complex(x, t, h, w, theta=10000.0, parts=None):
    """Independent formulation: each (2i, 2i+1) pair is a complex number
    multiplied by exp(i * pos * theta^(-2i/d))."""
    D = x.shape[-1]
    out = np.empty_like(x, dtype=np.float64)
    base = 0
    for pos, d in zip((t, h, w), parts or rope.split(D)):
        z = x[..., base:base + d:2] + 1j * x[..., base + 1:base + d:2]
        i = np.arange(d // 2)
        ang = np.asarray(pos, dtype=np.float64)[:, None] * np.power(theta, -2.0 * i / d)[None, :]
        z = z * np.exp(1j * ang)
        out[..., base:base + d:2] = z.real
        out[..., base + 1:base + d:2] = z.imag
        base += d
    return out


def test_rotate_matches_complex_multiplication():
    rng = np.random.default_rng(0)
    for D in (12, 64, 128):
        x = rng.normal(size=(37, D))
        t, h, w = (rng.integers(0, 60, size=37) for _ in range(3))
        np.testing.assert_allclose(rope.rotate(x, t, h, w), _rotate_complex(x, t, h, w),
                                   rtol=0, atol=1e-12)


@pytest.mark.parametrize("parts", [(72, 28, 28), (42, 44, 42), (70, 30, 28), (128, 0, 0)])
def test_rotate_explicit_split_matches_complex_multiplication(parts):
    # the C ABI takes any even (t, h, w) split of the head dim
    rng = np.random.default_rng(1)
    x = rng.normal(size=(29, 128))
    t, h, w = (rng.integers(0, 60, size=29) for _ in range(3))
    np.testing.assert_allclose(rope.rotate(x, t, h, w, parts=parts),
                               _rotate_complex(x, t, h, w, parts=parts), rtol=0, atol=1e-12)
    # only the temporal part moves when h = w = 0
    z = np.zeros_like(t)
    y = rope.rotate(x, t, z, z, parts=parts)
    np.testing.assert_array_equal(y[:, parts[0]:], x[:, parts[0]:])


def test_rotate_closed_form_small():
    # D = 12 -> parts of 4/4/4, freqs (1, 0.01) in each part.  The all-ones
    # vector at (t, h, w) = (1, 2, 3): pair (0,1) turns by 1 rad,
    # pair (2,3) by 0.01 rad, (4,5) by 2, (6,7) by 0.02, (8,9) by 3, (10,11) by 0.03.
    x = np.ones((1, 12))
    y = rope.rotate(x, [1], [2], [3])[0]
    for pair, a in enumerate([1.0, 0.01, 2.0, 0.02, 3.0, 0.03]):
        assert abs(y[2 * pair] - (np.cos(a) - np.sin(a))) < 1e-15
        assert abs(y[2 * pair + 1] - (np.sin(a) + np.cos(a))) < 1e-15


def test_rotation_invariants():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(50, 128))
    t, h, w = (rng.integers(0, 4000, size=50) for _ in range(3))
    y = rope.rotate(x, t, h, w)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    z = np.zeros(50, dtype=int)
    np.testing.assert_array_equal(rope.rotate(x, z, z, z), x)


def test_relative_position_identity():
    """<R(p)q, R(p')k> = <R(p - p' + c) q, R(c) k> for any c: the score depends
    only on the position difference (so the kernel can move the slot's
    temporal offset to the query side)."""
    rng = np.random.default_rng(2)
    q = rng.normal(size=(20, 128))
    k = rng.normal(size=(20, 128))
    pq = [rng.integers(0, 100, size=20) for _ in range(3)]
    pk = [rng.integers(0, 100, size=20) for _ in range(3)]
    direct = np.sum(rope.rotate(q, *pq) * rope.rotate(k, *pk), axis=1)
    c = [rng.integers(0, 7, size=20) for _ in range(3)]
    moved = np.sum(rope.rotate(q, *(a - b + cc for a, b, cc in zip(pq, pk, c)))
                   * rope.rotate(k, *c), axis=1)
    np.testing.assert_allclose(direct, moved, rtol=0, atol=1e-11)


def test_attention_matches_torch_sdpa_and_scipy():
    rng = np.random.default_rng(3)
    q = rng.normal(size=(33, 64))
    k = rng.normal(size=(70, 64))
    v = rng.normal(size=(70, 64))
    got = attention.softmax_attention(q, k, v, 0.125)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        scale=0.125)[0].numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    p = sp_softmax(q @ k.T * 0.125, axis=1)
    np.testing.assert_allclose(got, p @ v, rtol=0, atol=1e-12)


def test_attention_uniform_and_permutation():
    rng = np.random.default_rng(4)
    k = rng.normal(size=(40, 16))
    v = rng.normal(size=(40, 16))
    out = attention.softmax_attention(np.zeros((3, 16)), k, v, 1.0)
    np.testing.assert_allclose(out, np.broadcast_to(v.mean(0), (3, 16)), atol=1e-14)
    q = rng.normal(size=(5, 16))
    perm = rng.permutation(40)
    np.testing.assert_allclose(attention.softmax_attention(q, k, v, 0.3),
                               attention.softmax_attention(q, k[perm], v[perm], 0.3), atol=1e-13)


def _kv_source(cfg, layer=0, step=0):
    def kv_of(b):
        T, H, D = cfg.tokens_per_block, cfg.num_heads, cfg.head_dim
        k = gen.tensor_np(gen.qkv_key(cfg, layer, b, step, "k"), (T, H, D), cfg.qkv_dtype)
        v = gen.tensor_np(gen.qkv_key(cfg, layer, b, step, "v"), (T, H, D), cfg.qkv_dtype)
        return k, v
    return kv_of


def test_chunk_attention_zero_query_is_mean_of_context_values():
    cfg = C1_TINY
    kps = gen.poses(cfg)
    ctx = stream.plan_stream(cfg, kps)[12]
    kv_of = _kv_source(cfg)
    q = np.zeros((cfg.tokens_per_block, cfg.num_heads, cfg.head_dim))
    out = stream.chunk_attention(cfg, ctx, q, kv_of)
    V = np.concatenate([kv_of(b)[1] for b in ctx.blocks], axis=0).astype(np.float64)
    assert V.shape[0] == ctx.kv_len == 384
    np.testing.assert_allclose(out, np.broadcast_to(V.mean(0), out.shape), atol=1e-13)


def test_chunk_attention_shift_and_slot_permutation_invariance():
    """Adding a constant to every temporal position, or permuting slots
    together with their positions, leaves the output unchanged."""
    cfg = C1_TINY
    kps = gen.poses(cfg)
    ctx = stream.plan_stream(cfg, kps)[10]
    kv_of = _kv_source(cfg)
    q = gen.tensor_np(gen.qkv_key(cfg, 0, 10, 0, "q"), (64, 2, 64), "f32")
    base = stream.chunk_attention(cfg, ctx, q, kv_of)
    shifted = stream.Context(**{**ctx.__dict__, "t0": [t + 5 for t in ctx.t0]})
    np.testing.assert_allclose(stream.chunk_attention(cfg, shifted, q, kv_of), base, atol=1e-12)
    perm = [2, 0, 1, 3, 4, 5][:len(ctx.blocks) - 1] + [len(ctx.blocks) - 1]
    permuted = stream.Context(**{**ctx.__dict__,
                                 "blocks": [ctx.blocks[i] for i in perm],
                                 "t0": [ctx.t0[i] for i in perm]})
    np.testing.assert_allclose(stream.chunk_attention(cfg, permuted, q, kv_of), base, atol=1e-12)


def test_chunk_attention_reduces_to_library_attention_without_rope():
    """One slot at t0 = 0 of a 1x1x1 block: every position is 0, RoPE is the
    identity and the result is torch's dense attention."""
    cfg = C1_TINY.with_(frames_per_block=1, grid_h=1, grid_w=1)
    rng = np.random.default_rng(5)
    q = rng.normal(size=(1, 2, 64))
    k = rng.normal(size=(1, 2, 64))
    v = rng.normal(size=(1, 2, 64))
    ctx = stream.Context(block=0, blocks=[0], t0=[0], tokens_per_block=1)
    out = stream.chunk_attention(cfg, ctx, q, lambda b: (k, v))
    np.testing.assert_allclose(out, v, atol=1e-14)      # one key: weight 1
    # several keys from blocks sharing position 0 via the same slot start
    ks = rng.normal(size=(6, 2, 64))
    vs = rng.normal(size=(6, 2, 64))
    ctx6 = stream.Context(block=5, blocks=list(range(6)), t0=[0] * 6, tokens_per_block=1)
    out6 = stream.chunk_attention(cfg, ctx6, q, lambda b: (ks[b:b + 1], vs[b:b + 1]))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q.transpose(1, 0, 2)), torch.from_numpy(ks.transpose(1, 0, 2)),
        torch.from_numpy(vs.transpose(1, 0, 2)), scale=cfg.softmax_scale).numpy().transpose(1, 0, 2)
    np.testing.assert_allclose(out6, ref, atol=1e-12)


def test_row_subset_matches_full():
    cfg = C2_MID.with_(grid_h=4, grid_w=5, num_heads=2)
    kps = gen.poses(cfg)
    ctx = stream.plan_stream(cfg, kps)[9]
    kv_of = _kv_source(cfg)
    q = gen.tensor_np(gen.qkv_key(cfg, 0, 9, 0, "q"), (40, 2, 128), "bf16")
    full = stream.chunk_attention(cfg, ctx, q, kv_of)
    rows = [0, 7, 39]
    np.testing.assert_allclose(stream.chunk_attention(cfg, ctx, q, kv_of, rows=rows), full[rows],
                               atol=1e-13)
