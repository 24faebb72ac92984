"""Pins for the cache state machine, ConvKV and the e4m3 codec."""
import os

import numpy as np
import pytest
import torch

from oracle import convkv, e4m3, stream
from synth import C1_TINY, C2_MID, C3_14B, C4_CONVKV, C5_FP8, gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _pages_constants():
    out = {}
    for line in open(os.path.join(GOLDEN, "pages_constants.txt")):
        if line.startswith("#") or not line.strip():
            continue
        name, val = line.split("|")[0].split()
        out[name] = int(val)
    return out


def test_configs_follow_pages_constants():
    c = _pages_constants()
    for cfg in (C1_TINY, C2_MID, C3_14B, C4_CONVKV, C5_FP8):
        assert cfg.window == c["rolling_window_blocks"]
    for cfg in (C3_14B, C4_CONVKV, C5_FP8):
        assert cfg.n_steps == c["denoise_steps"]
    assert C4_CONVKV.conv_stride == c["convkv_compression_ratio"]


@pytest.mark.parametrize("cfg,steady,from_block", [
    (C1_TINY, 384, 5), (C2_MID, 9360, 5), (C3_14B, 32760, 6), (C5_FP8, 42120, 8)])
def test_constant_kv_length_prsink(cfg, steady, from_block):
    """Cache length is constant once warm, however long the stream runs."""
    n = cfg.n_blocks
    kps = gen.poses(cfg, n_blocks=n)
    ctxs = stream.plan_stream(cfg, kps, n)
    c = _pages_constants()
    for ctx in ctxs:
        b = ctx.block
        if b >= 1:
            assert ctx.blocks[0] == c["static_sink_block"]      # static sink is block 0
        assert ctx.blocks[-1] == b                               # current block last
        win = [j for j in range(max(1, b - 3), b)]
        assert ctx.blocks[len(ctx.blocks) - 1 - len(win):-1] == win
        assert all(1 <= j < b - 3 for j in ctx.dyn_ids)
        assert ctx.t0 == [s * cfg.frames_per_block for s in range(len(ctx.blocks))]
        if b >= from_block:
            assert ctx.kv_len == steady
        assert ctx.kv_len <= steady


def test_constant_kv_length_convkv():
    cfg = C4_CONVKV
    for b in range(cfg.n_blocks):
        ctx = stream.plan_convkv(cfg, b)
        expect = min(4096, 702 * max(0, b - 3)) + min(b + 1, 4) * 3510
        assert ctx.kv_len == expect
        if b >= 9:
            assert ctx.kv_len == 18136
        assert ctx.t0[0] == ctx.mem_tokens


def test_conv_matches_torch_conv1d():
    rng = np.random.default_rng(0)
    T, H, D = 3510, 2, 8
    x = rng.normal(size=(T, H, D))
    w = rng.normal(size=(H, D, 5))
    got = convkv.compress(x, w, 5)
    assert got.shape == (702, H, D)                 # 5:1
    xt = torch.from_numpy(x.reshape(T, H * D).T[None])          # [1, C, T]
    wt = torch.from_numpy(w.reshape(H * D, 1, 5))
    ref = torch.nn.functional.conv1d(xt, wt, stride=5, groups=H * D)[0].T.reshape(702, H, D)
    np.testing.assert_allclose(got, ref.numpy(), atol=1e-12)


def test_conv_closed_forms():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(50, 3, 4))
    w_first = np.zeros((3, 4, 5))
    w_first[..., 0] = 1.0
    np.testing.assert_array_equal(convkv.compress(x, w_first, 5), x[0::5])
    w_mean = np.full((3, 4, 5), 0.2)
    np.testing.assert_allclose(convkv.compress(x, w_mean, 5), x.reshape(10, 5, 3, 4).mean(1),
                               atol=1e-14)


def test_fifo_keeps_newest_in_order_and_saturates():
    mem = None
    chunks = []
    for e in range(8):
        new = np.full((702, 1, 1), float(e))
        chunks.append(new)
        mem = convkv.fifo_append(mem, new, 4096)
        assert mem.shape[0] == min(4096, 702 * (e + 1))
    allc = np.concatenate(chunks)
    np.testing.assert_array_equal(mem, allc[-4096:])


def test_convkv_memory_tracks_evictions():
    cfg = C4_CONVKV.with_(num_heads=1, head_dim=12, grid_h=2, grid_w=5, frames_per_block=1,
                          mem_slots=5)
    T = cfg.tokens_per_block                 # 10 tokens -> 2 compressed per eviction
    blocks = {b: (np.full((T, 1, 12), b + 1.0), np.full((T, 1, 12), -(b + 1.0))) for b in range(12)}
    w = np.zeros((2, 1, 12, 5))
    w[:, :, :, 0] = 1.0
    for b in range(12):
        mem = stream.convkv_memory(cfg, b, lambda e: blocks[e], w)
        n_ev = max(0, b - 3)
        if n_ev == 0:
            assert mem is None
            continue
        km, vm = mem
        expect = np.repeat(np.arange(1, n_ev + 1), 2)[-5:]
        np.testing.assert_array_equal(km[:, 0, 0], expect)
        np.testing.assert_array_equal(vm[:, 0, 0], -expect)


def _golden_e4m3():
    rows = []
    for line in open(os.path.join(GOLDEN, "e4m3_format.txt")):
        if line.startswith("#") or not line.strip():
            continue
        c, v = line.split()
        rows.append((int(c, 16), float(v)))
    return rows


def test_e4m3_golden_codes():
    for code, val in _golden_e4m3():
        got = float(e4m3.decode(np.uint8(code)))
        if np.isnan(val):
            assert np.isnan(got)
        else:
            assert got == val and np.signbit(got) == np.signbit(val)
            assert int(e4m3.encode(np.float64(val))) == code


def test_e4m3_all_codes_match_torch_and_roundtrip():
    codes = np.arange(256, dtype=np.uint8)
    mine = e4m3.decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(mine[ok], ref[ok])
    finite = codes[ok]
    np.testing.assert_array_equal(e4m3.encode(e4m3.decode(finite)), finite)


def test_e4m3_encode_matches_torch_rne_and_saturates():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.normal(size=20000) * 50, rng.uniform(-464, 464, 20000),
                        rng.normal(size=5000) * 1e-3]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(e4m3.encode(x), ref)
    # midpoints between consecutive codes go to the even code
    vals = e4m3.decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (vals[1:] + vals[:-1]) / 2
    got = e4m3.encode(mids)
    even = np.where(np.arange(1, 0x7F) % 2 == 0, np.arange(1, 0x7F), np.arange(0, 0x7E))
    np.testing.assert_array_equal(got, even.astype(np.uint8))
    # saturation (finite result) beyond the largest magnitude
    assert list(e4m3.encode(np.array([500.0, 1e9, -1e9]))) == [0x7E, 0x7E, 0xFE]


def test_quantize_scale_and_bound():
    rng = np.random.default_rng(8)
    x = rng.normal(size=(300, 64)).astype(np.float32) * 3
    codes, scale, y = e4m3.quantize(x)
    assert scale == np.float32(np.abs(x).max()) / np.float32(448)
    deq = e4m3.decode(codes) * np.float64(scale)
    # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 for normal codes
    big = np.abs(x) > 2 ** -6 * scale
    assert np.all(np.abs(deq[big] - x[big]) <= 2.0 ** -4 * np.abs(x[big]) + 1e-12)
    z_codes, z_scale, _ = e4m3.quantize(np.zeros((4, 4), np.float32))
    assert z_scale == 1.0 and not z_codes.any()


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(9)
    x = rng.normal(size=10000) * rng.choice([1e-3, 1, 1e3], size=10000)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(stream.bf16_round(x), ref)


def test_within_block_rotation_f32_close_to_fp64_rotation():
    from oracle import rope
    cfg = C5_FP8.with_(grid_h=6, grid_w=7, num_heads=2)
    rng = np.random.default_rng(10)
    x = rng.normal(size=(cfg.tokens_per_block, 2, 128)).astype(np.float32)
    f, h, w = rope.block_positions(cfg.frames_per_block, cfg.grid_h, cfg.grid_w)
    got = stream.rotate_within_block_f32(x, cfg)
    ref = rope.rotate(x, f, h, w)
    assert got.dtype == np.float32
    # each output is one fp32 product pair and a sum: error a few fp32 ulps
    np.testing.assert_allclose(got, ref, rtol=0, atol=4 * 2.0 ** -24 * 8)


def test_fp8_store_per_head_scales():
    rng = np.random.default_rng(11)
    x = rng.normal(size=(50, 3, 16)).astype(np.float32) * np.array([1, 10, 0])[None, :, None]
    codes, scales, deq, _ = stream.fp8_store(x.astype(np.float32))
    assert scales[2] == 1.0 and not codes[:, 2].any()
    assert np.isclose(scales[1], np.abs(x[:, 1]).max() / 448, rtol=1e-6)
    assert np.abs(deq - x).max() <= 2.0 ** -4 * np.abs(x).max()


def test_boundary_distance_flags_midpoints():
    vals = e4m3.decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (vals[1:] + vals[:-1]) / 2
    assert np.all(e4m3.boundary_distance(mids[5:]) == 0)
    assert np.all(e4m3.boundary_distance(vals[10:]) > 1e-3)


def _fp8_tc_golden():
    out = {}
    for line in open(os.path.join(GOLDEN, "fp8_tc_error.txt")):
        if line.startswith("#") or not line.strip():
            continue
        k, v = line.split()
        out[k] = float(v)
    return out


def test_fp8_tensor_core_tolerance_covers_simulated_rounding():
    """The e4m3 tensor-core tolerance of the GPU parity tests against the
    simulated effect of rounding the queries and probabilities to e4m3
    (tests/golden/make_fp8_tc_error.py, written from the oracle's storage
    functions): the simulation reproduces the oracle when it does not
    round, and the bounds cover the rounded result with margin, both on a
    small sample here and on the larger committed one."""
    import importlib.util
    from tests.harness import TOL
    spec = importlib.util.spec_from_file_location("make_fp8_tc_error",
                                                  os.path.join(GOLDEN, "make_fp8_tc_error.py"))
    sim = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(sim)
    o_ref, o_exact = sim.simulate(heads=(5,), n_rows=32, rounding=False)
    np.testing.assert_allclose(o_exact, o_ref, rtol=0, atol=1e-9)
    small = sim.errors(*sim.simulate(heads=(5, 30), n_rows=48))
    tol = TOL["e4m3_tc"]
    for e in (small, _fp8_tc_golden()):
        assert 0.01 < e["rel_l2"] and 1.4 * e["rel_l2"] <= tol["rel"], e
        assert 10 * e["max_abs"] <= tol["max_abs"] and 10 * e["mean_abs"] <= tol["mean_abs"], e
