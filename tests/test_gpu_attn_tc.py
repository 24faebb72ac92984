"""GPU parity of the tensor-core chunk attention (tcgen05) against the oracle,
at the mid shape over a whole stream and at the 14B shape on sampled
rows/heads, plus ragged tiles and the ConvKV memory slot."""
import numpy as np
import pytest

from oracle import stream as ostream
from synth import C2_MID, C3_14B, C4_CONVKV, C5_FP8, gen

from . import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bounded_kv_cache_la_b300 import build
    build.build()


def test_c2_stream_tensor_cores():
    """Mid stream, all 64 blocks through the tensor-core kernel; oracle on
    11 blocks (rows spanning the first tile, the ragged last tile)."""
    sc = C2_MID
    keep = {0, 1, 2, 4, 5, 6, 9, 12, 20, 33, 63}
    cache, ctxs, outs = H.run_stream(sc, 64, keep, attn_impl=1)
    ref = ostream.plan_stream(sc, gen.poses(sc), 64)
    heads = [0, 7, 11]
    vals = H.Values(sc, heads)
    rows = np.r_[0:130, 1500:1560]
    for b in sorted(keep):
        ctx = ref[b]
        if ctxs[b]["dyn_ids"] != ctx.dyn_ids:
            assert ctx.gap <= 1e-6
            continue
        o = H.oracle_output(sc, ctx, vals, 0, 0, 1, rows=rows)
        H.compare(outs[b][(0, 0)][rows][:, heads], o, "bf16", f"block {b}")


def test_tensor_cores_match_simt_kernel_all_rows():
    """Both kernels of the library on the same stream agree on every output
    (a cross-check of layouts; the oracle checks above are the parity)."""
    sc = C2_MID.with_(grid_h=13, grid_w=15)           # 390 tokens: 3 tiles + 6 rows
    keep = {3, 7, 11}
    _, _, o_tc = H.run_stream(sc, 12, keep, attn_impl=1)
    _, _, o_simt = H.run_stream(sc, 12, keep, attn_impl=2)
    for b in keep:
        d = np.abs(o_tc[b][(0, 0)] - o_simt[b][(0, 0)])
        assert d.max() < 1e-2 and d.mean() < 5e-4, (b, d.max(), d.mean())


def test_c3_14b_shape_sampled_rows():
    """14B shape (40 heads x 128, 4680 tokens, top-2 dynamic sink), external
    history; oracle on 4 heads x 192 rows of several blocks, incl. the
    ragged last query tile and every slot kind."""
    sc = C3_14B
    n = 12
    keep = {0, 5, 6, 11}
    cache, ctxs, outs = H.run_stream(sc, n, keep, n_steps=1, layers=1, attn_impl=1)
    ref = ostream.plan_stream(sc, gen.poses(sc, n_blocks=n), n)
    for b in range(n):
        assert ctxs[b]["kv_len"] == ref[b].kv_len
    assert ctxs[11]["kv_len"] == 32760
    heads = [0, 13, 26, 39]
    vals = H.Values(sc, heads)
    rows = np.r_[0:64, 2300:2364, 4616:4680]
    for b in sorted(keep):
        ctx = ref[b]
        if ctxs[b]["dyn_ids"] != ctx.dyn_ids:
            assert ctx.gap <= 1e-6
            continue
        o = H.oracle_output(sc, ctx, vals, 0, 0, 1, rows=rows)
        H.compare(outs[b][(0, 0)][rows][:, heads], o, "bf16", f"block {b}")


def test_convkv_tensor_cores():
    """ConvKV memory slot (token count not a multiple of 128, ring wrapped)
    through the tensor-core kernel, two denoising steps."""
    sc = C4_CONVKV.with_(num_heads=4, grid_h=5, grid_w=9, mem_slots=240)
    keep = {4, 13, 15}
    _, ctxs, outs = H.run_stream(sc, 16, keep, n_steps=2, attn_impl=1)
    vals = H.Values(sc)
    w = gen.conv_weights_np(sc, 0)
    for b in sorted(keep):
        ctx = ostream.plan_convkv(sc, b)
        assert ctxs[b]["mem_tokens"] == ctx.mem_tokens
        for s in range(2):
            o = H.oracle_output(sc, ctx, vals, 0, s, 2, w_kv=w)
            H.compare(outs[b][(0, s)], o, "bf16", f"block {b} step {s}")


def test_uniform_scores_give_mean_of_values():
    """Zero queries: every output row is the mean of V over the context."""
    import torch
    sc = C2_MID.with_(grid_h=6, grid_w=11)
    cache = H.make_cache(sc.with_(num_layers=1), attn_impl=1)
    kps = gen.poses(sc, n_blocks=8)
    vs = []
    for b in range(8):
        cache.la_select_context(kps[b])
        q, k, v = H.torch_values(sc, 0, b, 0)
        out = torch.empty_like(q)
        cache.la_chunk_attention(0, torch.zeros_like(q), k, v, out)
        if b == 7:
            ctx = ostream.plan_stream(sc, kps, 8)[7]
            V = np.concatenate([H.Values(sc).get(0, blk, 0, "v") for blk in ctx.blocks]).astype(np.float64)
            ref = np.broadcast_to(V.mean(0), out.shape)
            H.compare(out.float().cpu().numpy(), ref, "bf16", "uniform")
        cache.la_cache_append_block(0, k, v)


def test_fp8_tensor_cores_stream():
    """FP8 stress shape (4680 tokens, pose top-4, e4m3 K/V with per-(head,
    block) scales) at 4 heads, external history: the kind::f8f6f4 kernel
    against the oracle over the dequantised cache, on blocks before and
    after the dynamic sink fills."""
    sc = C5_FP8.with_(num_heads=4)
    n = 12
    keep = {0, 4, 5, 8, 11}
    _, ctxs, outs = H.run_stream(sc, n, keep, n_steps=1, layers=1, attn_impl=1)
    ref = ostream.plan_stream(sc, gen.poses(sc, n_blocks=n), n)
    for b in range(n):
        assert ctxs[b]["kv_len"] == ref[b].kv_len
    assert ctxs[11]["kv_len"] == 9 * sc.tokens_per_block
    vals = H.Values(sc)
    rows = np.r_[0:160, 2300:2400, 4560:4680]
    for b in sorted(keep):
        ctx = ref[b]
        if ctxs[b]["dyn_ids"] != ctx.dyn_ids:
            assert ctx.gap <= 1e-6
            continue
        o = H.oracle_output(sc, ctx, vals, 0, 0, 1, rows=rows)
        H.compare(outs[b][(0, 0)][rows], o, "e4m3_tc", f"block {b}")


def test_fp8_tensor_cores_match_simt_kernel():
    """The e4m3 tensor-core kernel and the CUDA-core kernel (which keeps Q
    and P in fp32) agree on a ragged shape within the e4m3 bound."""
    sc = C5_FP8.with_(num_heads=3, grid_h=13, grid_w=15, history_mode="resident")  # 585 tokens
    keep = {3, 7, 11}
    _, _, o_tc = H.run_stream(sc, 12, keep, attn_impl=1)
    _, _, o_simt = H.run_stream(sc, 12, keep, attn_impl=2)
    for b in keep:
        H.compare(o_tc[b][(0, 0)], o_simt[b][(0, 0)].astype(np.float64), "e4m3_tc", f"block {b}")


def test_fp8_14b_shape_sampled_rows():
    """All 40 heads of the FP8 stress shape; oracle on 3 heads x 192 rows
    once the top-4 dynamic sink is full (42120 keys)."""
    sc = C5_FP8
    n = 10
    keep = {9}
    _, ctxs, outs = H.run_stream(sc, n, keep, n_steps=1, layers=1, attn_impl=1)
    ref = ostream.plan_stream(sc, gen.poses(sc, n_blocks=n), n)
    assert ctxs[9]["kv_len"] == ref[9].kv_len == 42120
    heads = [0, 21, 39]
    vals = H.Values(sc, heads)
    rows = np.r_[0:64, 2300:2364, 4616:4680]
    ctx = ref[9]
    if ctxs[9]["dyn_ids"] != ctx.dyn_ids:
        assert ctx.gap <= 1e-6
        return
    o = H.oracle_output(sc, ctx, vals, 0, 0, 1, rows=rows)
    H.compare(outs[9][(0, 0)][rows][:, heads], o, "e4m3_tc", "block 9")


def test_convkv_full_shape_sampled_rows():
    """ConvKV at its full shape (40 heads x 128, 3510 tokens per block,
    4096-token memory): blocks 9 (memory just saturated: 6 evictions x 702
    tokens > 4096) and 11, oracle on 3 heads x 192 rows."""
    sc = C4_CONVKV
    n = 12
    keep = {9, 11}
    _, ctxs, outs = H.run_stream(sc, n, keep, n_steps=1, layers=1, attn_impl=1)
    heads = [0, 19, 39]
    vals = H.Values(sc, heads)
    w = gen.conv_weights_np(sc, 0)[:, heads]
    rows = np.r_[0:64, 1700:1764, 3446:3510]
    for b in sorted(keep):
        ctx = ostream.plan_convkv(sc, b)
        assert ctxs[b]["mem_tokens"] == ctx.mem_tokens == 4096
        assert ctxs[b]["kv_len"] == ctx.kv_len == 18136
        o = H.oracle_output(sc, ctx, vals, 0, 0, 1, rows=rows, w_kv=w)
        H.compare(outs[b][(0, 0)][rows][:, heads], o, "bf16", f"block {b}")


def test_single_ragged_query_tile_odd_heads():
    """48 tokens per block (one partial query tile per head) and 3 heads:
    every item is a per-slot piece of that tile, merged after the kernel;
    all rows against the oracle."""
    sc = C2_MID.with_(num_heads=3, frames_per_block=3, grid_h=4, grid_w=4)
    keep = {0, 3, 4, 6, 9}
    _, ctxs, outs = H.run_stream(sc, 10, keep, attn_impl=1)
    ref = ostream.plan_stream(sc, gen.poses(sc, n_blocks=10), 10)
    vals = H.Values(sc)
    for b in sorted(keep):
        ctx = ref[b]
        assert ctxs[b]["kv_len"] == ctx.kv_len
        if ctxs[b]["dyn_ids"] != ctx.dyn_ids:
            assert ctx.gap <= 1e-6
            continue
        o = H.oracle_output(sc, ctx, vals, 0, 0, 1)
        H.compare(outs[b][(0, 0)], o, "bf16", f"block {b}")


def test_largest_dynamic_sink():
    """Top-8 dynamic sink (the most the C ABI takes): 13 slots once warm;
    ids bit-exact where the gap allows, outputs against the oracle."""
    sc = C5_FP8.with_(num_heads=2, grid_h=6, grid_w=10, kv_dtype="bf16", dyn_topk=8,
                      history_mode="resident")                 # 180 tokens per block
    n = 16
    keep = {12, 15}
    _, ctxs, outs = H.run_stream(sc, n, keep, attn_impl=1)
    ref = ostream.plan_stream(sc, gen.poses(sc, n_blocks=n), n)
    assert ctxs[15]["n_slots"] == 13 and ctxs[15]["kv_len"] == 13 * sc.tokens_per_block
    vals = H.Values(sc)
    for b in range(n):
        assert ctxs[b]["kv_len"] == ref[b].kv_len
        if ref[b].gap > 1e-6:
            assert ctxs[b]["dyn_ids"] == ref[b].dyn_ids
    for b in sorted(keep):
        ctx = ref[b]
        if ctxs[b]["dyn_ids"] != ctx.dyn_ids:
            assert ctx.gap <= 1e-6
            continue
        o = H.oracle_output(sc, ctx, vals, 0, 0, 1)
        H.compare(outs[b][(0, 0)], o, "bf16", f"block {b}")


def _all_rows_against_oracle(sc, n, keep, tol):
    _, ctxs, outs = H.run_stream(sc, n, keep, attn_impl=1)
    ref = ostream.plan_stream(sc, gen.poses(sc, n_blocks=n), n)
    vals = H.Values(sc)
    checked = 0
    for b in sorted(keep):
        ctx = ref[b]
        assert ctxs[b]["kv_len"] == ctx.kv_len
        if ctxs[b]["dyn_ids"] != ctx.dyn_ids:
            assert ctx.gap <= 1e-6
            continue
        o = H.oracle_output(sc, ctx, vals, 0, 0, 1)
        H.compare(outs[b][(0, 0)], o, tol, f"block {b}")
        checked += 1
    assert checked >= len(keep) - 1


def test_odd_frame_and_block_sizes():
    """Frames of 5 x 7 tokens and 105 tokens per block, both odd: the query
    rotation's token pairs that straddle a frame boundary and a last token
    without a partner; all rows against the oracle."""
    sc = C2_MID.with_(num_heads=3, frames_per_block=3, grid_h=5, grid_w=7)
    _all_rows_against_oracle(sc, 10, {0, 4, 6, 9}, "bf16")


@pytest.mark.parametrize("dims,kv", [((72, 28, 28), "bf16"), ((70, 30, 28), "bf16"),
                                     ((42, 44, 42), "bf16"), ((42, 44, 42), "e4m3")])
def test_other_rope_splits(dims, kv):
    """Other (t, h, w) splits of the head dim: a temporal part wider than half
    a row (whole-row query copies), one that is not a multiple of 4 (pairs
    read one at a time), and the e4m3 path; all rows against the oracle."""
    sc = C2_MID.with_(num_heads=2, frames_per_block=2, grid_h=6, grid_w=9, rope_dims=dims,
                      kv_dtype=kv)
    _all_rows_against_oracle(sc, 8, {0, 4, 7}, "bf16" if kv == "bf16" else "e4m3_tc")
