"""The parity gates at full shapes, through the C ABI against the oracle:

* retrieval ids bit-exact (where the oracle's k-th/(k+1)-th gap exceeds
  1e-6) and the KV length on every block of the whole 14B-shape stream
  (3600 blocks, periodic poses with phase jumps) and of the FP8 stress stream
  (10000 blocks of 50 repeating pose clusters) ("LiveAnimate", 方法: dynamic
  sink by pose retrieval);
* the mid stream: every block, every row, every head;
* the 14B-shape, ConvKV and FP8 stress streams: every head x 256 query rows
  (first tile, two middle tiles, the ragged last tile) on blocks 0, 1, 4, 5,
  9, 10, 100 and the last block of the stream, which is reached by loading
  the pose history and supplying the sink and window blocks ("LiveAnimate",
  实验: cost and state stay constant however long the stream);
* one 14B-shape block checked on every row and head.

Oracle inputs come from the seeded generator (tests/harness.FullValues);
the oracle runs in a spawned process pool, a few heads per task.
"""
import multiprocessing as mp

import numpy as np
import pytest

from bounded_kv_cache_la_b300 import capi
from oracle import stream as ostream
from oracle import pose as opose
from synth import C2_MID, C3_14B, C4_CONVKV, C5_FP8, gen

from . import harness as H
from . import oracle_pool

pytestmark = pytest.mark.gpu

GATE_BLOCKS = (0, 1, 4, 5, 9, 10, 100)


@pytest.fixture(scope="module")
def pool():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bounded_kv_cache_la_b300 import build
    build.build()
    p = mp.get_context("spawn").Pool(8)
    yield p
    p.close()
    p.join()


def _rows(T):
    """256 query rows: the first tile's 64, 64 at a third and two thirds of
    the block, the last 64 (the ragged last tile); fewer on short blocks."""
    r = np.r_[0:64, T // 3:T // 3 + 64, 2 * T // 3:2 * T // 3 + 64, T - 64:T]
    return np.unique(np.clip(r, 0, T - 1))


def _oracle(pool, sc, ctx, vals, step, n_steps, rows, w_kv=None, group=8, row_chunk=None):
    """Oracle output of layer 0 for every head (and the given rows), one
    pool task per head group (and per chunk of rows)."""
    kv_of = vals.kv_of(0, lambda b: step if b == ctx.block else n_steps - 1)
    q = vals.get(0, ctx.block, step, "q")
    mem = ostream.convkv_memory(sc, ctx.block, kv_of, w_kv) if ctx.mem_tokens else None
    rows = np.arange(sc.tokens_per_block) if rows is None else np.asarray(rows)
    chunks = [rows] if row_chunk is None else np.array_split(rows, -(-len(rows) // row_chunk))
    tasks, where = [], []
    for h0 in range(0, sc.num_heads, group):
        hs = slice(h0, min(sc.num_heads, h0 + group))
        kv = {b: tuple(x[:, hs] for x in kv_of(b)) for b in ctx.blocks}
        m = None if mem is None else (mem[0][:, hs], mem[1][:, hs])
        for ci, rc in enumerate(chunks):
            tasks.append((sc, ctx, q[:, hs], kv, m, rc))
            where.append((hs, ci))
    outs = pool.map(oracle_pool.attend, tasks)
    out = np.zeros((len(rows), sc.num_heads, sc.head_dim))
    starts = np.cumsum([0] + [len(c) for c in chunks])
    for (hs, ci), o in zip(where, outs):
        out[starts[ci]:starts[ci + 1], hs] = o
    return out


def _check(pool, sc, ctx_ref, got_ctx, out, vals, rows, kind, w_kv=None, row_chunk=None):
    """One call's output against the oracle (returns False when the ids
    differ inside the tie gate, so there is nothing to compare)."""
    assert got_ctx["kv_len"] == ctx_ref.kv_len, (got_ctx, ctx_ref)
    if sc.policy == "prsink" and got_ctx["dyn_ids"] != ctx_ref.dyn_ids:
        assert ctx_ref.gap <= 1e-6, (got_ctx, ctx_ref)
        return False
    o = _oracle(pool, sc, ctx_ref, vals, 0, 1, rows, w_kv=w_kv, row_chunk=row_chunk)
    got = out.float().cpu().numpy()
    got = got if rows is None else got[rows]
    H.compare(got, o, kind, f"{sc.name} block {ctx_ref.block}")
    return True


def _fill_picks(cache, sc, ctx):
    for i, bid in enumerate(ctx["dyn_ids"]):
        if ctx["need_fill"][i]:
            _, k, v = H.torch_values(sc, 0, bid, 0)
            cache.la_fill_block(0, bid, k, v)


def _attend(cache, sc, b):
    import torch
    q, k, v = H.torch_values(sc, 0, b, 0)
    out = torch.empty_like(q)
    cache.la_chunk_attention(0, q, k, v, out)
    return out, k, v


def _stream_from_start(pool, sc, n, checks, kind, rows_of=lambda b: None, w_kv=None,
                       row_chunk=None):
    """Streams blocks 0..n-1 (one layer, one denoising step) and checks the
    blocks in `checks` as they are generated."""
    cache = H.make_cache(sc.with_(num_layers=1), attn_impl=1)
    kps = gen.poses(sc, n_blocks=n)
    if sc.policy == "prsink":
        descs = np.stack([opose.descriptor(k) for k in kps])
    vals = H.FullValues(sc)
    checked = 0
    for b in range(n):
        ctx = cache.la_select_context(kps[b] if sc.policy == "prsink" else None)
        _fill_picks(cache, sc, ctx)
        out, k, v = _attend(cache, sc, b)
        if b in checks:
            ref = (ostream.plan_prsink(sc, b, descs[:b], descs[b]) if sc.policy == "prsink"
                   else ostream.plan_convkv(sc, b))
            vals.prune(set(ref.blocks) | set(range(max(0, b - 12), b + 1)))
            checked += _check(pool, sc, ref, ctx, out, vals, rows_of(b), kind, w_kv, row_chunk)
        cache.la_cache_append_block(0, k, v)
    st, msg = cache.la_get_error()
    assert st == capi.LA_OK, msg
    cache.close()
    return checked


def _resume_late(pool, sc, b, kind):
    """Block b of an external-history stream: pose history 0..b-1 loaded, the
    sink and window blocks supplied, the picks filled, then one call."""
    n = sc.n_blocks
    kps = gen.poses(sc, n_blocks=n)
    descs = np.stack([opose.descriptor(k) for k in kps[:b + 1]])
    cache = H.make_cache(sc.with_(num_layers=1), attn_impl=1, max_history=b + 2)
    cache.la_cache_load_history(kps[:b].reshape(b, 34))
    for blk in [0] + list(range(b - sc.window, b)):
        _, k, v = H.torch_values(sc, 0, blk, 0)
        cache.la_fill_window(0, blk, k, v)
    ctx = cache.la_select_context(kps[b])
    _fill_picks(cache, sc, ctx)
    out, _, _ = _attend(cache, sc, b)
    st, msg = cache.la_get_error()
    assert st == capi.LA_OK, msg
    ref = ostream.plan_prsink(sc, b, descs[:b], descs[b])
    ok = _check(pool, sc, ref, ctx, out, H.FullValues(sc), _rows(sc.tokens_per_block), kind)
    cache.close()
    return ok


@pytest.mark.parametrize("base", [C3_14B, C5_FP8], ids=["c3_14b_3600", "c5_fp8_10000"])
def test_selection_over_whole_stream(pool, base):
    """Ids and KV length on every block of the whole stream (tiny pages:
    only the retrieval and the context plan are under test)."""
    import torch
    sc = base.with_(frames_per_block=1, grid_h=4, grid_w=4, num_heads=2, kv_dtype="bf16",
                    history_mode="resident", num_layers=1)
    n = base.n_blocks
    kps = gen.poses(sc, n_blocks=n)
    ref = ostream.plan_stream(sc, kps, n)
    cache = capi.Cache(capi.config_for(sc, max_history=n))
    kv = torch.zeros((sc.tokens_per_block, sc.num_heads, sc.head_dim), dtype=torch.bfloat16,
                     device="cuda")
    gated = 0
    for b in range(n):
        ctx = cache.la_select_context(kps[b])
        assert ctx["kv_len"] == ref[b].kv_len, b
        if ref[b].gap > 1e-6:
            assert ctx["dyn_ids"] == ref[b].dyn_ids, (b, ctx["dyn_ids"], ref[b].dyn_ids)
        else:
            gated += 1
        cache.la_cache_append_block(0, kv, kv)
    assert ref[-1].kv_len == (2 + base.dyn_topk + base.window) * sc.tokens_per_block
    assert gated <= n // 100, gated
    st, msg = cache.la_get_error()
    assert st == capi.LA_OK, msg


def test_c2_every_block_row_and_head(pool):
    sc = C2_MID
    checked = _stream_from_start(pool, sc, sc.n_blocks, set(range(sc.n_blocks)), "bf16")
    assert checked >= sc.n_blocks - 2


@pytest.mark.parametrize("base,kind", [(C3_14B, "bf16"), (C5_FP8, "e4m3_tc")],
                         ids=["c3_14b", "c5_fp8"])
def test_gate_blocks_external_history(pool, base, kind):
    sc = base.with_(n_steps=1)
    early = [b for b in GATE_BLOCKS if b <= 10]
    checked = _stream_from_start(pool, sc, 11, set(early), kind,
                                 rows_of=lambda b: _rows(sc.tokens_per_block))
    checked += _resume_late(pool, sc, 100, kind)
    checked += _resume_late(pool, sc, sc.n_blocks - 1, kind)
    assert checked >= len(early) + 1


def test_gate_blocks_convkv(pool):
    """Streamed from block 0 to the last block (999): the memory fills at
    block 9 and stays at 4096 tokens."""
    sc = C4_CONVKV.with_(n_steps=1)
    w = gen.conv_weights_np(sc, 0)
    checks = set(GATE_BLOCKS) | {sc.n_blocks - 1}
    checked = _stream_from_start(pool, sc, sc.n_blocks, checks, "bf16",
                                 rows_of=lambda b: _rows(sc.tokens_per_block), w_kv=w)
    assert checked == len(checks)


def test_c3_one_block_every_row_and_head(pool):
    """Block 11 of the 14B-shape stream (32760 keys): all 4680 x 40 rows."""
    sc = C3_14B.with_(n_steps=1)
    checked = _stream_from_start(pool, sc, 12, {11}, "bf16", row_chunk=1170)
    assert checked == 1
