"""GPU parity of the tensor-core attention's running-max rescale.

The online softmax of the tensor-core kernel keeps a lazy running max: it
moves only when a row's scores grow by more than 8 (log2 units), and then O
and the row sum are rescaled by 2^(m_old - m_new) before more keys are
added ("LiveAnimate" (ai-feeds.com), 方法: the block attends to its whole
bounded context in one softmax).  Random inputs almost never move it after
the first key tile.  Here every cached block carries one "hot" key
(tests/hot_keys.py) whose score is pinned, the same for every query row, to
about 3 + 9.5 * block id, so along the slot order (static sink, dynamic
sink, window, current block: ascending block ids) the max jumps by more
than 8 at every slot, in key tiles and tile halves that vary from block to
block.  A rescale that is skipped, or applied to O but not to the sum, moves
the output by about the size of V (tests/test_rescale_case.py shows that on
the CPU) and fails the comparison with the oracle.

The one V element of 8 per block gives an e4m3 cache one V scale for every
block, so the kernel's probabilities carry no per-slot factor and the hot
key's is exactly 1, whose e4m3 rounding is exact (a one-hot row would
otherwise show that rounding, up to 2^-4 relative, in full).
"""
import pytest

from oracle import stream as ostream
from synth import C2_MID, C5_FP8, gen

from . import harness as H
from .hot_keys import HotKeys

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bounded_kv_cache_la_b300 import build
    build.build()


def _hot_stream(sc, n_blocks, keep, kind):
    import torch
    hk = HotKeys(sc)
    cache = H.make_cache(sc.with_(num_layers=1), attn_impl=1)
    kps = gen.poses(sc, n_blocks=n_blocks)
    plan = ostream.plan_stream(sc, kps, n_blocks)
    outs = {}
    for b in range(n_blocks):
        ctx = cache.la_select_context(kps[b])
        assert ctx["kv_len"] == plan[b].kv_len
        q, k, v = hk.modify(b, *H.torch_values(sc, 0, b, 0))
        out = torch.empty_like(q)
        cache.la_chunk_attention(0, q, k, v, out)
        if b in keep:
            outs[b] = (ctx, out.float().cpu().numpy())
        cache.la_cache_append_block(0, k, v)
    torch.cuda.synchronize()
    st, msg = cache.la_get_error()
    assert st == 0, msg

    vals = H.Values(sc)
    checked = 0
    for b in sorted(keep):
        ctx_dev, got = outs[b]
        ctx = plan[b]
        if ctx_dev["dyn_ids"] != ctx.dyn_ids:
            assert ctx.gap <= 1e-6
            continue
        # the slot order must be ascending in block id for the max to climb
        assert list(ctx.blocks) == sorted(ctx.blocks)
        ref = ostream.chunk_attention(sc, ctx, hk.q_of(vals, b), hk.kv_of(vals))
        H.compare(got, ref, kind, f"block {b}")
        checked += 1
    assert checked >= 2


def test_running_max_rescale_bf16():
    """bf16 cache: 390-token blocks (key tiles 128, 128, 128, 6), pose top-1
    dynamic sink, 2 heads; every slot of blocks 6..11 raises the max."""
    sc = C2_MID.with_(grid_h=13, grid_w=15, num_heads=2)
    _hot_stream(sc, 12, {6, 9, 11}, "bf16")


def test_running_max_rescale_e4m3():
    """e4m3 cache (per-(head, block) scales), pose top-4 dynamic sink,
    resident history, 2 heads."""
    sc = C5_FP8.with_(grid_h=13, grid_w=15, num_heads=2, history_mode="resident")
    _hot_stream(sc, 14, {9, 13}, "e4m3_tc")
