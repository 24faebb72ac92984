"""Static-sink refresh (the cache side of a rolling sink frame: the sink's
K/V are re-encoded from the cached reference and replaced between blocks),
against the oracle with block 0's K/V substituted from the refresh onward."""
import numpy as np
import pytest

from bounded_kv_cache_la_b300 import capi
from oracle import stream as ostream
from synth import C2_MID, C4_CONVKV, C5_FP8, gen

from . import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bounded_kv_cache_la_b300 import build
    build.build()


REFRESH_STEP = 99          # generator step id of the re-encoded sink values


def _run(sc, n, refresh_at, keep, tol):
    import torch
    cache = H.make_cache(sc.with_(num_layers=1), attn_impl=1)
    kps = gen.poses(sc, n_blocks=n)
    ref = ostream.plan_stream(sc, kps, n)
    outs = {}
    for b in range(n):
        if b == refresh_at:
            _, k_new, v_new = H.torch_values(sc, 0, 0, REFRESH_STEP)
            cache.la_refresh_sink(0, k_new, v_new)
        ctx = cache.la_select_context(kps[b])
        for i, bid in enumerate(ctx["dyn_ids"]):
            if ctx["need_fill"][i]:
                _, k, v = H.torch_values(sc, 0, bid, 0)
                cache.la_fill_block(0, bid, k, v)
        q, k, v = H.torch_values(sc, 0, b, 0)
        out = torch.empty_like(q)
        cache.la_chunk_attention(0, q, k, v, out)
        if b in keep:
            outs[b] = (out.float().cpu().numpy(), ctx)
        cache.la_cache_append_block(0, k, v)
    torch.cuda.synchronize()
    st, msg = cache.la_get_error()
    assert st == capi.LA_OK, msg
    vals = H.Values(sc)
    for b, (o_gpu, ctx) in sorted(outs.items()):
        want = ref[b]
        if ctx["dyn_ids"] != want.dyn_ids:
            assert want.gap <= 1e-6
            continue
        refreshed = b >= refresh_at

        def kv_of(blk):
            step = REFRESH_STEP if (blk == 0 and refreshed) else 0
            return vals.get(0, blk, step, "k"), vals.get(0, blk, step, "v")

        o = ostream.chunk_attention(sc, want, vals.get(0, b, 0, "q"), kv_of)
        H.compare(o_gpu, o, tol, f"block {b}")
    return cache


def test_sink_refresh_bf16():
    sc = C2_MID.with_(grid_h=13, grid_w=15)                   # 390 tokens, 12 heads
    _run(sc, 10, refresh_at=6, keep={3, 6, 9}, tol="bf16")


def test_sink_refresh_e4m3_external_history():
    sc = C5_FP8.with_(num_heads=3, grid_h=6, grid_w=10)       # 180 tokens, top-4
    _run(sc, 12, refresh_at=7, keep={5, 7, 11}, tol="e4m3_tc")


def test_sink_refresh_call_rules():
    import torch
    sc = C2_MID.with_(grid_h=4, grid_w=4)
    cache = H.make_cache(sc.with_(num_layers=1))
    q, k, v = H.torch_values(sc, 0, 0, 0)
    with pytest.raises(capi.LaError) as e:                      # no committed block 0 yet
        cache.la_refresh_sink(0, k, v)
    assert e.value.status == capi.LA_ERR_STATE
    kps = gen.poses(sc, n_blocks=2)
    cache.la_select_context(kps[0])
    out = torch.empty_like(q)
    cache.la_chunk_attention(0, q, k, v, out)
    cache.la_cache_append_block(0, k, v)
    cache.la_select_context(kps[1])
    with pytest.raises(capi.LaError) as e:                      # inside a block
        cache.la_refresh_sink(0, k, v)
    assert e.value.status == capi.LA_ERR_STATE
    conv = H.make_cache(C4_CONVKV.with_(num_heads=2, grid_h=5, grid_w=9, mem_slots=240, num_layers=1))
    qc, kc, vc = H.torch_values(C4_CONVKV.with_(num_heads=2, grid_h=5, grid_w=9), 0, 0, 0)
    with pytest.raises(capi.LaError) as e:                      # ConvKV has no sink
        conv.la_refresh_sink(0, kc, vc)
    assert e.value.status == capi.LA_ERR_UNSUPPORTED
