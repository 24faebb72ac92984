"""Host-memory history tier with fetch-ahead ("SoulX-LiveAct", 上手实践指南:
block offload): while block b runs, the retrieval of block b + 1 is done
early (la_prefetch_context) and the picked blocks' K/V are written from
page-locked host memory on a separate copy stream.  Outputs must match the
oracle, be identical to the plain path (retrieval at select, fills from
device memory), and the dynamic sinks must agree."""
import numpy as np
import pytest

from bounded_kv_cache_la_b300 import capi
from oracle import stream as ostream
from synth import C3_14B, C5_FP8, gen

from . import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bounded_kv_cache_la_b300 import build
    build.build()


def _run(sc, n, ahead):
    import torch
    L = 2
    cache = H.make_cache(sc.with_(num_layers=L), attn_impl=1)
    kps = gen.poses(sc, n_blocks=n + 1)
    side = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    host = {}                          # the host tier: final K/V of every block, pinned

    def final_kv(layer, blk, device):
        _, k, v = H.torch_values(sc, layer, blk, 0)
        if device:
            return k, v
        key = (layer, blk)
        if key not in host:
            host[key] = (k.cpu().pin_memory(), v.cpu().pin_memory())
        return host[key]

    outs, dyns, filled_at_select = {}, {}, 0
    for b in range(n):
        ctx = cache.la_select_context(kps[b], stream=main)
        dyns[b] = ctx["dyn_ids"]
        for i, blk in enumerate(ctx["dyn_ids"]):
            if ctx["need_fill"][i]:
                filled_at_select += 1
                for l in range(L):
                    cache.la_fill_block(l, blk, *final_kv(l, blk, True), stream=main)
        ev = None
        if ahead and b + 1 < n:
            nxt = cache.la_prefetch_context(kps[b + 1], stream=main)
            with torch.cuda.stream(side):
                side.wait_stream(main)
                for i, blk in enumerate(nxt["dyn_ids"]):
                    if nxt["need_fill"][i]:
                        for l in range(L):
                            cache.la_fill_block(l, blk, *final_kv(l, blk, False), stream=side)
                ev = torch.cuda.Event()
                ev.record(side)
        for l in range(L):
            q, k, v = H.torch_values(sc, l, b, 0)
            out = torch.empty_like(q)
            cache.la_chunk_attention(l, q, k, v, out, stream=main)
            outs[(b, l)] = out
        for l in range(L):
            _, k, v = H.torch_values(sc, l, b, 0)
            cache.la_cache_append_block(l, k, v, stream=main)
        if ev is not None:
            main.wait_event(ev)
    torch.cuda.synchronize()
    st, msg = cache.la_get_error()
    assert st == capi.LA_OK, msg
    return outs, dyns, filled_at_select


@pytest.mark.parametrize("sc", [C3_14B.with_(num_heads=4, grid_h=10, grid_w=13),   # 390 tokens, top-2
                                C5_FP8.with_(num_heads=3, grid_h=6, grid_w=10)],   # e4m3, top-4
                         ids=["bf16_top2", "e4m3_top4"])
def test_fetch_ahead_from_host_matches_plain_path(sc):
    n = 14
    plain, dyn_p, _ = _run(sc, n, ahead=False)
    fetched, dyn_f, at_select = _run(sc, n, ahead=True)
    assert dyn_p == dyn_f
    assert at_select == 0                    # every pick was in place at select
    assert sum(len(d) for d in dyn_f.values()) > 0
    import torch
    for key in plain:
        assert torch.equal(plain[key], fetched[key]), key
    # the fetched-ahead path against the oracle: a warm-up block, the first
    # block with a full dynamic sink, the last block; both layers
    ref = ostream.plan_stream(sc, gen.poses(sc, n_blocks=n + 1), n)
    first_full = min(b for b in range(n) if len(ref[b].dyn_ids) == sc.dyn_topk)
    vals = H.Values(sc)
    kind = "bf16" if sc.kv_dtype == "bf16" else "e4m3_tc"
    for b in (2, first_full, n - 1):
        assert dyn_f[b] == ref[b].dyn_ids or ref[b].gap <= 1e-6, (b, dyn_f[b], ref[b])
        if dyn_f[b] != ref[b].dyn_ids:
            continue
        for l in range(2):
            o = H.oracle_output(sc, ref[b], vals, l, 0, 1)
            H.compare(fetched[(b, l)].float().cpu().numpy(), o, kind, f"block {b} layer {l}")


def test_prefetch_call_rules():
    sc = C3_14B.with_(num_heads=2, grid_h=4, grid_w=4, num_layers=1)
    cache = H.make_cache(sc)
    kps = gen.poses(sc, n_blocks=3)
    with pytest.raises(capi.LaError) as e:          # no block in progress
        cache.la_prefetch_context(kps[1])
    assert e.value.status == capi.LA_ERR_STATE
    cache.la_select_context(kps[0])
    cache.la_prefetch_context(kps[1])
    with pytest.raises(capi.LaError) as e:          # once per block
        cache.la_prefetch_context(kps[1])
    assert e.value.status == capi.LA_ERR_STATE
    bad = np.full(34, np.nan, np.float32)
    res = H.make_cache(sc.with_(history_mode="resident"))
    res.la_select_context(kps[0])
    with pytest.raises(capi.LaError) as e:          # resident history needs no fetch
        res.la_prefetch_context(kps[1])
    assert e.value.status == capi.LA_ERR_UNSUPPORTED
