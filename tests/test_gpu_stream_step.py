"""la_stream_step (one call per block; its last denoising step writes the
block's pages straight into the block's own frame) against the oracle on a
warm-up block, the first block with a full context and the last block, and
against the per-call C ABI path on the same inputs: every output and every
stored page identical."""
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


def _tensors(sc, L, S, b):
    """[step * L + layer] lists of q, k, v for block b."""
    q, k, v = [], [], []
    for s in range(S):
        for l in range(L):
            qq, kk, vv = H.torch_values(sc, l, b, s)
            q.append(qq); k.append(kk); v.append(vv)
    return q, k, v


def _oracle_plan(sc, kps, n):
    if sc.policy == "convkv":
        return [ostream.plan_convkv(sc, b) for b in range(n)]
    return ostream.plan_stream(sc, kps, n)


def _full_context(sc, ref):
    """First block whose context is complete (full dynamic sink, or a full
    ConvKV memory)."""
    if sc.policy == "convkv":
        return min(c.block for c in ref if c.mem_tokens == sc.mem_slots)
    return min(c.block for c in ref if len(c.dyn_ids) == sc.dyn_topk)


def _compare(sc, n, L=2, S=2):
    import torch
    scl = sc.with_(num_layers=L)
    kps = gen.poses(sc, n_blocks=n)
    ref = _oracle_plan(sc, kps, n)
    checks = {2, _full_context(sc, ref), n - 1}
    vals = H.Values(sc)
    w = [gen.conv_weights_np(sc, l) for l in range(L)] if sc.policy == "convkv" else [None] * L
    kind = "e4m3_tc" if sc.kv_dtype == "e4m3" else "bf16"
    pose = lambda b: kps[b] if sc.policy == "prsink" else np.zeros((17, 2), np.float32)
    fill = lambda layer, blk: tuple(H.torch_values(sc, layer, blk, S - 1)[1:])
    fused, percall = H.make_cache(scl, attn_impl=1), H.make_cache(scl, attn_impl=1)
    T, Hh, D = sc.tokens_per_block, sc.num_heads, sc.head_dim
    for b in range(n):
        q, k, v = _tensors(sc, L, S, b)
        out_f = [torch.empty_like(x) for x in q]
        fused.la_stream_step(pose(b), S, q, k, v, out_f, fill=fill)
        ctx = percall.la_select_context(pose(b) if sc.policy == "prsink" else None)
        for i, blk in enumerate(ctx["dyn_ids"]):
            if ctx["need_fill"][i]:
                for l in range(L):
                    percall.la_fill_block(l, blk, *fill(l, blk))
        out_p = [torch.empty_like(x) for x in q]
        for i in range(S * L):
            percall.la_chunk_attention(i % L, q[i], k[i], v[i], out_p[i])
        for l in range(L):
            percall.la_cache_append_block(l, k[(S - 1) * L + l], v[(S - 1) * L + l])
        torch.cuda.synchronize()
        for i in range(S * L):
            assert torch.equal(out_f[i], out_p[i]), (b, i)
        if b in checks:
            assert ctx["kv_len"] == ref[b].kv_len
            if sc.policy == "prsink" and ctx["dyn_ids"] != ref[b].dyn_ids:
                assert ref[b].gap <= 1e-6
                continue
            for i in range(S * L):
                s_, l = divmod(i, L)
                o = H.oracle_output(sc, ref[b], vals, l, s_, S, w_kv=w[l])
                H.compare(out_f[i].float().cpu().numpy(), o, kind, f"block {b} step {s_} layer {l}")
    for cache in (fused, percall):
        st, msg = cache.la_get_error()
        assert st == capi.LA_OK, msg
    # pages of the last committed blocks (window), byte for byte
    elt = {"bf16": 2, "e4m3": 1}[sc.kv_dtype]
    for blk in range(max(0, n - sc.window), n):
        for l in range(L):
            for which in range(3 if sc.policy == "convkv" else 2):
                pf, sf = fused.la_debug_page(l, blk, which)
                pp, sp = percall.la_debug_page(l, blk, which)
                nb = T * Hh * D * elt
                assert torch.equal(fused.view(pf, nb), percall.view(pp, nb)), (blk, l, which)
                if sf:
                    assert torch.equal(fused.view(sf, 4 * Hh), percall.view(sp, 4 * Hh))


def test_stream_step_matches_per_call_bf16():
    _compare(C2_MID.with_(num_heads=4, grid_h=13, grid_w=15), 8)


def test_stream_step_matches_per_call_e4m3_external():
    _compare(C5_FP8.with_(num_heads=3, grid_h=6, grid_w=10), 10)


def test_stream_step_matches_per_call_convkv():
    # 135 tokens per block -> 27 compressed per eviction: the 240-slot memory
    # is full from block 12
    _compare(C4_CONVKV.with_(num_heads=4, grid_h=5, grid_w=9, mem_slots=240), 14)
