"""Degenerate inputs of the method on the GPU path: exact ties and zero-norm
poses in the retrieval, no dynamic sink, no static sink, and the most slots
the C ABI takes."""
import numpy as np
import pytest

from oracle import pose as opose
from oracle import stream as ostream
from synth import C2_MID, gen

from . import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bounded_kv_cache_la_b300 import build
    build.build()


def _tie_poses(n_blocks):
    """Poses drawn from 4 fixed templates plus one with every keypoint at the
    same point (zero-norm descriptor, score 0 against anything), repeated
    exactly, so most scores tie exactly."""
    rng = np.random.default_rng(11)
    templates = [rng.uniform(0.2, 0.8, size=(17, 2)) for _ in range(4)]
    templates.append(np.full((17, 2), 0.5))
    order = [0, 1, 2, 3, 4, 2, 0, 4, 1, 3]
    return np.stack([templates[order[b % len(order)]] for b in range(n_blocks)]).astype(np.float32)


@pytest.mark.parametrize("k", [1, 3, 8])
def test_retrieval_exact_ties_and_zero_norm_poses(k):
    """Ids bit-exact on every block, exact ties included: equal scores go to
    the lower block id, zero-norm poses score 0."""
    import torch
    sc = C2_MID.with_(num_heads=1, frames_per_block=1, grid_h=2, grid_w=4, dyn_topk=k)
    n = 40
    kps = _tie_poses(n)
    assert opose.descriptor(kps[4]).any() == False            # noqa: E712 -- the zero pose
    cache = H.make_cache(sc, attn_impl=1)
    ref = ostream.plan_stream(sc, kps, n)
    T, D = sc.tokens_per_block, sc.head_dim
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    ties = 0
    for b in range(n):
        ctx = cache.la_select_context(kps[b])
        assert ctx["dyn_ids"] == ref[b].dyn_ids, (b, ctx["dyn_ids"], ref[b].dyn_ids, ref[b].dyn_scores)
        np.testing.assert_allclose(ctx["dyn_scores"][:len(ref[b].dyn_ids)], ref[b].dyn_scores, atol=2e-6)
        assert ctx["kv_len"] == ref[b].kv_len
        ties += ref[b].gap == 0.0
        kk = torch.randn((T, 1, D), generator=g, device="cuda").to(torch.bfloat16)
        cache.la_cache_append_block(0, kk, kk)
    torch.cuda.synchronize()
    st, msg = cache.la_get_error()
    assert st == 0, msg
    assert ties > 10                      # the stream really exercised exact ties


@pytest.mark.parametrize("sink,k", [(1, 0), (0, 1), (0, 0)])
def test_without_dynamic_or_static_sink(sink, k):
    """PR-Sink with the dynamic sink or the static sink (or both) switched off:
    the context is then the window (plus sink) and the current block."""
    sc = C2_MID.with_(num_heads=2, frames_per_block=2, grid_h=6, grid_w=9, static_sink=sink,
                      dyn_topk=k)
    _, ctxs, outs = H.run_stream(sc, 9, {0, 3, 8}, attn_impl=1)
    ref = ostream.plan_stream(sc, gen.poses(sc, n_blocks=9), 9)
    assert ctxs[8]["n_slots"] == sink + k + sc.window + 1
    vals = H.Values(sc)
    for b in (0, 3, 8):
        assert ctxs[b]["kv_len"] == ref[b].kv_len
        if ctxs[b]["dyn_ids"] != ref[b].dyn_ids:
            assert ref[b].gap <= 1e-6
            continue
        o = H.oracle_output(sc, ref[b], vals, 0, 0, 1)
        H.compare(outs[b][(0, 0)], o, "bf16", f"block {b}")


def test_sixteen_slots():
    """Static sink + top-8 + a window of 6 + current = 16 slots, the most the
    C ABI takes; tensor path against the oracle once the context is full."""
    sc = C2_MID.with_(num_heads=2, frames_per_block=1, grid_h=10, grid_w=13, dyn_topk=8,
                      window=6)                                   # 130 tokens per block
    n = 17
    _, ctxs, outs = H.run_stream(sc, n, {16}, attn_impl=1)
    ref = ostream.plan_stream(sc, gen.poses(sc, n_blocks=n), n)
    assert ctxs[16]["n_slots"] == 16 and ctxs[16]["kv_len"] == 16 * sc.tokens_per_block
    vals = H.Values(sc)
    if ctxs[16]["dyn_ids"] == ref[16].dyn_ids:
        o = H.oracle_output(sc, ref[16], vals, 0, 0, 1)
        H.compare(outs[16][(0, 0)], o, "bf16", "block 16")
    else:
        assert ref[16].gap <= 1e-6


@pytest.mark.parametrize("impl", [1, 2], ids=["tensor", "simt"])
def test_misaligned_tensors_rejected_cache_stays_usable(impl):
    """Q/K/V/O pointers that are not 16-byte aligned are refused before any
    work is enqueued (the kernels move rows in 16-byte vectors), and the
    cache goes on working with aligned ones."""
    import torch
    from bounded_kv_cache_la_b300 import capi
    sc = C2_MID.with_(num_heads=2, grid_h=4, grid_w=4)
    cache = H.make_cache(sc.with_(num_layers=1), attn_impl=impl)
    kps = gen.poses(sc, n_blocks=2)
    cache.la_select_context(kps[0])
    q, k, v = H.torch_values(sc, 0, 0, 0)
    out = torch.empty_like(q)
    buf = torch.zeros(q.numel() + 8, dtype=q.dtype, device="cuda")
    shifted = buf[2:2 + q.numel()].view_as(q)            # 4 bytes past a 16-byte boundary
    shifted.copy_(q)
    for args in ((shifted, k, v, out), (q, shifted, v, out), (q, k, shifted, out),
                 (q, k, v, shifted)):
        with pytest.raises(capi.LaError) as e:
            cache.la_chunk_attention(0, *args)
        assert e.value.status == capi.LA_ERR_INVALID_ARG
    with pytest.raises(capi.LaError) as e:
        cache.la_cache_append_block(0, shifted, v)
    assert e.value.status == capi.LA_ERR_INVALID_ARG
    cache.la_chunk_attention(0, q, k, v, out)
    cache.la_cache_append_block(0, k, v)
    torch.cuda.synchronize()
    st, msg = cache.la_get_error()
    assert st == capi.LA_OK, msg
