"""GPU parity: the C-ABI path against the CPU oracle on the same seeded
inputs (retrieval ids bit-exact where the top-k gap allows, stored pages,
ConvKV memory, attention outputs within the stated tolerances)."""
import numpy as np
import pytest

from bounded_kv_cache_la_b300 import capi
from oracle import e4m3, rope, stream as ostream
from synth import C1_TINY, C2_MID, C3_14B, C4_CONVKV, C5_FP8, gen

from . import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bounded_kv_cache_la_b300 import build
    build.build()


def _check_selection(sc, ctxs, n):
    """Ids bit-exact wherever the oracle's k-th/(k+1)-th gap exceeds 1e-6."""
    ref = ostream.plan_stream(sc, gen.poses(sc, n_blocks=n), n)
    exact = 0
    for got, want in zip(ctxs, ref):
        assert got["kv_len"] == want.kv_len
        assert got["t0"] == want.t0
        if want.gap > 1e-6:
            assert got["dyn_ids"] == want.dyn_ids, (want.block, got, want)
            assert got["blocks"] == want.blocks
            np.testing.assert_allclose(got["dyn_scores"], want.dyn_scores, atol=1e-5)
            exact += 1
    return ref, exact


def test_generator_torch_cuda_matches_numpy():
    import torch
    key = gen.qkv_key(C2_MID, 0, 3, 0, "k")
    a = gen.tensor_np(key, (300, 12, 128), "bf16")
    b = gen.tensor_torch(key, (300, 12, 128), "bf16", "cuda").float().cpu().numpy()
    np.testing.assert_array_equal(a, b)


def test_c1_tiny_full_stream_simt():
    """c1: all 24 blocks, all rows, fp32 path."""
    sc = C1_TINY
    cache, ctxs, outs = H.run_stream(sc, 24, set(range(24)))
    ref, exact = _check_selection(sc, ctxs, 24)
    assert exact >= 18
    vals = H.Values(sc)
    for ctx in ref:
        o = H.oracle_output(sc, ctx, vals, 0, 0, 1)
        H.compare(outs[ctx.block][(0, 0)], o, "f32", f"block {ctx.block}")


def test_c2_mid_stream_simt_and_pages():
    sc = C2_MID
    keep = {0, 1, 2, 4, 5, 6, 9, 12, 20, 33, 63}
    cache, ctxs, outs = H.run_stream(sc, 64, keep, attn_impl=2)
    ref, exact = _check_selection(sc, ctxs, 64)
    assert exact >= 55
    heads = [0, 5, 11]
    vals = H.Values(sc, heads)
    rows = np.r_[0:200, 1400:1560]
    for b in sorted(keep):
        ctx = ref[b]
        if ctx.gap <= 1e-6 and ctx.dyn_ids:
            continue
        o = H.oracle_output(sc, ctx, vals, 0, 0, 1, rows=rows)
        H.compare(outs[b][(0, 0)][rows][:, heads], o, "bf16", f"block {b}")
    # stored pages of block 7: values verbatim, keys turned by the within-block position
    import torch
    T, Hh, D = sc.tokens_per_block, sc.num_heads, sc.head_dim
    kp, _ = cache.la_debug_page(0, 7, 0)
    vp, _ = cache.la_debug_page(0, 7, 1)
    kpage = cache.view(kp, T * Hh * D * 2).view(torch.bfloat16).view(Hh, T, D).float().cpu().numpy()
    vpage = cache.view(vp, T * Hh * D * 2).view(torch.bfloat16).view(Hh, T, D).float().cpu().numpy()
    full = H.Values(sc)
    v_ref = full.get(0, 7, 0, "v").transpose(1, 0, 2)
    np.testing.assert_array_equal(vpage, v_ref)
    k_raw = full.get(0, 7, 0, "k")
    k_ref = ostream.rotate_within_block_f32(k_raw, sc)          # fp32 single roundings
    k_ref = ostream.bf16_round(k_ref.astype(np.float64)).transpose(1, 0, 2)
    same = np.mean(kpage == k_ref)
    assert same > 0.999, same
    np.testing.assert_allclose(kpage, k_ref, rtol=2 ** -7, atol=1e-30)


def test_external_history_retrieval_at_10000_blocks():
    """c5 pose workload: 10000-block history loaded, retrieval at block 10000
    matches the oracle."""
    sc = C5_FP8.with_(grid_h=4, grid_w=4, num_heads=2)
    import torch
    n = 10000
    kps = gen.poses(sc, n_blocks=n + 1)
    cache = H.make_cache(sc.with_(num_layers=1), max_history=n + 8)
    cache.la_cache_load_history(kps[:n].reshape(n, 34))
    from oracle import pose
    descs = np.stack([pose.descriptor(k) for k in kps[:n + 1]])
    for b in (n,):
        # the window and sink must hold pages before attention; selection alone needs none
        ctx = cache.la_select_context(kps[b])
        want = ostream.plan_prsink(sc, b, descs[:b], descs[b])
        assert ctx["kv_len"] == want.kv_len
        if want.gap > 1e-6:
            assert ctx["dyn_ids"] == want.dyn_ids
        np.testing.assert_allclose(ctx["dyn_scores"], want.dyn_scores, atol=1e-5)


def test_convkv_memory_and_attention():
    """ConvKV at reduced size: memory rings equal the oracle's FIFO of
    compressed tokens; attention over memory + window + current."""
    sc = C4_CONVKV.with_(num_heads=4, grid_h=5, grid_w=9, mem_slots=240)
    _convkv_case(sc, 16, {0, 3, 4, 8, 12, 15})        # 135 tokens -> 27 per eviction


@pytest.mark.parametrize("kernel,stride", [(3, 2), (4, 4), (7, 5)])
def test_convkv_other_kernel_sizes(kernel, stride):
    """Kernel sizes other than 5 (the per-tap weight path), windows that
    overlap (3/2), tile (4/4) or reach past the stride (7/5), and evictions
    that do not divide the block evenly."""
    sc = C4_CONVKV.with_(num_heads=3, grid_h=5, grid_w=9, mem_slots=200, conv_kernel=kernel,
                         conv_stride=stride)
    _convkv_case(sc, 12, {4, 8, 11})


def _convkv_case(sc, n, keep):
    import torch
    cache, ctxs, outs = H.run_stream(sc, n, keep, n_steps=2)
    vals = H.Values(sc)
    w = gen.conv_weights_np(sc, 0)
    for b in range(n):
        want = ostream.plan_convkv(sc, b)
        assert ctxs[b]["kv_len"] == want.kv_len
        assert ctxs[b]["mem_tokens"] == want.mem_tokens
    for b in sorted(keep):
        ctx = ostream.plan_convkv(sc, b)
        for s in range(2):
            o = H.oracle_output(sc, ctx, vals, 0, s, 2, w_kv=w)
            H.compare(outs[b][(0, s)], o, "bf16", f"block {b} step {s}")
    # memory after the stream: blocks 0..n-4 evicted
    kraw, vr, krot, n_tok, oldest = cache.la_debug_memory(0)
    kv_of = vals.kv_of(0, lambda b: 1)
    km, vm = ostream.convkv_memory(sc, n, kv_of, w)
    cap, Hh, D = sc.mem_slots, sc.num_heads, sc.head_dim
    assert n_tok == km.shape[0] == cap
    ring_idx = (oldest + np.arange(n_tok)) % cap
    kring = cache.view(kraw, Hh * cap * D * 2).view(torch.bfloat16).view(Hh, cap, D).float().cpu().numpy()
    vring = cache.view(vr, Hh * cap * D * 2).view(torch.bfloat16).view(Hh, cap, D).float().cpu().numpy()
    got_k = kring[:, ring_idx].transpose(1, 0, 2)
    got_v = vring[:, ring_idx].transpose(1, 0, 2)
    # fp32 accumulation then bf16: within one bf16 ulp of the fp64 sum rounded
    np.testing.assert_allclose(got_k, km, rtol=2 ** -7, atol=1e-6)
    np.testing.assert_allclose(got_v, vm, rtol=2 ** -7, atol=1e-6)
    assert np.mean(got_k == km) > 0.99


def test_fp8_pages_and_attention_simt():
    import torch
    sc = C5_FP8.with_(grid_h=6, grid_w=10, num_heads=3, n_blocks=14, history_mode="resident")
    keep = {0, 5, 9, 13}
    cache, ctxs, outs = H.run_stream(sc, 14, keep, attn_impl=2)
    ref, _ = _check_selection(sc, ctxs, 14)
    vals = H.Values(sc)
    for b in sorted(keep):
        ctx = ref[b]
        if ctx.gap <= 1e-6 and ctx.dyn_ids:
            continue
        o = H.oracle_output(sc, ctx, vals, 0, 0, 1)
        H.compare(outs[b][(0, 0)], o, "e4m3", f"block {b}")
    # codes and scales of block 6
    T, Hh, D = sc.tokens_per_block, sc.num_heads, sc.head_dim
    kp, ks = cache.la_debug_page(0, 6, 0)
    vp, vs = cache.la_debug_page(0, 6, 1)
    kc = cache.view(kp, T * Hh * D).view(Hh, T, D).cpu().numpy().transpose(1, 0, 2)
    vc = cache.view(vp, T * Hh * D).view(Hh, T, D).cpu().numpy().transpose(1, 0, 2)
    kscale = cache.view(ks, 4 * Hh).view(torch.float32).cpu().numpy()
    vscale = cache.view(vs, 4 * Hh).view(torch.float32).cpu().numpy()
    k_raw = vals.get(0, 6, 0, "k")
    v_raw = vals.get(0, 6, 0, "v")
    rk, sk, _, yk = ostream.fp8_store(ostream.rotate_within_block_f32(k_raw, sc))
    rv, sv, _, yv = ostream.fp8_store(v_raw.astype(np.float32))
    np.testing.assert_array_equal(vc, rv)
    np.testing.assert_array_equal(vscale, sv)
    np.testing.assert_array_equal(kscale, sk)
    decided = e4m3.boundary_distance(yk) > 1e-6
    np.testing.assert_array_equal(kc[decided], rk[decided])


def test_call_order_errors():
    from bounded_kv_cache_la_b300 import capi
    import torch
    sc = C1_TINY
    cache = H.make_cache(sc)
    q, k, v = H.torch_values(sc, 0, 0, 0)
    out = torch.empty_like(q)
    with pytest.raises(capi.LaError) as e:
        cache.la_chunk_attention(0, q, k, v, out)          # before select
    assert e.value.status == capi.LA_ERR_STATE
    with pytest.raises(capi.LaError):
        cache.la_cache_append_block(0, k, v)
    cache.la_select_context(gen.poses(sc)[0])
    with pytest.raises(capi.LaError) as e:
        cache.la_select_context(gen.poses(sc)[0])          # twice
    assert e.value.status == capi.LA_ERR_STATE
    with pytest.raises(capi.LaError) as e:
        cache.la_chunk_attention(5, q, k, v, out)          # bad layer
    assert e.value.status == capi.LA_ERR_INVALID_ARG
    cache.la_chunk_attention(0, q, k, v, out)
    cache.la_cache_append_block(0, k, v)
    st, msg = cache.la_get_error()
    assert st == capi.LA_OK, msg
    bad = np.full(34, np.nan, np.float32)
    with pytest.raises(capi.LaError) as e:
        cache.la_select_context(bad)
    assert e.value.status == capi.LA_ERR_INVALID_ARG


def test_history_load_rows_equal_retrieval_rows():
    """la_cache_load_history writes every pose row in one launch; the rows
    must be bit-identical to those the retrieval kernel writes block by
    block (here through la_pose_topk_noalloc), so the scores agree exactly."""
    import torch
    sc = C5_FP8.with_(grid_h=4, grid_w=4, num_heads=2)
    n = 700
    kps = gen.poses(sc, n_blocks=n + 1)
    cache = H.make_cache(sc.with_(num_layers=1), max_history=n + 8)
    cache.la_cache_load_history(kps[:n].reshape(n, 34))
    ctx = cache.la_select_context(kps[n])
    table = torch.zeros((n + 1, 36), dtype=torch.float32, device="cuda")
    inv = torch.zeros(n + 1, dtype=torch.float32, device="cuda")
    k = sc.dyn_topk
    ids = torch.empty(k + 1, dtype=torch.int32, device="cuda")
    scores = torch.empty(k + 1, dtype=torch.float32, device="cuda")
    n_out = torch.empty(1, dtype=torch.int32, device="cuda")
    status = torch.empty(1, dtype=torch.int32, device="cuda")
    for b in range(n):
        capi.la_pose_topk_noalloc(table, inv, kps[b], b, 0, 0, 0, ids, scores, n_out, status)
    capi.la_pose_topk_noalloc(table, inv, kps[n], n, 1, n - sc.window, k, ids, scores, n_out,
                              status)
    torch.cuda.synchronize()
    assert int(status.item()) == capi.LA_OK
    got = sorted(zip(ids.cpu().numpy()[:k].tolist(), scores.cpu().numpy()[:k].tolist()))
    assert [g[0] for g in got] == ctx["dyn_ids"]
    assert [np.float32(g[1]) for g in got] == [np.float32(x) for x in ctx["dyn_scores"]]


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_head_dim_64_cuda_cores(kv):
    """Head dim 64 with bf16 operands (bf16 or e4m3 cache) goes through the
    CUDA-core kernel: blocks of 3 x 5 x 7 = 105 tokens (each slot ends in a
    partial 32-key tile, the last 16-row query tile is partial), all rows
    against the oracle, before and after the dynamic sink fills."""
    sc = C1_TINY.with_(qkv_dtype="bf16", kv_dtype=kv, frames_per_block=3, grid_h=5, grid_w=7,
                       num_heads=3)
    keep = {0, 4, 6, 9}
    _, ctxs, outs = H.run_stream(sc, 10, keep)
    ref = ostream.plan_stream(sc, gen.poses(sc, n_blocks=10), 10)
    vals = H.Values(sc)
    for b in sorted(keep):
        ctx = ref[b]
        assert ctxs[b]["kv_len"] == ctx.kv_len
        if ctxs[b]["dyn_ids"] != ctx.dyn_ids:
            assert ctx.gap <= 1e-6
            continue
        o = H.oracle_output(sc, ctx, vals, 0, 0, 1)
        H.compare(outs[b][(0, 0)], o, "bf16" if kv == "bf16" else "e4m3", f"block {b}")
