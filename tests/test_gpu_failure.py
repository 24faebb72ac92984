"""Failure detection without a GPU fault: a tensor-core attention launch is
made to wait on a barrier that nothing completes (a 0.1 s limit); the
kernel must report LA_ERR_TIMEOUT through the error word, exit cleanly
(copies drained, tensor memory freed), and leave the CUDA context usable.
And a slot table naming a frame past the pool must be caught by the
attention kernels' bounds check before any load."""
import time

import numpy as np
import pytest

from bounded_kv_cache_la_b300 import capi
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


def test_stalled_wait_is_reported_and_context_survives():
    import torch
    sc = C2_MID.with_(num_heads=2, grid_h=6, grid_w=11)          # 132 tokens
    cache = H.make_cache(sc.with_(num_layers=1), attn_impl=1)
    kps = gen.poses(sc, n_blocks=3)
    cache.la_select_context(kps[0])
    q, k, v = H.torch_values(sc, 0, 0, 0)
    out = torch.empty_like(q)
    cache.la_debug_inject(capi.LA_INJECT_ATTN_STALL, 1)
    t0 = time.perf_counter()
    cache.la_chunk_attention(0, q, k, v, out)
    st, msg = cache.la_get_error()                              # synchronises the device
    elapsed = time.perf_counter() - t0
    assert st == capi.LA_ERR_TIMEOUT, msg
    assert "kernel 5" in msg                                    # the tensor-core attention
    assert elapsed < 10.0
    with pytest.raises(capi.LaError) as e:                       # the cache stays failed
        cache.la_chunk_attention(0, q, k, v, out)
    assert e.value.status == capi.LA_ERR_STATE
    cache.close()
    # the context is still usable: a fresh cache gives oracle-matching output
    _, ctxs, outs = H.run_stream(sc, 3, {2}, attn_impl=1)
    ctx = ostream.plan_stream(sc, kps, 3)[2]
    o = H.oracle_output(sc, ctx, H.Values(sc), 0, 0, 1)
    H.compare(outs[2][(0, 0)], o, "bf16", "after the injected timeout")


def test_inject_rules():
    sc = C2_MID.with_(num_heads=2, grid_h=4, grid_w=4)
    cache = H.make_cache(sc.with_(num_layers=1), attn_impl=2)   # CUDA-core kernel: no waits
    with pytest.raises(capi.LaError) as e:
        cache.la_debug_inject(capi.LA_INJECT_ATTN_STALL, 1)
    assert e.value.status == capi.LA_ERR_UNSUPPORTED
    tc = H.make_cache(sc.with_(num_layers=1), attn_impl=1)
    with pytest.raises(capi.LaError) as e:
        tc.la_debug_inject(99, 1)
    assert e.value.status == capi.LA_ERR_INVALID_ARG


@pytest.mark.parametrize("impl,kid", [(1, 5), (2, 4)])
def test_bad_frame_is_caught_before_any_load(impl, kid):
    """An attention launch gets a slot table whose first slot names a frame
    past the pool (la_debug_inject): the kernel (tensor-core: kernel 5,
    CUDA-core: kernel 4) rejects it, the error word reports LA_ERR_DEVICE,
    later calls report LA_ERR_STATE, and a fresh cache on the same context
    matches the oracle."""
    import torch
    sc = C2_MID.with_(num_heads=2, grid_h=6, grid_w=11)          # 132 tokens
    cache, _, _ = H.run_stream(sc, 5, set(), attn_impl=impl)
    kps = gen.poses(sc, n_blocks=6)
    cache.la_select_context(kps[5])
    q, k, v = H.torch_values(sc, 0, 5, 0)
    out = torch.empty_like(q)
    cache.la_debug_inject(capi.LA_INJECT_BAD_FRAME, 1)
    cache.la_chunk_attention(0, q, k, v, out)
    st, msg = cache.la_get_error()
    assert st == capi.LA_ERR_DEVICE, msg
    assert f"kernel {kid}" in msg, msg
    with pytest.raises(capi.LaError) as e:
        cache.la_chunk_attention(0, q, k, v, out)
    assert e.value.status == capi.LA_ERR_STATE
    cache.close()
    _, _, outs = H.run_stream(sc, 3, {2}, attn_impl=impl)
    ctx = ostream.plan_stream(sc, gen.poses(sc, n_blocks=3), 3)[2]
    o = H.oracle_output(sc, ctx, H.Values(sc), 0, 0, 1)
    H.compare(outs[2][(0, 0)], o, "bf16", "after the injected bad frame")
