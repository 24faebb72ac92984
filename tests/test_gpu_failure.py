"""Failure detection without a GPU fault: a tensor-core attention launch is
made to wait on a barrier that nothing completes (a 0.1 s limit); the
kernel must report LA_ERR_TIMEOUT through the error word, exit cleanly
(copies drained, tensor memory freed), and leave the CUDA context usable."""
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
