"""Checkpoint and resume between blocks (la_cache_save_state /
la_cache_restore): a stream saved after block n1 and resumed on a fresh pool
(another device address) gives outputs bit-identical to the uninterrupted
stream, for PR-Sink with EXTERNAL history (frames, fills, dynamic sink) and
for ConvKV (ring position)."""
import ctypes

import numpy as np
import pytest

from bounded_kv_cache_la_b300 import capi
from synth import C3_14B, C4_CONVKV, gen

from . import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bounded_kv_cache_la_b300 import build
    build.build()


def _drive(cache, sc, kps, blocks, n_steps=2):
    """select / fills / attention per step / appends for the given blocks;
    returns {block: [outputs per step]} (CPU float32)."""
    import torch
    outs = {}
    for b in blocks:
        ctx = cache.la_select_context(kps[b] if sc.policy == "prsink" else None)
        for i, bid in enumerate(ctx["dyn_ids"]):
            if ctx["need_fill"][i]:
                _, k, v = H.torch_values(sc, 0, bid, n_steps - 1)
                cache.la_fill_block(0, bid, k, v)
        got = []
        for s in range(n_steps):
            q, k, v = H.torch_values(sc, 0, b, s)
            out = torch.empty_like(q)
            cache.la_chunk_attention(0, q, k, v, out)
            got.append(out.float().cpu().numpy())
        _, k, v = H.torch_values(sc, 0, b, n_steps - 1)
        cache.la_cache_append_block(0, k, v)
        outs[b] = got
    torch.cuda.synchronize()
    st, msg = cache.la_get_error()
    assert st == capi.LA_OK, msg
    return outs


def _conv_w(sc):
    import torch
    if sc.policy != "convkv":
        return None
    return torch.stack([gen.conv_weights_torch(sc, 0, "cuda")]).contiguous()


@pytest.mark.parametrize("sc,n1,n", [
    (C3_14B.with_(num_layers=1, num_heads=2, frames_per_block=2, grid_h=6, grid_w=9, n_steps=2), 9, 14),
    (C4_CONVKV.with_(num_layers=1, num_heads=2, grid_h=5, grid_w=9, mem_slots=120, n_steps=2), 8, 13),
])
def test_resume_matches_uninterrupted_stream(sc, n1, n):
    kps = gen.poses(sc, n_blocks=n)
    cfg = capi.config_for(sc, max_history=n + 2, attn_impl=1)
    w = _conv_w(sc)
    ref = _drive(capi.Cache(cfg, conv_w=w), sc, kps, range(n))

    first = capi.Cache(cfg, conv_w=w)
    _drive(first, sc, kps, range(n1))
    pool, state = first.save_checkpoint()
    first.close()
    del first
    pad = capi.Cache(cfg, conv_w=w)          # keeps the old address taken: a new pool elsewhere
    resumed = capi.Cache(cfg, conv_w=w, restore=(pool, state))
    got = _drive(resumed, sc, kps, range(n1, n))
    for b in range(n1, n):
        for s in range(len(ref[b])):
            np.testing.assert_array_equal(got[b][s], ref[b][s], err_msg=f"block {b} step {s}")
    pad.close()


def test_checkpoint_rules():
    import torch
    sc = C3_14B.with_(num_layers=1, num_heads=2, frames_per_block=1, grid_h=4, grid_w=4)
    kps = gen.poses(sc, n_blocks=6)
    cfg = capi.config_for(sc, max_history=8, attn_impl=1)
    cache = capi.Cache(cfg)
    _drive(cache, sc, kps, range(3), n_steps=1)
    cache.la_select_context(kps[3])
    n = cache.lib.la_cache_state_bytes(cache.h)
    buf = ctypes.create_string_buffer(n)
    assert cache.lib.la_cache_save_state(cache.h, buf, n) == capi.LA_ERR_STATE   # mid-block
    q, k, v = H.torch_values(sc, 0, 3, 0)
    out = torch.empty_like(q)
    cache.la_chunk_attention(0, q, k, v, out)
    cache.la_cache_append_block(0, k, v)
    assert cache.lib.la_cache_save_state(cache.h, buf, n - 1) == capi.LA_ERR_INVALID_ARG   # too small
    pool, state = cache.save_checkpoint()
    other = capi.config_for(sc.with_(dyn_topk=1), max_history=8, attn_impl=1)
    with pytest.raises(capi.LaError) as e:                     # another config
        capi.Cache(other, restore=(pool[:capi.la_cache_required_bytes(other)], state))
    assert e.value.status == capi.LA_ERR_INVALID_ARG
    with pytest.raises(capi.LaError) as e:                     # a truncated blob
        capi.Cache(cfg, restore=(pool, state[:-3]))
    assert e.value.status == capi.LA_ERR_INVALID_ARG
    bad = bytearray(state)
    bad[0] ^= 0xFF
    with pytest.raises(capi.LaError) as e:                     # not a state blob
        capi.Cache(cfg, restore=(pool, bytes(bad)))
    assert e.value.status == capi.LA_ERR_INVALID_ARG
    resumed = capi.Cache(cfg, restore=(pool, state))
    _drive(resumed, sc, kps, range(4, 6), n_steps=1)
