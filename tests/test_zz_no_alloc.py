"""The allocation-free pose retrieval (la_pose_topk_noalloc) against the
cache's own retrieval (la_select_context), through the C ABI.

Some callers cannot call cudaMalloc when they need a retrieval (a host that
forbids allocation once serving has started, or a real-time path where an
allocation's implicit synchronisation would stall the stream).  For them the
library runs the same retrieval kernel with its scratch in a fixed device
array instead of the cache pool.  This file runs last so that a stop at the
first failure has already run every other test; it passes alone in a fresh
process too (the library looks the array up on its first call).
"""
import numpy as np
import pytest

from bounded_kv_cache_la_b300 import capi
from synth import C5_FP8, gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bounded_kv_cache_la_b300 import build
    build.build()


def _ranked(ids, scores, n_found, k):
    """(chosen ids ascending, their scores, gap) from a ranked list."""
    ids = [int(x) for x in ids[:n_found]]
    scores = [float(x) for x in scores[:n_found]]
    gap = scores[k - 1] - scores[k] if n_found > k and k > 0 else np.inf
    pairs = sorted(zip(ids[:k], scores[:k]))
    return [p[0] for p in pairs], [p[1] for p in pairs], gap


def _outputs(k):
    """ids, scores, n_out, status on the device; status starts at a value
    the call must overwrite."""
    import torch
    ids = torch.empty(k + 1, dtype=torch.int32, device="cuda")
    scores = torch.empty(k + 1, dtype=torch.float32, device="cuda")
    n_out = torch.empty(1, dtype=torch.int32, device="cuda")
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    return ids, scores, n_out, status


def test_noalloc_retrieval_matches_select_context():
    import torch
    # 50 repeating pose clusters, top-4: every block after the warm-up has
    # many candidates.  Tiny pages: only the retrieval is under test.
    sc = C5_FP8.with_(grid_h=4, grid_w=4, num_heads=2, kv_dtype="bf16", n_blocks=48,
                      history_mode="resident", num_layers=1)
    n, k = sc.n_blocks, sc.dyn_topk
    cfg = capi.config_for(sc, max_history=n)
    cache = capi.Cache(cfg)
    kps = gen.poses(sc, n_blocks=n)
    T, Hh, D = sc.tokens_per_block, sc.num_heads, sc.head_dim
    kv = torch.zeros((T, Hh, D), dtype=torch.bfloat16, device="cuda")

    # caller-owned buffers only; the call itself allocates nothing
    table = torch.zeros((n, 36), dtype=torch.float32, device="cuda")
    inv_norm = torch.zeros(n, dtype=torch.float32, device="cuda")
    ids, scores, n_out, status = _outputs(k)

    consecutive = best = 0
    for b in range(n):
        ctx = cache.la_select_context(kps[b])
        c0 = 1
        c1 = max(c0, b - sc.window)
        status.fill_(12345)
        capi.la_pose_topk_noalloc(table, inv_norm, kps[b], b, c0, c1, k, ids, scores, n_out,
                                  status)
        torch.cuda.synchronize()
        assert int(status.item()) == capi.LA_OK
        n_found = int(n_out.item())
        assert n_found == min(k + 1, c1 - c0)
        got_ids = ids.cpu().numpy()
        assert (got_ids[n_found:] == -1).all(), (b, got_ids)      # ranks past the candidates
        got_ids, got_scores, gap = _ranked(got_ids, scores.cpu().numpy(), n_found, k)
        if ctx["gap"] > 1e-6:
            assert got_ids == ctx["dyn_ids"], (b, got_ids, ctx)
        np.testing.assert_allclose(sorted(got_scores), sorted(ctx["dyn_scores"]), atol=1e-5)
        if np.isfinite(ctx["gap"]):
            assert abs(gap - ctx["gap"]) <= 1e-5
        consecutive = consecutive + 1 if c1 > c0 else 0
        best = max(best, consecutive)
        cache.la_cache_append_block(0, kv, kv)
    assert best >= 2                     # at least two scored calls in a row
    st, msg = cache.la_get_error()
    assert st == capi.LA_OK, msg


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import torch
    rows = capi.LA_NOALLOC_MAX_ROWS + 1
    table = torch.zeros((rows, 36), dtype=torch.float32, device="cuda")
    inv_norm = torch.zeros(rows, dtype=torch.float32, device="cuda")
    ids, scores, n_out, status = _outputs(1)
    kp = np.full((17, 2), 0.5, np.float32)
    with pytest.raises(capi.LaError) as e:
        capi.la_pose_topk_noalloc(table, inv_norm, kp, -1, 0, rows, 1, ids, scores, n_out, status)
    assert e.value.status == capi.LA_ERR_INVALID_ARG
    # the query's own row inside the candidate range: rejected before any work
    for row in (0, 5, rows - 2):
        with pytest.raises(capi.LaError) as e:
            capi.la_pose_topk_noalloc(table, inv_norm, kp, row, 0, rows - 1, 1, ids, scores,
                                      n_out, status)
        assert e.value.status == capi.LA_ERR_INVALID_ARG
    # at the limit it runs: 65536 all-zero rows tie at score 0, and the
    # lowest ids win the tie
    capi.la_pose_topk_noalloc(table, inv_norm, kp, -1, 0, rows - 1, 1, ids, scores, n_out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == capi.LA_OK
    assert int(n_out.item()) == 2
    assert ids.cpu().tolist() == [0, 1]
    assert scores.cpu().tolist() == [0.0, 0.0]


def test_noalloc_ids_are_table_rows():
    """Candidates [c0, c1) with c0 > 0: the ids returned are table rows, and
    ranks past the candidates read -1."""
    import torch
    n = 40
    table = torch.zeros((n, 36), dtype=torch.float32, device="cuda")
    inv_norm = torch.zeros(n, dtype=torch.float32, device="cuda")
    rng = np.random.default_rng(3)
    kps = rng.uniform(0.2, 0.8, size=(n, 17, 2)).astype(np.float32)
    k = 4
    ids, scores, n_out, status = _outputs(k)
    for b in range(n):                       # write every row (no candidates)
        capi.la_pose_topk_noalloc(table, inv_norm, kps[b], b, 0, 0, k, ids, scores, n_out, status)
    # the query equals row 23's pose: row 23 must rank first, by its table id
    capi.la_pose_topk_noalloc(table, inv_norm, kps[23], -1, 20, 30, k, ids, scores, n_out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == capi.LA_OK
    assert int(n_out.item()) == k + 1
    got = ids.cpu().tolist()
    assert got[0] == 23 and all(20 <= i < 30 for i in got), got
    assert abs(float(scores[0].item()) - 1.0) < 1e-5
    # two candidates, four picks: ranks 2.. hold -1
    capi.la_pose_topk_noalloc(table, inv_norm, kps[23], -1, 22, 24, k, ids, scores, n_out, status)
    torch.cuda.synchronize()
    assert int(n_out.item()) == 2
    got = ids.cpu().tolist()
    assert got[0] == 23 and got[1] == 22 and got[2:] == [-1] * (k - 1), got
