"""Pins for the oracle's pose descriptor and retrieval (not its own retyping)."""
import numpy as np
import pytest
from scipy.spatial import distance

from oracle import pose
from synth import C1_TINY, C3_14B, C5_FP8, gen


def test_descriptor_is_centred_and_flattened_xy():
    kp = np.arange(34, dtype=np.float64).reshape(17, 2)
    d = pose.descriptor(kp)
    assert d.shape == (34,)
    assert abs(d[0::2].sum()) < 1e-12 and abs(d[1::2].sum()) < 1e-12
    # x-coordinates are even entries: x_k = 2k, mean 16 -> x_0 - 16 = -16
    assert d[0] == -16.0 and d[1] == -16.0 and d[32] == 16.0


def test_cosine_matches_scipy_distance():
    rng = np.random.default_rng(3)
    q = rng.normal(size=34)
    P = rng.normal(size=(50, 34))
    got = pose.cosine_scores(q, P)
    ref = np.array([1.0 - distance.cosine(q, p) for p in P])
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_retrieval_identity_translation_and_scale():
    rng = np.random.default_rng(0)
    kps = rng.uniform(0, 1, size=(40, 17, 2))
    descs = np.stack([pose.descriptor(k) for k in kps])
    j_star = 17
    # query equal to a stored pose, then translated and scaled about its centre
    q = kps[j_star]
    q2 = (q - q.mean(0)) * 1.7 + q.mean(0) + np.array([0.13, -0.05])
    for query in (q, q2):
        s = pose.cosine_scores(pose.descriptor(query), descs)
        assert int(np.argmax(s)) == j_star
        assert abs(s[j_star] - 1.0) < 1e-12


def test_zero_norm_scores_zero():
    z = np.full((17, 2), 0.25)          # all keypoints equal: centred to zero
    d = pose.descriptor(z)
    P = np.random.default_rng(1).normal(size=(5, 34))
    assert np.all(pose.cosine_scores(d, P) == 0)
    assert np.all(pose.cosine_scores(P[0], np.stack([d, P[1]]))[0] == 0)


def _brute_force_topk(scores, ids, k):
    """Element i is selected iff fewer than k candidates beat it, where j
    beats i if it scores higher, or ties and has the lower id."""
    sel = []
    for i in range(len(ids)):
        beats = sum(1 for j in range(len(ids)) if j != i and
                    (scores[j] > scores[i] or (scores[j] == scores[i] and ids[j] < ids[i])))
        if beats < k:
            sel.append(ids[i])
    return sorted(sel)


@pytest.mark.parametrize("k", [1, 2, 4, 7])
def test_topk_matches_brute_force_with_ties(k):
    rng = np.random.default_rng(k)
    for trial in range(30):
        n = int(rng.integers(0, 12))
        ids = sorted(rng.choice(100, size=n, replace=False).tolist())
        scores = rng.integers(0, 4, size=n).astype(np.float64) / 4   # many ties
        got, got_s, gap = pose.select_topk(scores, ids, k)
        assert got == _brute_force_topk(scores, ids, k)
        assert got == sorted(got)
        assert len(got) == min(k, n)


def test_gap_definition():
    ids = [3, 5, 9, 11]
    scores = np.array([0.5, 0.9, 0.7, 0.7])
    got, got_s, gap = pose.select_topk(scores, ids, 2)
    assert got == [5, 9] and got_s == [0.9, 0.7]
    assert gap == 0.0                     # 9 and 11 tie; lower id wins
    got, _, gap = pose.select_topk(scores, ids, 1)
    assert got == [5] and abs(gap - 0.2) < 1e-15


def test_tiny_stream_brute_force_selection():
    """c1: every block's dynamic sink equals a brute force over all history."""
    from oracle import stream
    cfg = C1_TINY
    kps = gen.poses(cfg)
    ctxs = stream.plan_stream(cfg, kps)
    for ctx in ctxs:
        b = ctx.block
        cand = [j for j in range(1, b) if j < b - 3]
        if not cand:
            assert ctx.dyn_ids == []
            continue
        qd = pose.descriptor(kps[b])
        sc = [1.0 - distance.cosine(qd, pose.descriptor(kps[j])) for j in cand]
        assert ctx.dyn_ids == _brute_force_topk(sc, cand, cfg.dyn_topk)


def test_periodic_pose_recurs():
    """With a noise-free periodic pose, retrieval picks a block one period back
    (a block whose pose equals the query)."""
    cfg = C1_TINY.with_(pose=C1_TINY.pose.__class__("sinusoid", period=8, noise=0.0))
    from oracle import stream
    kps = gen.poses(cfg)
    for ctx in stream.plan_stream(cfg, kps):
        if ctx.block >= 12:
            assert (ctx.block - ctx.dyn_ids[0]) % 8 == 0
            assert abs(ctx.dyn_scores[0] - 1.0) < 1e-9


def test_cluster_poses_retrieve_same_cluster():
    cfg = C5_FP8
    kps = gen.poses(cfg, n_blocks=160)
    from oracle import stream
    ctxs = stream.plan_stream(cfg, kps, 160)
    for ctx in ctxs[60:]:
        same = [j for j in range(1, ctx.block - 3) if (ctx.block - j) % 50 == 0]
        assert 1 <= len(same) <= cfg.dyn_topk
        assert set(same) <= set(ctx.dyn_ids)
        s_same = [s for j, s in zip(ctx.dyn_ids, ctx.dyn_scores) if j in same]
        s_other = [s for j, s in zip(ctx.dyn_ids, ctx.dyn_scores) if j not in same]
        assert not s_other or min(s_same) > max(s_other)


def test_pose_recipe_ranges():
    for cfg in (C1_TINY, C3_14B, C5_FP8):
        p = gen.poses(cfg, n_blocks=200)
        assert p.shape == (200, 17, 2)
        assert p.min() >= 0 and p.max() <= 1
