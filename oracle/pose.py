"""Pose descriptor and pose retrieval for the dynamic sink.

Follows "LiveAnimate" (ai-feeds.com), 方法 / 核心洞察: the dynamic sink holds
history blocks retrieved by pose similarity, so that appearance context
returns when a pose recurs.

Readings of what the page leaves open:
  * descriptor: the 17 (x, y) keypoints, each axis centred by its mean over
    the keypoints, flattened as [x0, y0, x1, y1, ..., x16, y16];
  * similarity: cosine; a zero-norm descriptor scores 0;
  * candidates: history blocks that are neither the static sink, nor in the
    rolling window, nor the current block;
  * top-k under the total order (score descending, block id ascending);
    fewer than k candidates -> all of them; the chosen ids are used in
    ascending id order.
"""
from __future__ import annotations

import numpy as np


def descriptor(kp: np.ndarray) -> np.ndarray:
    """[17, 2] keypoints -> centred, flattened [34] (fp64)."""
    kp = np.asarray(kp, dtype=np.float64).reshape(17, 2)
    c = kp - kp.mean(axis=0, keepdims=True)
    return c.reshape(34)


def cosine_scores(q: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Cosine similarity of descriptor q [34] with each row of table [N, 34]."""
    q = np.asarray(q, dtype=np.float64)
    table = np.asarray(table, dtype=np.float64).reshape(-1, q.shape[0])
    qn = np.sqrt(np.sum(q * q))
    tn = np.sqrt(np.sum(table * table, axis=1))
    dots = table @ q
    out = np.zeros(table.shape[0], dtype=np.float64)
    ok = (tn > 0) & (qn > 0)
    out[ok] = dots[ok] / (tn[ok] * qn)
    return out


def candidates(b: int, window: int, static_sink: int) -> list[int]:
    """History blocks eligible for retrieval when block b is generated."""
    win = set(range(max(0, b - window), b))
    sink = {0} if static_sink else set()
    return [j for j in range(b) if j not in win and j not in sink]


def select_topk(scores: np.ndarray, ids: list[int], k: int):
    """Top-k of (id, score) pairs under (score desc, id asc).

    Returns (chosen ids ascending, their scores in that order, gap) where gap
    is score_k - score_{k+1} in the total order (inf when there is no
    (k+1)-th candidate or no candidate at all)."""
    scores = np.asarray(scores, dtype=np.float64)
    ids_a = np.asarray(ids, dtype=np.int64)
    order = np.lexsort((ids_a, -scores))     # primary: -score, secondary: id
    top = order[:k]
    gap = np.inf
    if len(order) > k and k > 0:
        gap = float(scores[order[k - 1]] - scores[order[k]])
    chosen = sorted(top.tolist(), key=lambda i: ids_a[i])
    return [int(ids_a[i]) for i in chosen], [float(scores[i]) for i in chosen], gap
