"""Router top-k and softmax of the oracle (test infrastructure only).

The pages name the step and its outputs but do not spell it out: in "CURRENT_BUG.md
-- DeepSeek-V4 Blackwell NVFP4", "Test Plan -- Finding the NaN", Phase 1 item 1,
topk_ids and topk_weights "from the router" are the runner's inputs, and
"Architecture: DeepSeek-V4 MegaMoE" fixes 384 experts, top-6.  The plain reading
taken here:

  score[t, e] = fl32(logits[t, e] + bias[e])          (bias optional, selection only)
  topk_ids[t] = the k experts of highest score, in descending score; equal
                scores are ordered by ascending expert index
  topk_weights[t, j] = exp(l_j) / sum_i exp(l_i) over the k selected logits
                (float64 here)

The score comparison decides integers (the ids), so it is taken in float32,
the precision the logits come in.  A shared expert that every token visits is
an optional extra column (its id, weight 1).
"""

from __future__ import annotations

import numpy as np


def router_topk(logits, k: int, bias=None, shared_expert=None):
    """Returns (topk_ids [T, k'] int64, topk_weights [T, k'] float64),
    k' = k (+1 with a shared expert)."""
    lg = np.asarray(logits, dtype=np.float32)
    if lg.ndim != 2:
        raise ValueError("logits must be [T, E]")
    T, E = lg.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    score = lg if bias is None else (lg + np.asarray(bias, dtype=np.float32)[None, :])
    score = score.astype(np.float32)
    # sort each row by descending score, then ascending expert index
    idx = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((idx, -score), axis=-1)
    ids = order[:, :k].astype(np.int64)
    sel = np.take_along_axis(lg, ids, axis=1).astype(np.float64)
    ex = np.exp(sel - sel.max(axis=1, keepdims=True))
    w = ex / ex.sum(axis=1, keepdims=True)
    if shared_expert is not None:
        ids = np.concatenate([ids, np.full((T, 1), int(shared_expert), np.int64)], axis=1)
        w = np.concatenate([w, np.ones((T, 1))], axis=1)
    return ids, w
