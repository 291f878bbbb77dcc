"""CPU oracle for the draft side of tree speculation -- TEST INFRASTRUCTURE.

Only the tests, the package's smoke check and the benchmark's CPU-baseline
leg may import this module.  The product path (the CUDA library and its
Python binding) never calls it, and it shares no code with that path.

What it computes follows the SwiftSpec review page (pith.science, paper
2506.11309):

* "Assumptions & free parameters" (the domain assumption on maximum-likelihood
  tree expansion, Algorithm 1 and Section 3.1) and "Core claim": the draft
  grows its tree by maximum-likelihood expansion, scoring a path by the sum of
  the log-softmax probabilities along it and adding the best-scoring leaves;
  the expansion width is w (8 on the page).
* "What carries the argument": after each verification the draft tree
  re-roots at the last verified token and the cache keeps only the
  still-useful subtree, contiguously after the verified prefix.

The page describes these steps in prose only.  The readings taken where it
is silent:

  F1  One expansion scores every child candidate (f, v) of the frontier nodes
      (the nodes whose draft logits are given) as
          score(f, v) = cum[frontier[f]] + log_softmax(z_f)[v]
      and adds the w highest-scoring candidates as new leaves.  Equal scores
      go to the lower frontier position, then to the lower token id.
  F2  The new leaves are appended in that order (best first); a new leaf's
      cumulative log-probability is its score.
  F3  Draft-side re-rooting after a verification with accepted path
      a_0..a_m and bonus token t: the new root is the child b of a_m whose
      token is t (the lowest node index if several), and the survivors are b
      and its descendants in ascending node order.  If a_m has no such
      child nothing survives.  The path moves into the prefix at rows
      [P, P + m + 1), the survivors follow contiguously, and cumulative
      log-probabilities are re-based so that the new root has 0.

Everything is plain fp64 NumPy, the steps in order.  Pinned by
tests/test_oracle_expand.py.
"""
from __future__ import annotations

from typing import Sequence

import numpy as np

from .tree_verify import ancestors_inclusive, check_tree


def log_softmax(z) -> np.ndarray:
    """Row-wise log-softmax in fp64: z - max - log(sum(exp(z - max)))."""
    z = np.asarray(z, dtype=np.float64)
    mx = z.max(axis=-1, keepdims=True)
    return z - mx - np.log(np.exp(z - mx).sum(axis=-1, keepdims=True))


def candidate_scores(logits, frontier: Sequence[int], cum: Sequence[float]) -> np.ndarray:
    """score[f, v] = cum[frontier[f]] + log_softmax(logits[f])[v] (reading F1)."""
    lp = log_softmax(logits)
    base = np.array([float(cum[int(u)]) for u in frontier], dtype=np.float64)
    return base[:, None] + lp


def ml_expand(logits, frontier: Sequence[int], cum: Sequence[float], w: int):
    """One maximum-likelihood expansion (readings F1, F2).

    Returns (parent, token, score) of the w new leaves, best first; parent
    holds tree node indices (frontier[f])."""
    scores = candidate_scores(logits, frontier, cum)
    nf, vocab = scores.shape
    if not 1 <= w <= nf * vocab:
        raise ValueError("w out of range")
    flat = scores.ravel()
    # the sort key: score descending, then frontier position, then token id;
    # the flat index f * V + v orders the last two
    order = np.lexsort((np.arange(flat.size), -flat))[:w]
    f, v = np.divmod(order, vocab)
    parent = np.array([int(frontier[int(i)]) for i in f], dtype=np.int32)
    return parent, v.astype(np.int32), flat[order]


def draft_reroot(parent: Sequence[int], token: Sequence[int], cum: Sequence[float],
                 path: Sequence[int], bonus: int, prefix_len: int) -> dict:
    """Draft-side re-root map (reading F3).

    Returns new_pos [N] (old node -> cache row, or -1), and for the r
    survivors (new node k < r) new_parent [N] (-1 for the new root and past
    r), new_token [N] (-1 past r), new_cum [N] (0 past r)."""
    check_tree(parent)
    n = len(parent)
    path = [int(a) for a in path]
    m = len(path) - 1
    am_ = path[-1]
    b = None
    for c in range(n):
        if int(parent[c]) == am_ and int(token[c]) == int(bonus):
            b = c
            break
    surv = [] if b is None else [i for i in range(n) if b in ancestors_inclusive(parent, i)]
    keep = path + surv
    new_pos = np.full(n, -1, dtype=np.int32)
    for idx, node in enumerate(keep):
        new_pos[node] = prefix_len + idx
    rank = {node: k for k, node in enumerate(surv)}
    new_parent = np.full(n, -1, dtype=np.int32)
    new_token = np.full(n, -1, dtype=np.int32)
    new_cum = np.zeros(n, dtype=np.float64)
    for k, node in enumerate(surv):
        new_parent[k] = -1 if node == b else rank[int(parent[node])]
        new_token[k] = int(token[node])
        new_cum[k] = float(cum[node]) - float(cum[b])
    return {"new_pos": new_pos, "new_parent": new_parent, "new_token": new_token,
            "new_cum": new_cum, "n_survivors": len(surv), "new_root": -1 if b is None else b}
