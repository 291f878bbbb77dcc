"""CPU oracle for tree-masked speculative verification -- TEST INFRASTRUCTURE.

Only the tests, the package's smoke check and the benchmark's CPU-baseline
leg may import this module.  The product path (the CUDA library and its
Python binding) never calls it, and it shares no code with that path.

What it computes follows the SwiftSpec review page (pith.science, paper
2506.11309):

* "What carries the argument" and "Core claim": the KV cache holds the
  verified tokens contiguously as a prefix with the draft-tree tokens right
  after it; after each verification the tree re-roots at the last verified
  token and the cache is reorganised to keep the still-useful subtree.
* "What carries the argument" and "Referee Report" (summary, Section 3.3): the
  target verifies the tree with a mask attention kernel, i.e. each tree token
  attends the prefix and the tokens on its own root-to-node path.
* "Referee Report", major comment 3 (Section 3.2): the target-side cache
  management is not described by the paper; the readings used here are
  listed with each function.

Everything is plain fp64 NumPy with the algorithm's steps in order: no
blocking, no split-KV, no online softmax.  A library matmul serves as the dot
product step.  Every function is pinned by the tests in tests/test_oracle_*.py
against closed forms, library routines, brute force and invariants.
"""
from __future__ import annotations

import math
from typing import Sequence

import numpy as np


# ---------------------------------------------------------------------------
# the draft tree and its ancestor mask
# ---------------------------------------------------------------------------

def check_tree(parent: Sequence[int]) -> None:
    """A draft tree (or forest) in node order: parent[i] = -1 marks a root,
    otherwise 0 <= parent[i] < i.  Node 0 is always a root (the last verified
    token, review page "What carries the argument")."""
    for i, p in enumerate(parent):
        if not (-1 <= int(p) < i):
            raise ValueError(f"parent[{i}] = {p} is not in [-1, {i})")


def ancestors_inclusive(parent: Sequence[int], i: int) -> list[int]:
    """anc*(i): node i followed by its ancestors, walking parent pointers up
    to a root.  A node attends itself (a chain of nodes is then exactly causal
    attention)."""
    out = [i]
    while int(parent[out[-1]]) >= 0:
        out.append(int(parent[out[-1]]))
    return out


def ancestor_mask(parent: Sequence[int]) -> np.ndarray:
    """Explicit tree mask: mask[i, j] is True when tree node i may attend tree
    node j, i.e. j is i or an ancestor of i."""
    check_tree(parent)
    n = len(parent)
    mask = np.zeros((n, n), dtype=bool)
    for i in range(n):
        mask[i, ancestors_inclusive(parent, i)] = True
    return mask


def ancestor_bitmask(parent: Sequence[int]) -> np.ndarray:
    """The same mask packed as ceil(N/32) little-endian uint32 words per node:
    bit (j mod 32) of word j // 32 of row i is mask[i, j]."""
    mask = ancestor_mask(parent)
    n = len(parent)
    words = (n + 31) // 32
    out = np.zeros((n, words), dtype=np.uint32)
    for i in range(n):
        for j in range(n):
            if mask[i, j]:
                out[i, j // 32] |= np.uint32(1 << (j % 32))
    return out


# ---------------------------------------------------------------------------
# tree-masked GQA attention (one layer)
# ---------------------------------------------------------------------------

def kv_head_of(h: int, hq: int, hkv: int) -> int:
    """Grouped-query attention: the G = hq / hkv consecutive query heads
    h = g*G .. g*G+G-1 share KV head g."""
    return h // (hq // hkv)


def default_scale(d: int) -> float:
    """Softmax scale 1/sqrt(d) (scaled dot-product attention)."""
    return 1.0 / math.sqrt(d)


def tree_attention(q, k_cache, v_cache, prefix_len: int, parent: Sequence[int],
                   scale: float | None = None, nodes: Sequence[int] | None = None) -> np.ndarray:
    """Tree-masked attention of one layer, in fp64.

    q        [N][Hq][d]   query of each tree node and head
    k_cache  [Hkv][cap][d] keys: rows [0, P) are the verified prefix, rows
    v_cache  [Hkv][cap][d] P + j hold tree node j (review page, "What carries
                           the argument": prefix first, tree tokens right after)
    Returns  [N][Hq][d]   o[i, h] = softmax(q[i,h] . K_sel^T * scale) . V_sel,
             where K_sel/V_sel are the rows [0, P) plus {P + j : j in anc*(i)}
             of KV head h // G.
    The stored values (already rounded to their storage type) are upcast to
    fp64; nothing is rounded afterwards.  With `nodes` given, only those tree
    nodes are computed and the result is [len(nodes)][Hq][d] in that order
    (a sample of a large case).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k_cache, dtype=np.float64)
    v = np.asarray(v_cache, dtype=np.float64)
    n, hq, d = q.shape
    hkv = k.shape[0]
    if hq % hkv:
        raise ValueError("hq must be a multiple of hkv")
    check_tree(parent)
    if prefix_len + n > k.shape[1]:
        raise ValueError("cache capacity below prefix + tree")
    if scale is None:
        scale = default_scale(d)
    mask = ancestor_mask(parent)
    todo = list(range(n)) if nodes is None else [int(x) for x in nodes]
    out = np.empty((len(todo), hq, d), dtype=np.float64)
    for o, i in enumerate(todo):
        rows = list(range(prefix_len)) + [prefix_len + j for j in range(n) if mask[i, j]]
        sel = {}
        for h in range(hq):
            g = kv_head_of(h, hq, hkv)
            if g not in sel:
                sel[g] = (k[g, rows, :], v[g, rows, :])
            keys, vals = sel[g]
            s = (keys @ q[i, h]) * scale
            w = np.exp(s - s.max())
            out[o, h] = (w @ vals) / w.sum()
    return out


# ---------------------------------------------------------------------------
# greedy acceptance
# ---------------------------------------------------------------------------

def target_argmax(logits) -> np.ndarray:
    """am[i] = argmax over the vocabulary of the target's logits for node i,
    compared in the logits' own precision; ties go to the lowest token id and
    a NaN counts as the maximum (NumPy's argmax)."""
    return np.argmax(np.asarray(logits), axis=1).astype(np.int32)


def greedy_walk(am: Sequence[int], token: Sequence[int], parent: Sequence[int]) -> list[int]:
    """Greedy verification of the draft tree against the target's argmax.

    Starting at the root (node 0), step to the child c of the current node u
    whose draft token equals am[u]; when several children carry that token
    the lowest node index is taken.  Stop when no child matches.  Returns the
    accepted path a_0 = 0, a_1, ..., a_m.
    """
    check_tree(parent)
    n = len(parent)
    path = [0]
    while True:
        u = path[-1]
        nxt = None
        for c in range(n):
            if int(parent[c]) == u and int(token[c]) == int(am[u]):
                nxt = c
                break
        if nxt is None:
            return path
        path.append(nxt)


def accepted_tokens(path: Sequence[int], am: Sequence[int], token: Sequence[int]) -> list[int]:
    """Tokens emitted by one verification: the accepted draft tokens
    token[a_1..a_m] followed by the target's own next token am[a_m] (the
    bonus token).  The root's token was emitted by the previous step."""
    return [int(token[a]) for a in path[1:]] + [int(am[path[-1]])]


# ---------------------------------------------------------------------------
# re-rooting and KV compaction
# ---------------------------------------------------------------------------

def strict_descendants(parent: Sequence[int], u: int) -> list[int]:
    """Nodes strictly below u, in ascending node order."""
    return [i for i in range(len(parent)) if i != u and u in ancestors_inclusive(parent, i)]


def reroot(parent: Sequence[int], path: Sequence[int], prefix_len: int):
    """Cache layout after a verification (review page, "What carries the
    argument" and "Core claim"; the target side is undescribed per "Referee
    Report", major comment 3, so the survivor rule is a reading).

    keep = the accepted path a_0..a_m followed by the strict descendants of
    a_m in ascending node order.  The path moves into the prefix at rows
    [P, P + m + 1); the survivors follow it contiguously.

    Returns (new_pos, new_parent, r):
      new_pos[i]    (old node index) P + rank of i in keep, or -1 if dropped
      new_parent[k] (new node index k < r) rank(parent) - (m + 1), or -1 when
                    the parent is a_m (now the last prefix row); -1 for k >= r
      r             number of surviving tree nodes
    """
    n = len(parent)
    path = [int(a) for a in path]
    m = len(path) - 1
    desc = strict_descendants(parent, path[-1])
    keep = path + desc
    rank = {node: idx for idx, node in enumerate(keep)}
    new_pos = np.full(n, -1, dtype=np.int32)
    for node, idx in rank.items():
        new_pos[node] = prefix_len + idx
    new_parent = np.full(n, -1, dtype=np.int32)
    for k, node in enumerate(desc):
        p = int(parent[node])
        new_parent[k] = -1 if p == path[-1] else rank[p] - (m + 1)
    return new_pos, new_parent, len(desc)


def kv_compact(cache, prefix_len: int, new_pos: Sequence[int]) -> np.ndarray:
    """Out-of-place compaction of a cache [..., cap, d]: the row of tree node
    i (row P + i) is copied to row new_pos[i] for every kept node; every other
    row keeps its old contents.  Works on any dtype bit for bit."""
    old = np.asarray(cache)
    new = old.copy()
    for i, pos in enumerate(new_pos):
        if int(pos) >= 0:
            new[..., int(pos), :] = old[..., prefix_len + i, :]
    return new


# ---------------------------------------------------------------------------
# the results of one verification, laid out like the library's outputs
# ---------------------------------------------------------------------------

def tree_accept(logits, token: Sequence[int], parent: Sequence[int], prefix_len: int) -> dict:
    """argmax + greedy walk + re-root map, padded to fixed sizes:
    path [N] (-1 after a_m), out_tokens [N+1] (-1 after the bonus token)."""
    n = len(parent)
    am = target_argmax(logits)
    path = greedy_walk(am, token, parent)
    toks = accepted_tokens(path, am, token)
    new_pos, new_parent, r = reroot(parent, path, prefix_len)
    path_out = np.full(n, -1, dtype=np.int32)
    path_out[:len(path)] = path
    tok_out = np.full(n + 1, -1, dtype=np.int32)
    tok_out[:len(toks)] = toks
    return {"am": am, "m": len(path) - 1, "path": path_out, "out_tokens": tok_out,
            "new_pos": new_pos, "new_parent": new_parent, "n_survivors": r}
