"""Seeded synthetic inputs for tree-masked verification.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark. It only *draws* inputs (draft trees, draft token ids, Q/K/V values,
target logits); it holds none of the verification arithmetic (no ancestor
mask, no attention, no acceptance walk, no compaction). Tree bookkeeping here
(node depths and fan-out counts) exists only to respect the shape limits of
each workload while drawing parents.

Workloads stand in for the SwiftSpec paper's model families and datasets,
which are not available here (SwiftSpec review page, "Referee Report",
Section 5.1 and Section 5.2): GQA shapes of Llama-3-8B, Llama-3-70B and
Qwen2-72B with N(0,1) activations, and draft trees of width 8 built by
expansions (review page, "Assumptions & free parameters": bs = 8, w = 8).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch


# --------------------------------------------------------------------------
# draft trees: parent[0] = -1 (the root, the last verified token), and
# -1 <= parent[i] < i for i > 0 (parents precede children in node order)
# --------------------------------------------------------------------------

def chain_tree(n: int) -> np.ndarray:
    """A single path 0 -> 1 -> ... -> n-1."""
    return np.arange(-1, n - 1, dtype=np.int32)


def complete_binary_tree(n: int) -> np.ndarray:
    """Heap-ordered complete binary tree: parent[i] = (i - 1) // 2."""
    p = (np.arange(n, dtype=np.int64) - 1) // 2
    p[0] = -1
    return p.astype(np.int32)


def uniform_parent_tree(rng: np.random.Generator, n: int, max_depth: int = 8,
                        max_fanout: int = 8) -> np.ndarray:
    """Each node's parent is uniform among the earlier nodes that can still
    take a child: the child's depth stays <= max_depth and the parent's
    fan-out stays <= max_fanout."""
    parent = np.full(n, -1, dtype=np.int32)
    depth = np.zeros(n, dtype=np.int64)
    fan = np.zeros(n, dtype=np.int64)
    for i in range(1, n):
        cand = [j for j in range(i) if depth[j] < max_depth and fan[j] < max_fanout]
        j = int(cand[rng.integers(len(cand))])
        parent[i] = j
        depth[i] = depth[j] + 1
        fan[j] += 1
    return parent


def random_parent_tree(rng: np.random.Generator, n: int, max_depth: int = 16) -> np.ndarray:
    """Parent uniform among earlier nodes whose depth is < max_depth."""
    return uniform_parent_tree(rng, n, max_depth=max_depth, max_fanout=n)


def ml_expansion_tree(rng: np.random.Generator, n: int = 64, width: int = 8,
                      expansions: int = 8, mu: float = -1.0, sigma: float = 0.5,
                      deep: bool = False) -> np.ndarray:
    """A tree grown by `expansions` rounds of `width` new nodes (the last
    round is cut so that the tree holds exactly n nodes with its root).

    Each new node draws its parent among the nodes that existed before the
    round, with probability proportional to exp(c_j), where c_j is a
    synthetic cumulative log-probability: c_root = 0 and
    c_child = c_parent + e with e ~ N(mu, sigma).  With deep=True the first
    node of round k is attached to a node of depth k-1, so that the tree
    reaches depth >= expansions (used for the full verify step, where the
    accepted path length is planted up to 8).
    """
    parent = [-1]
    c = [0.0]
    depth = [0]
    for k in range(1, expansions + 1):
        existing = len(parent)
        if existing >= n:
            break
        w = np.exp(np.asarray(c[:existing]) - max(c[:existing]))
        w = w / w.sum()
        for slot in range(width):
            if len(parent) >= n:
                break
            if deep and slot == 0:
                cand = [j for j in range(existing) if depth[j] == k - 1]
                j = int(cand[rng.integers(len(cand))])
            else:
                j = int(rng.choice(existing, p=w))
            parent.append(j)
            c.append(c[j] + float(rng.normal(mu, sigma)))
            depth.append(depth[j] + 1)
    while len(parent) < n:  # only if expansions * width + 1 < n
        j = int(rng.integers(len(parent)))
        parent.append(j)
        depth.append(depth[j] + 1)
    return np.asarray(parent, dtype=np.int32)


def node_depths(parent: np.ndarray) -> np.ndarray:
    """Depth of each node (root depth 0); parents precede children."""
    d = np.zeros(len(parent), dtype=np.int64)
    for i in range(1, len(parent)):
        d[i] = 0 if parent[i] < 0 else d[parent[i]] + 1
    return d


def draft_tokens(rng: np.random.Generator, parent: np.ndarray, vocab: int,
                 distinct_siblings: bool = True) -> np.ndarray:
    """Draft token ids uniform in [0, vocab).  With distinct_siblings, two
    children of one node never carry the same token (a real top-w draft never
    proposes a token twice under one parent)."""
    n = len(parent)
    tok = rng.integers(0, vocab, size=n).astype(np.int32)
    if distinct_siblings:
        seen: dict[int, set] = {}
        for i in range(1, n):
            s = seen.setdefault(int(parent[i]), set())
            while int(tok[i]) in s:
                tok[i] = rng.integers(0, vocab)
            s.add(int(tok[i]))
    return tok


# --------------------------------------------------------------------------
# values
# --------------------------------------------------------------------------

def normal(rng: np.random.Generator, shape, dtype: str) -> torch.Tensor:
    """N(0,1) draws stored in `dtype` ("f32" or "bf16"; bf16 is the
    round-to-nearest-even rounding of an fp32 draw).  Returned on the CPU."""
    x = torch.from_numpy(rng.standard_normal(size=shape, dtype=np.float32))
    if dtype == "bf16":
        return x.to(torch.bfloat16)
    if dtype == "f32":
        return x
    raise ValueError(dtype)


def planted_logits(rng: np.random.Generator, parent: np.ndarray, token: np.ndarray,
                   vocab: int, m: int) -> tuple[np.ndarray, np.ndarray]:
    """Target logits ~N(0,1) over `vocab`, with a planted maximum so that a
    greedy walk from the root accepts exactly m draft tokens.

    A node v of depth m is drawn; along the root->v path each node's row gets
    its child's token as a clear maximum, and v's row gets as maximum a token
    that none of v's children carries.  Sibling tokens must be distinct (see
    draft_tokens).  Returns (logits float32 [N][vocab], planted path)."""
    n = len(parent)
    depth = node_depths(parent)
    cand = np.flatnonzero(depth == m)
    if len(cand) == 0:
        raise ValueError(f"tree has no node at depth {m}")
    v = int(cand[rng.integers(len(cand))])
    path = [v]
    while path[-1] != 0:
        path.append(int(parent[path[-1]]))
    path = path[::-1]
    logits = rng.standard_normal(size=(n, vocab), dtype=np.float32)
    for a, b in zip(path[:-1], path[1:]):
        logits[a, int(token[b])] = logits[a].max() + 1.0
    child_tokens = {int(token[c]) for c in range(n) if parent[c] == v}
    bonus = int(rng.integers(vocab))
    while bonus in child_tokens:
        bonus = int(rng.integers(vocab))
    logits[v, bonus] = logits[v].max() + 1.0
    return logits, np.asarray(path, dtype=np.int32)


# --------------------------------------------------------------------------
# named workloads
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    name: str
    hq: int
    hkv: int
    d: int
    dtype: str             # "f32" or "bf16"
    prefix: int            # P
    parent: np.ndarray     # int32 [N]
    layers: int            # L
    cap: int               # cache rows per (layer, KV head) >= P + N
    vocab: int = 0
    token: Optional[np.ndarray] = None
    logits: Optional[np.ndarray] = None       # float32 [N][V]
    planted_path: Optional[np.ndarray] = None
    seed: int = 0

    @property
    def n(self) -> int:
        return len(self.parent)


def _tree_for(name: str, rng: np.random.Generator, n: int) -> np.ndarray:
    if name == "tiny":
        return complete_binary_tree(n)
    if name == "l3_8b":
        return uniform_parent_tree(rng, n, max_depth=8, max_fanout=8)
    if name == "l3_70b":
        return ml_expansion_tree(rng, n=n, width=8, expansions=8)
    if name == "q2_72b":
        return random_parent_tree(rng, n, max_depth=16)
    if name == "full_step":
        return ml_expansion_tree(rng, n=n, width=8, expansions=8, deep=True)
    raise ValueError(name)


_SHAPES = {
    # name: (hq, hkv, d, dtype, prefix, n, layers, vocab)
    "tiny": (4, 1, 64, "f32", 128, 15, 1, 1000),
    "l3_8b": (32, 8, 128, "bf16", 2048, 64, 1, 128256),
    "l3_70b": (64, 8, 128, "bf16", 8192, 64, 8, 0),
    "q2_72b": (64, 8, 128, "bf16", 4096, 64, 1, 0),
    "full_step": (64, 8, 128, "bf16", 4096, 64, 80, 128256),
}


def make_workload(name: str, seed: int = 0, prefix: Optional[int] = None,
                  n: Optional[int] = None, layers: Optional[int] = None,
                  planted_m: Optional[int] = None, with_logits: Optional[bool] = None,
                  parent: Optional[np.ndarray] = None) -> Workload:
    """Trees, tokens and logits for a named workload.  Q/K/V are drawn
    separately (make_qkv), so that large caches are only made when needed.

    tiny       4/1 heads, d64, fp32, P=128, complete binary tree of 15, V=1000
    l3_8b      32/8 heads, d128, bf16, P=2048, 64 nodes (depth <= 8, fan-out <= 8), V=128256
    l3_70b     64/8 heads, d128, bf16, P=8192, 64 nodes grown by 8 expansions of 8, 8 layers
    q2_72b     64/8 heads, d128, bf16, P in {1K..32K}, N in {8..128}, depth <= 16
    full_step  64/8 heads, d128, bf16, P=4096, 64 nodes (depth >= 8), 80 layers, V=128256,
               argmax planted so that m ~ U{0..8}
    """
    hq, hkv, d, dt, p0, n0, l0, vocab = _SHAPES[name]
    rng = np.random.default_rng(seed)
    P = p0 if prefix is None else prefix
    N = n0 if n is None else n
    L = l0 if layers is None else layers
    par = _tree_for(name, rng, N) if parent is None else np.asarray(parent, np.int32)
    N = len(par)
    w = Workload(name=name, hq=hq, hkv=hkv, d=d, dtype=dt, prefix=P, parent=par,
                 layers=L, cap=P + N, vocab=vocab, seed=seed)
    if with_logits is None:
        with_logits = vocab > 0
    if with_logits and vocab > 0:
        w.token = draft_tokens(rng, par, vocab, distinct_siblings=True)
        if name == "full_step" or planted_m is not None:
            m = int(rng.integers(0, 9)) if planted_m is None else planted_m
            w.logits, w.planted_path = planted_logits(rng, par, w.token, vocab, m)
        else:
            w.logits = rng.standard_normal(size=(N, vocab), dtype=np.float32)
    return w


def make_qkv(w: Workload, layer: Optional[int] = None, seed_offset: int = 1000):
    """Q [N][Hq][d] and the K and V caches [Hkv][cap][d] of one layer
    (layer given) or of all layers stacked [L][Hkv][cap][d] (layer None),
    drawn N(0,1) in the workload's dtype on the CPU.  Each layer has its own
    stream so that one layer can be drawn without the others."""
    layers = range(w.layers) if layer is None else [layer]
    qs, ks, vs = [], [], []
    for l in layers:
        rng = np.random.default_rng([w.seed, seed_offset, l])
        qs.append(normal(rng, (w.n, w.hq, w.d), w.dtype))
        ks.append(normal(rng, (w.hkv, w.cap, w.d), w.dtype))
        vs.append(normal(rng, (w.hkv, w.cap, w.d), w.dtype))
    if layer is not None:
        return qs[0], ks[0], vs[0]
    return torch.stack(qs), torch.stack(ks), torch.stack(vs)


def lm_head_inputs(seed: int, n: int, d_model: int, vocab: int, w_scale: float = 0.02,
                   integer: bool = False):
    """Final hidden states H [n][d_model] and LM-head weights W [vocab][d_model],
    bf16 on the CPU.  H ~ N(0, 1) (a normalised hidden state), W ~ N(0, w_scale^2)
    (an initialised linear layer); with `integer` both hold small integers in
    [-2, 2], whose dot products are exact in float32 and tie often."""
    rng = np.random.default_rng(seed)
    if integer:
        h = rng.integers(-2, 3, size=(n, d_model)).astype(np.float32)
        w = rng.integers(-2, 3, size=(vocab, d_model)).astype(np.float32)
        return torch.from_numpy(h).to(torch.bfloat16), torch.from_numpy(w).to(torch.bfloat16)
    h = normal(rng, (n, d_model), "bf16")
    w = (torch.from_numpy(rng.standard_normal(size=(vocab, d_model), dtype=np.float32)) *
         w_scale).to(torch.bfloat16)
    return h, w
