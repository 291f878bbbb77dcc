"""Pins of the oracle's tree-masked attention against things other than itself:
a hand-derived worked example, library attention on the special cases that
reduce to it (a chain is causal attention, one node is decode attention, any
node is plain attention over its own path) and the masking invariant.

Tree-masked attention follows the SwiftSpec review page, "What carries the
argument" (prefix then tree tokens in the cache; mask attention on the target).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import synth

F = torch.nn.functional


def _read_attention_golden(path):
    rows = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            ex, node, head, o0, o1 = line.split()
            rows[(ex, int(node), int(head))] = (float(o0), float(o1))
    return rows


def _example_a():
    w = [1, 2, 1, 4, 2, 8]
    v = [(1, 0), (0, 1), (2, 2), (4, 0), (0, 4), (8, 8)]
    k = np.array([[[math.log(x), 0.0] for x in w]])
    vv = np.array([v], dtype=np.float64)
    q = np.array([[[math.sqrt(2.0), 0.0]] for _ in range(4)])
    return q, k, vv, 2, [-1, 0, 0, 1]


def _example_b():
    c = [1, 2, 1, 2]
    q = np.array([[[math.sqrt(2.0) * ch, 0.0] for ch in c]])
    k = np.array([[[math.log(1), 0.0], [math.log(3), 0.0]],
                  [[math.log(3), 0.0], [math.log(1), 0.0]]])
    v = np.array([[[1, 0], [0, 1]], [[2, 2], [6, -2]]], dtype=np.float64)
    return q, k, v, 1, [-1]


def check_worked_examples(golden_dir):
    gold = _read_attention_golden(os.path.join(golden_dir, "attention_worked_example.txt"))
    for ex, make in (("A", _example_a), ("B", _example_b)):
        q, k, v, P, parent = make()
        out = oracle.tree_attention(q, k, v, P, parent)
        for (e, node, head), want in gold.items():
            if e == ex:
                np.testing.assert_allclose(out[node, head], want, rtol=0, atol=1e-12)


def test_worked_examples(golden_dir):
    check_worked_examples(golden_dir)


def _causal_reference(q_seq, k_seq, v_seq, scale):
    # q_seq, k_seq, v_seq: [H][S][d] fp64; torch's own causal mask
    return F.scaled_dot_product_attention(torch.from_numpy(q_seq), torch.from_numpy(k_seq),
                                          torch.from_numpy(v_seq), is_causal=True,
                                          scale=scale).numpy()


def check_chain_is_causal(seed=0, P=37, N=9, hq=4, hkv=2, d=16):
    rng = np.random.default_rng(seed)
    G = hq // hkv
    q = rng.standard_normal((N, hq, d))
    k = rng.standard_normal((hkv, P + N, d))
    v = rng.standard_normal((hkv, P + N, d))
    out = oracle.tree_attention(q, k, v, P, synth.chain_tree(N))
    scale = 1.0 / math.sqrt(d)
    for h in range(hq):
        g = h // G
        # the whole sequence (prefix positions get arbitrary queries) under a causal mask
        q_seq = np.concatenate([rng.standard_normal((P, d)), q[:, h, :]], axis=0)[None]
        ref = _causal_reference(q_seq, k[g][None], v[g][None], scale)[0, P:]
        np.testing.assert_allclose(out[:, h, :], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed,P,N", [(0, 37, 9), (1, 0, 5), (2, 128, 1), (3, 5, 40)])
def test_chain_tree_equals_causal_attention(seed, P, N):
    check_chain_is_causal(seed, P, N)


def check_single_node_is_decode(seed=0, P=100, hq=8, hkv=2, d=32):
    rng = np.random.default_rng(seed)
    G = hq // hkv
    q = rng.standard_normal((1, hq, d))
    k = rng.standard_normal((hkv, P + 3, d))  # capacity above P + N: rows past P+N unused
    v = rng.standard_normal((hkv, P + 3, d))
    out = oracle.tree_attention(q, k, v, P, [-1])
    qt = torch.from_numpy(q[0][:, None, :])                     # [Hq][1][d]
    kt = torch.from_numpy(np.repeat(k[:, :P + 1], G, axis=0))   # [Hq][P+1][d]
    vt = torch.from_numpy(np.repeat(v[:, :P + 1], G, axis=0))
    ref = F.scaled_dot_product_attention(qt, kt, vt).numpy()[:, 0, :]
    np.testing.assert_allclose(out[0], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed,P", [(0, 100), (1, 0), (2, 1), (3, 513)])
def test_single_node_equals_decode_attention(seed, P):
    check_single_node_is_decode(seed, P)


def check_node_is_attention_over_own_path(seed=0, P=20, N=30, hq=6, hkv=3, d=8):
    nx = pytest.importorskip("networkx")
    rng = np.random.default_rng(seed)
    G = hq // hkv
    parent = synth.random_parent_tree(rng, N, max_depth=6)
    q = rng.standard_normal((N, hq, d))
    k = rng.standard_normal((hkv, P + N, d))
    v = rng.standard_normal((hkv, P + N, d))
    scale = 0.3
    out = oracle.tree_attention(q, k, v, P, parent, scale=scale)
    tree = nx.DiGraph()
    tree.add_nodes_from(range(N))
    tree.add_edges_from((int(p), i) for i, p in enumerate(parent) if p >= 0)
    for i in range(N):
        path = nx.shortest_path(tree, 0, i)  # the root-to-node path
        rows = list(range(P)) + [P + j for j in path]
        for h in range(hq):
            g = h // G
            ref = F.scaled_dot_product_attention(
                torch.from_numpy(q[i, h][None, None]), torch.from_numpy(k[g, rows][None]),
                torch.from_numpy(v[g, rows][None]), scale=scale).numpy()[0, 0]
            np.testing.assert_allclose(out[i, h], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_node_equals_attention_over_its_path(seed):
    check_node_is_attention_over_own_path(seed)


def check_masked_rows_have_no_influence(seed=0, P=16, N=24, hq=4, hkv=1, d=8):
    rng = np.random.default_rng(seed)
    parent = synth.random_parent_tree(rng, N, max_depth=5)
    q = rng.standard_normal((N, hq, d))
    k = rng.standard_normal((hkv, P + N + 4, d))
    v = rng.standard_normal((hkv, P + N + 4, d))
    base = oracle.tree_attention(q, k, v, P, parent)
    path = [N - 1]
    while parent[path[-1]] >= 0:
        path.append(int(parent[path[-1]]))
    anc = set(path)
    k2, v2 = k.copy(), v.copy()
    for j in range(N):
        if j not in anc:
            k2[:, P + j] *= 1e3
            v2[:, P + j] *= -1e3
    k2[:, P + N:] = 7e5  # rows past the tree are never read
    v2[:, P + N:] = -7e5
    pert = oracle.tree_attention(q, k2, v2, P, parent)
    assert np.array_equal(pert[N - 1], base[N - 1])


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_masked_rows_have_no_influence(seed):
    check_masked_rows_have_no_influence(seed)


def test_bitmask_matches_boolean_mask():
    rng = np.random.default_rng(5)
    for n in (1, 2, 31, 32, 33, 64, 100, 128):
        parent = synth.random_parent_tree(rng, n, max_depth=16)
        bits = oracle.ancestor_bitmask(parent)
        mask = oracle.ancestor_mask(parent)
        assert bits.shape == (n, (n + 31) // 32)
        for i in range(n):
            for j in range(n):
                assert bool((int(bits[i, j // 32]) >> (j % 32)) & 1) == mask[i, j]


def test_mask_of_known_trees():
    # complete binary tree of 7: node 6 sees 6, 2, 0; node 3 sees 3, 1, 0
    m = oracle.ancestor_mask(synth.complete_binary_tree(7))
    assert set(np.flatnonzero(m[6])) == {0, 2, 6}
    assert set(np.flatnonzero(m[3])) == {0, 1, 3}
    assert set(np.flatnonzero(m[0])) == {0}
    # forest: two roots
    m = oracle.ancestor_mask([-1, 0, -1, 2])
    assert set(np.flatnonzero(m[3])) == {2, 3}


def test_rejects_invalid_trees():
    for bad in ([0], [-1, 1], [-1, 2, 0], [-1, -2]):
        with pytest.raises(ValueError):
            oracle.check_tree(bad)
