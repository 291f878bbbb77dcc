"""Pins of the oracle's greedy acceptance and re-root map: a hand-derived
worked example, brute force over every labelled tree of up to six nodes
against a closed (non-iterative) statement of the rule, special cases and the
generator's planted path lengths.

Acceptance follows the SwiftSpec review page, "What carries the argument"
(the tree re-roots at the last verified token) and "Core claim" (verified
tokens join the prefix); greedy matching against the target's argmax is the
reading used throughout this library.
"""
import itertools
import os

import numpy as np
import pytest

import oracle
from workloads import synth


def _read_accept_golden(path):
    out = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            ex, plant, m, path_, toks, new_pos, r, new_parent = [s.strip() for s in line.split("|")]
            out.append({
                "plant": [tuple(int(x) for x in p.split(":")) for p in plant.split()],
                "m": int(m), "path": [int(x) for x in path_.split()],
                "out_tokens": [int(x) for x in toks.split()],
                "new_pos": [int(x) for x in new_pos.split()], "r": int(r),
                "new_parent": [int(x) for x in new_parent.split()],
            })
    return out


GOLD_PARENT = [-1, 0, 0, 1, 1, 2, 3, 6]
GOLD_TOKEN = [9, 5, 6, 7, 7, 8, 3, 2]


def check_accept_worked_examples(golden_dir):
    for ex in _read_accept_golden(os.path.join(golden_dir, "accept_worked_example.txt")):
        logits = np.zeros((8, 100), dtype=np.float32)
        for row, tok in ex["plant"]:
            logits[row, tok] = 1.0
        res = oracle.tree_accept(logits, GOLD_TOKEN, GOLD_PARENT, 10)
        m = ex["m"]
        assert res["m"] == m
        assert list(res["path"][:m + 1]) == ex["path"]
        assert all(x == -1 for x in res["path"][m + 1:])
        assert list(res["out_tokens"][:m + 1]) == ex["out_tokens"]
        assert all(x == -1 for x in res["out_tokens"][m + 1:])
        assert list(res["new_pos"]) == ex["new_pos"]
        assert res["n_survivors"] == ex["r"]
        assert list(res["new_parent"][:ex["r"]]) == ex["new_parent"]
        assert all(x == -1 for x in res["new_parent"][ex["r"]:])


def test_accept_worked_examples(golden_dir):
    check_accept_worked_examples(golden_dir)


def _all_trees(n):
    # every parent array with parent[i] in [0, i) for i >= 1: (n-1)! labelled trees
    for choice in itertools.product(*[range(i) for i in range(1, n)]):
        yield [-1] + list(choice)


def _closed_form_accepted_node(parent, token, am):
    """The deepest node v such that every edge (u -> w) on the root-to-v path
    satisfies: w is the lowest-indexed child of u whose token is am[u].
    Stated without iterating the walk: each node's eligibility is checked
    from its own path, which is read off networkx."""
    nx = pytest.importorskip("networkx")
    n = len(parent)
    g = nx.DiGraph()
    g.add_nodes_from(range(n))
    g.add_edges_from((parent[i], i) for i in range(1, n))
    best = 0
    best_depth = 0
    for v in range(n):
        path = nx.shortest_path(g, 0, v)
        ok = True
        for u, w in zip(path[:-1], path[1:]):
            matching = [c for c in g.successors(u) if token[c] == am[u]]
            if not matching or min(matching) != w:
                ok = False
                break
        if ok and len(path) - 1 > best_depth:
            best, best_depth = v, len(path) - 1
    return best, (nx.shortest_path(g, 0, best) if best else [0])


def check_bruteforce_small_trees(max_n=6, alphabet=3, trials=3, seed=0):
    rng = np.random.default_rng(seed)
    count = 0
    for n in range(1, max_n + 1):
        for parent in _all_trees(n):
            for _ in range(trials):
                token = rng.integers(0, alphabet, size=n).tolist()
                am = rng.integers(0, alphabet, size=n).tolist()
                path = oracle.greedy_walk(am, token, parent)
                v, ref_path = _closed_form_accepted_node(parent, token, am)
                assert path[-1] == v and path == ref_path, (parent, token, am)
                count += 1
    return count


def test_bruteforce_all_labelled_trees_up_to_six_nodes():
    assert check_bruteforce_small_trees() > 400


def test_special_cases():
    # no root child matches -> m = 0, one emitted token (the bonus)
    parent = [-1, 0, 0]
    token = [1, 2, 3]
    logits = np.zeros((3, 10), dtype=np.float32)
    logits[0, 4] = 1
    res = oracle.tree_accept(logits, token, parent, 5)
    assert res["m"] == 0 and list(res["out_tokens"][:1]) == [4]
    assert list(res["new_pos"]) == [5, 6, 7] and res["n_survivors"] == 2
    # a fully planted chain -> m = depth
    n = 9
    parent = synth.chain_tree(n)
    token = np.arange(100, 100 + n)
    logits = np.zeros((n, 200), dtype=np.float32)
    for i in range(n - 1):
        logits[i, token[i + 1]] = 3.0
    logits[n - 1, 7] = 3.0
    res = oracle.tree_accept(logits, token, parent, 0)
    assert res["m"] == n - 1
    assert list(res["out_tokens"]) == list(token[1:]) + [7, -1]
    assert list(res["new_pos"]) == list(range(n)) and res["n_survivors"] == 0
    # single node tree
    res = oracle.tree_accept(np.zeros((1, 3), np.float32), [0], [-1], 11)
    assert res["m"] == 0 and list(res["new_pos"]) == [11] and list(res["out_tokens"]) == [0, -1]


def test_argmax_ties_and_nan_follow_first_occurrence():
    row = np.array([[0.5, 2.0, 2.0, -1.0], [-0.0, 0.0, -1.0, -2.0],
                    [1.0, np.nan, 3.0, np.nan], [-np.inf, -np.inf, -np.inf, -np.inf]],
                    dtype=np.float32)
    assert list(oracle.target_argmax(row)) == [1, 0, 1, 0]


@pytest.mark.parametrize("seed", range(6))
def test_planted_path_length_is_recovered(seed):
    # the generator plants a path of length m (it draws a node at depth m and
    # sets each row's maximum to the next token); the oracle must find it
    m = seed % 9
    w = synth.make_workload("full_step", seed=seed, planted_m=m, layers=1)
    res = oracle.tree_accept(w.logits, w.token, w.parent, w.prefix)
    assert res["m"] == m
    assert list(res["path"][:m + 1]) == list(w.planted_path)


@pytest.mark.parametrize("m", range(4))
def test_tiny_planted_variants(m):
    w = synth.make_workload("tiny", seed=m, planted_m=m)
    res = oracle.tree_accept(w.logits, w.token, w.parent, w.prefix)
    assert res["m"] == m and list(res["path"][:m + 1]) == list(w.planted_path)
