"""Pins of the oracle's re-root map and KV compaction: compaction is a
permutation copy that leaves the prefix alone, the kept set is the accepted
path plus the subtree under its last node (read off networkx), and re-rooting
preserves every survivor's attention output (the KV-cache reorganisation
invariant the SwiftSpec review page lists as unproven under "Assumptions &
free parameters"; it is checked here directly).
"""
import numpy as np
import pytest

import oracle
from workloads import synth


def _random_case(seed, N=24, P=11, vocab=5):
    rng = np.random.default_rng(seed)
    parent = synth.random_parent_tree(rng, N, max_depth=7)
    token = rng.integers(0, vocab, size=N)
    logits = rng.standard_normal((N, vocab)).astype(np.float32)
    return rng, parent, token, logits, P


@pytest.mark.parametrize("seed", range(20))
def test_keep_set_is_path_plus_subtree(seed):
    nx = pytest.importorskip("networkx")
    _, parent, token, logits, P = _random_case(seed)
    res = oracle.tree_accept(logits, token, parent, P)
    m = res["m"]
    path = list(res["path"][:m + 1])
    g = nx.DiGraph()
    g.add_nodes_from(range(len(parent)))
    g.add_edges_from((int(parent[i]), i) for i in range(1, len(parent)))
    keep = set(path) | nx.descendants(g, path[-1])
    kept = {i for i, p in enumerate(res["new_pos"]) if p >= 0}
    assert kept == keep
    pos = [int(res["new_pos"][i]) for i in sorted(kept)]
    assert pos == list(range(P, P + len(kept)))           # contiguous, in node order
    assert res["n_survivors"] == len(keep) - (m + 1)
    # the survivors' new parents point at the same nodes as before
    order = sorted(kept)
    surv = order[m + 1:]
    for k, node in enumerate(surv):
        npar = int(res["new_parent"][k])
        if npar == -1:
            assert int(parent[node]) == path[-1]
        else:
            assert surv[npar] == int(parent[node])


@pytest.mark.parametrize("seed", range(10))
def test_compaction_is_a_permutation_copy(seed):
    rng, parent, token, logits, P = _random_case(seed)
    N = len(parent)
    cap = P + N + 3
    cache = rng.standard_normal((2, 3, cap, 4)).astype(np.float32)
    res = oracle.tree_accept(logits, token, parent, P)
    new = oracle.kv_compact(cache, P, res["new_pos"])
    assert np.array_equal(new[..., :P, :], cache[..., :P, :])          # prefix untouched
    assert np.array_equal(new[..., P + N:, :], cache[..., P + N:, :])  # past the tree untouched
    kept = [i for i in range(N) if res["new_pos"][i] >= 0]
    moved = new[..., P:P + len(kept), :]
    want = cache[..., [P + i for i in kept], :]
    assert np.array_equal(moved, want)
    # the multiset of kept rows is preserved
    a = sorted(map(bytes, moved.reshape(-1, 4)))
    b = sorted(map(bytes, want.reshape(-1, 4)))
    assert a == b


def check_reroot_preserves_attention(seed, N=20, P=9, hq=4, hkv=2, d=8):
    rng, parent, token, logits, _ = _random_case(seed, N=N, P=P)
    res = oracle.tree_accept(logits, token, parent, P)
    m, r = res["m"], res["n_survivors"]
    q = rng.standard_normal((N, hq, d))
    k = rng.standard_normal((hkv, P + N, d))
    v = rng.standard_normal((hkv, P + N, d))
    before = oracle.tree_attention(q, k, v, P, parent)
    k2 = oracle.kv_compact(k, P, res["new_pos"])
    v2 = oracle.kv_compact(v, P, res["new_pos"])
    survivors = [i for i in range(N) if res["new_pos"][i] >= P + m + 1]
    if r == 0:
        return 0
    new_parent = res["new_parent"][:r]
    after = oracle.tree_attention(q[survivors], k2, v2, P + m + 1, new_parent)
    np.testing.assert_allclose(after, before[survivors], rtol=0, atol=1e-12)
    return r


def test_reroot_preserves_survivor_attention():
    total = 0
    for seed in range(40):
        total += check_reroot_preserves_attention(seed)
    assert total > 0  # some cases do keep a subtree


def test_reroot_on_full_step_tree():
    w = synth.make_workload("full_step", seed=3, layers=1)
    res = oracle.tree_accept(w.logits, w.token, w.parent, w.prefix)
    kept = [i for i in range(w.n) if res["new_pos"][i] >= 0]
    assert len(kept) == res["m"] + 1 + res["n_survivors"]
    assert all(res["new_pos"][i] <= w.prefix + i for i in kept)  # rows only move down
