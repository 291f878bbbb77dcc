"""Pins of the draft-side oracle (oracle/tree_expand.py) to facts it does not
compute itself: SciPy's log-softmax, hand-derived worked examples
(tests/golden/expand_worked_example.txt), a brute-force ranking of candidate
paths by their probability (a product of softmax probabilities, no
logarithms), the special case that reduces to an argmax, and the structural
invariants of re-rooting."""
import itertools
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "expand_worked_example.txt")


def _fixture():
    rows = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows[(parts[0], parts[1])] = parts[2:]
    return rows


def _ints(v):
    return [int(x) for x in v]


def _floats(v):
    return [float(x) for x in v]


# ------------------------------------------------------------ log-softmax

def check_log_softmax_matches_scipy(seed):
    sp = pytest.importorskip("scipy.special")
    z = np.random.default_rng(seed).standard_normal((5, 300)) * 4
    assert np.allclose(oracle.log_softmax(z), sp.log_softmax(z, axis=-1), atol=1e-12)
    assert np.allclose(np.exp(oracle.log_softmax(z)).sum(axis=-1), 1.0, atol=1e-12)


def test_log_softmax_matches_scipy():
    for seed in range(3):
        check_log_softmax_matches_scipy(seed)


def test_log_softmax_is_shift_invariant_and_stable():
    z = np.random.default_rng(1).standard_normal((2, 50))
    assert np.allclose(oracle.log_softmax(z), oracle.log_softmax(z + 1000.0), atol=1e-9)


# ------------------------------------------------------------ expansion

def check_worked_expansion():
    fx = _fixture()
    probs = np.array([_floats(fx[("expand", "probs0")]), _floats(fx[("expand", "probs1")])])
    frontier = _ints(fx[("expand", "frontier")])
    cum = {u: c for u, c in zip(frontier, _floats(fx[("expand", "cum_frontier")]))}
    cum_arr = np.zeros(max(frontier) + 1)
    for u, c in cum.items():
        cum_arr[u] = c
    w = int(fx[("expand", "w")][0])
    parent, token, score = oracle.ml_expand(np.log(probs), frontier, cum_arr, w)
    assert list(parent) == _ints(fx[("expand", "parent")])
    assert list(token) == _ints(fx[("expand", "token")])
    assert np.allclose(score, _floats(fx[("expand", "score")]), atol=1e-5)


def test_worked_expansion():
    check_worked_expansion()


def check_brute_force_by_probability(seed, nf=3, vocab=7, w=6):
    # rank every candidate child by the probability of its root-to-child path,
    # exp(cum[parent]) * softmax(z)[v], computed with exponentials only
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((nf, vocab)) * 2
    frontier = list(rng.choice(np.arange(10, 30), size=nf, replace=False))
    cum = np.zeros(30)
    cum[frontier] = -rng.uniform(0, 3, size=nf)
    cands = []
    for f, v in itertools.product(range(nf), range(vocab)):
        e = [math.exp(x) for x in z[f]]
        prob = math.exp(cum[frontier[f]]) * e[v] / sum(e)
        cands.append((-prob, f, v))
    cands.sort()
    want = cands[:w]
    parent, token, score = oracle.ml_expand(z, frontier, cum, w)
    assert [int(p) for p in parent] == [frontier[f] for _, f, _ in want]
    assert [int(t) for t in token] == [v for _, _, v in want]
    assert np.allclose(np.exp(score), [-p for p, _, _ in want], rtol=1e-12)


def test_brute_force_by_probability():
    for seed in range(10):
        check_brute_force_by_probability(seed)


def check_single_root_is_argmax(seed):
    z = np.random.default_rng(seed).standard_normal((1, 1000))
    parent, token, score = oracle.ml_expand(z, [0], [0.0], 1)
    assert parent[0] == 0 and token[0] == int(np.argmax(z[0]))
    assert np.isclose(score[0], z[0].max() - math.log(np.exp(z[0]).sum()))


def test_single_root_is_argmax():
    for seed in range(3):
        check_single_root_is_argmax(seed)


def check_ties_go_to_lower_position_then_token():
    z = np.zeros((2, 5))
    parent, token, _ = oracle.ml_expand(z, [4, 2], [0.0, 0.0, 0.0, 0.0, 0.0], 7)
    assert list(parent) == [4, 4, 4, 4, 4, 2, 2]
    assert list(token) == [0, 1, 2, 3, 4, 0, 1]


def test_ties_go_to_lower_position_then_token():
    check_ties_go_to_lower_position_then_token()


def test_selected_dominate_the_rest():
    rng = np.random.default_rng(5)
    z = rng.standard_normal((8, 500))
    cum = -rng.uniform(0, 4, size=8)
    parent, token, score = oracle.ml_expand(z, list(range(8)), cum, 8)
    lp = z - z.max(1, keepdims=True)
    lp -= np.log(np.exp(lp).sum(1, keepdims=True))
    allsc = cum[:, None] + lp
    chosen = set(zip(parent.tolist(), token.tolist()))
    rest = [allsc[f, v] for f in range(8) for v in range(500) if (f, v) not in chosen]
    assert score.min() >= max(rest)
    assert all(np.diff(score) <= 0)


# ------------------------------------------------------------ re-rooting

def check_worked_reroot(case):
    fx = _fixture()
    parent = _ints(fx[("reroot", "parent")])
    token = _ints(fx[("reroot", "token")])
    cum = _floats(fx[("reroot", "cum")])
    P = int(fx[("reroot", "prefix")][0])
    key = "reroot" + case
    res = oracle.draft_reroot(parent, token, cum, _ints(fx[(key, "path")]),
                              int(fx[(key, "bonus")][0]), P)
    assert list(res["new_pos"]) == _ints(fx[(key, "new_pos")])
    r = int(fx[(key, "r")][0])
    assert res["n_survivors"] == r
    if r:
        assert list(res["new_parent"][:r]) == _ints(fx[(key, "new_parent")])
        assert list(res["new_token"][:r]) == _ints(fx[(key, "new_token")])
        assert np.allclose(res["new_cum"][:r], _floats(fx[(key, "new_cum")]))
    assert all(x == -1 for x in res["new_parent"][r:])


@pytest.mark.parametrize("case", ["A", "B", "C"])
def test_worked_reroot(case):
    check_worked_reroot(case)


def _random_tree(rng, n):
    parent = [-1] + [int(rng.integers(0, i)) for i in range(1, n)]
    token = [int(rng.integers(0, 3)) for _ in range(n)]
    return parent, token


@pytest.mark.parametrize("seed", range(20))
def test_reroot_preserves_the_subtree(seed):
    rng = np.random.default_rng(seed)
    n, P = 30, 100
    parent, token = _random_tree(rng, n)
    cum = list(-np.cumsum(rng.uniform(0, 1, size=n)))
    path = oracle.ancestors_inclusive(parent, int(rng.integers(0, n)))[::-1]
    bonus = int(rng.integers(0, 3))
    res = oracle.draft_reroot(parent, token, cum, path, bonus, P)
    r = res["n_survivors"]
    kept = [i for i in range(n) if res["new_pos"][i] >= 0]
    rows = sorted(res["new_pos"][i] for i in kept)
    assert rows == list(range(P, P + len(path) + r))      # contiguous, distinct
    for k, a in enumerate(path):
        assert res["new_pos"][a] == P + k                  # the path first, in order
    surv = sorted(kept, key=lambda i: res["new_pos"][i])[len(path):]
    assert surv == sorted(surv)                            # ascending node order
    if r:
        b = surv[0]
        assert parent[b] == path[-1] and token[b] == bonus
        for k, node in enumerate(surv):
            assert res["new_token"][k] == token[node]
            assert np.isclose(res["new_cum"][k], cum[node] - cum[b])
            if k:
                assert surv[res["new_parent"][k]] == parent[node]
    else:
        assert not any(parent[c] == path[-1] and token[c] == bonus for c in range(n))
