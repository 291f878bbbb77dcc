"""Pins of the sampling-verification oracle (oracle/tree_sample.py): its
Philox4x64-10 against NumPy's own Philox bit generator, the drawn tokens'
distribution against softmax(z / T) by a chi-square test, the limits of the
temperature, and the lossless-walk invariant (every emitted token is the
target's draw at its node)."""
import numpy as np
import pytest

import oracle
from workloads import synth


@pytest.mark.parametrize("key", [(1, 2), (0, 0), (2**63 + 5, 7), (123456789, 987654321)])
def test_philox_matches_numpy(key):
    # NumPy's generator advances its counter before each block: the block
    # it returns from counter c is the function's output at counter c + 1
    bg = np.random.Philox(key=np.array(key, dtype=np.uint64),
                          counter=np.array([0, 0, 0, 0], dtype=np.uint64))
    raw = bg.random_raw(12)
    for c in range(3):
        assert oracle.philox4x64_10([c + 1, 0, 0, 0], key) == [int(x) for x in raw[4 * c:4 * c + 4]]


def test_philox_counter_words_all_matter():
    base = oracle.philox4x64_10([5, 6, 7, 8], [9, 10])
    for w in range(4):
        ctr = [5, 6, 7, 8]
        ctr[w] += 1
        assert oracle.philox4x64_10(ctr, [9, 10]) != base


def test_uniforms_are_open_and_uniform():
    u = np.array([oracle.node_uniform(3, 0, i) for i in range(20000)])
    assert (u > 0).all() and (u < 1).all()
    # a 20-bin histogram of 20000 uniforms
    stats = pytest.importorskip("scipy.stats")
    counts = np.histogram(u, bins=20, range=(0, 1))[0]
    assert stats.chisquare(counts).pvalue > 1e-4


def check_drawn_distribution(T, seed=0):
    stats = pytest.importorskip("scipy.stats")
    z = np.array([[0.5, -1.0, 2.0, 0.0, 1.0, -3.0]])
    nodes = 6000
    logits = np.repeat(z, nodes, axis=0)
    s = oracle.sample_tokens(logits, T, seed, 0)
    counts = np.bincount(s, minlength=6)
    e = np.exp(z[0] / T)
    expected = e / e.sum() * nodes
    assert stats.chisquare(counts, expected).pvalue > 1e-4


@pytest.mark.parametrize("T", [0.5, 1.0, 2.0])
def test_drawn_distribution_is_the_softmax(T):
    check_drawn_distribution(T)


def test_low_temperature_is_argmax():
    rng = np.random.default_rng(0)
    logits = rng.standard_normal((50, 300))
    s = oracle.sample_tokens(logits, 1e-3, 1, 0)
    assert np.array_equal(s, np.argmax(logits, axis=1))


def test_masked_tokens_are_never_drawn():
    z = np.zeros((2000, 7))
    z[:, [1, 4]] = -np.inf
    s = oracle.sample_tokens(z, 1.0, 5, 9)
    assert not np.isin(s, [1, 4]).any()


def test_inversion_edges():
    assert oracle.draw_by_inversion([0.25, 0.25, 0.5], 0.0) == 0
    assert oracle.draw_by_inversion([0.25, 0.25, 0.5], 0.25) == 1    # strictly above
    assert oracle.draw_by_inversion([0.0, 0.5, 0.5], 0.1) == 1       # zero mass skipped
    assert oracle.draw_by_inversion([0.5, 0.5, 0.0], 1.0) == 1       # rounding past the end


@pytest.mark.parametrize("seed", range(6))
def test_emitted_tokens_are_the_draws_on_the_path(seed):
    rng = np.random.default_rng(seed)
    n, vocab = 40, 5
    parent = synth.uniform_parent_tree(rng, n, max_depth=8, max_fanout=4)
    token = rng.integers(0, vocab, size=n).astype(np.int32)
    logits = rng.standard_normal((n, vocab))
    res = oracle.tree_accept_sampled(logits, token, parent, 10, 0.8, seed, 3)
    m = res["m"]
    path = res["path"][:m + 1]
    s = res["sampled"]
    # each emitted token is the draw at its node: accepted children carry the
    # draw at their parent, and the bonus is the draw at the last node
    assert list(res["out_tokens"][:m + 1]) == [int(s[a]) for a in path]
    assert all(token[path[k + 1]] == s[path[k]] for k in range(m))
    assert not any(parent[c] == path[-1] and token[c] == s[path[-1]] for c in range(n))


def test_offsets_and_seeds_change_the_draws():
    logits = np.zeros((500, 50))
    a = oracle.sample_tokens(logits, 1.0, 1, 0)
    assert not np.array_equal(a, oracle.sample_tokens(logits, 1.0, 1, 1))
    assert not np.array_equal(a, oracle.sample_tokens(logits, 1.0, 2, 0))
