"""GPU parity of sampling verification (through the C ABI) against the
oracle.  The draws are decided in float32 with double sums on the GPU and in
fp64 by the oracle: where the uniform lies well inside a token's
cumulative-probability interval the drawn tokens must agree exactly; within
1e-5 of a boundary the GPU's token must be one of the two tokens at that
boundary.  The walk over the drawn tokens is integer work and bit-exact, and
the draws' distribution must be the softmax (chi-square)."""
import numpy as np
import pytest
import torch

import oracle
from workloads import synth

tvp = pytest.importorskip("speculative_decoding_tree_masked_gb300")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
EDGE = 1e-5


def _check_draws(logits, T, seed, offset, got):
    p = oracle.target_probs(logits, T)
    for i in range(p.shape[0]):
        u = oracle.node_uniform(seed, offset, i)
        want = oracle.draw_by_inversion(p[i], u)
        g = int(got[i])
        if g == want:
            continue
        c = np.cumsum(p[i])
        lo = c[g - 1] if g > 0 else 0.0
        assert p[i][g] > 0
        assert lo - EDGE <= u < c[g] + EDGE, (i, g, want, u, lo, c[g])


@pytest.mark.parametrize("n,vocab,T", [(64, 128256, 1.0), (64, 128256, 0.7), (16, 1000, 2.0),
                                       (128, 33, 1.0), (3, 5, 0.3), (1, 131, 1.5)])
@pytest.mark.parametrize("seed", [0, 1])
def test_draws_match_oracle(n, vocab, T, seed):
    rng = np.random.default_rng(seed)
    logits = (rng.standard_normal((n, vocab)) * 3).astype(np.float32)
    parent = synth.uniform_parent_tree(rng, n, max_depth=8, max_fanout=8)
    token = rng.integers(0, vocab, size=n).astype(np.int32)
    res = tvp.tree_accept_sampled(torch.from_numpy(logits).to(DEV),
                                  torch.from_numpy(token).to(DEV),
                                  torch.from_numpy(parent).to(DEV), 50, T, 1234 + seed, 7)
    torch.cuda.synchronize()
    s = res["sampled"].cpu().numpy()
    _check_draws(logits.astype(np.float64), T, 1234 + seed, 7, s)
    # the walk over the GPU's own draws is the oracle's walk over them
    path = oracle.greedy_walk(s, token, parent)
    m = len(path) - 1
    assert int(res["m"].item()) == m
    assert res["path"].cpu().numpy()[:m + 1].tolist() == path
    assert res["out_tokens"].cpu().numpy()[:m + 1].tolist() == \
        oracle.accepted_tokens(path, s, token)
    new_pos, new_parent, r = oracle.reroot(parent, path, 50)
    assert res["new_pos"].cpu().tolist() == new_pos.tolist()
    assert int(res["n_survivors"].item()) == r


def test_draws_follow_the_softmax():
    stats = pytest.importorskip("scipy.stats")
    z = np.array([0.5, -1.0, 2.0, 0.0, 1.0, -3.0, 0.25], dtype=np.float32)
    n, T = 128, 0.8
    logits = torch.from_numpy(np.tile(z, (n, 1))).to(DEV)
    parent = torch.from_numpy(synth.chain_tree(n)).to(DEV)
    token = torch.zeros(n, dtype=torch.int32, device=DEV)
    counts = np.zeros(len(z))
    for off in range(60):
        res = tvp.tree_accept_sampled(logits, token, parent, 0, T, 99, off)
        counts += np.bincount(res["sampled"].cpu().numpy(), minlength=len(z))
    e = np.exp(z.astype(np.float64) / T)
    assert stats.chisquare(counts, e / e.sum() * counts.sum()).pvalue > 1e-4


def test_low_temperature_is_the_argmax():
    rng = np.random.default_rng(4)
    logits = torch.from_numpy(rng.standard_normal((32, 5000)).astype(np.float32)).to(DEV)
    parent = torch.from_numpy(synth.chain_tree(32)).to(DEV)
    token = torch.zeros(32, dtype=torch.int32, device=DEV)
    res = tvp.tree_accept_sampled(logits, token, parent, 0, 1e-4, 3, 0)
    assert np.array_equal(res["sampled"].cpu().numpy(), logits.argmax(dim=1).cpu().numpy())


def test_masked_tokens_and_empty_rows():
    z = np.zeros((4, 64), dtype=np.float32)
    z[:, ::3] = -np.inf
    z[2, :] = -np.inf
    parent = torch.from_numpy(synth.chain_tree(4)).to(DEV)
    token = torch.zeros(4, dtype=torch.int32, device=DEV)
    for off in range(10):
        res = tvp.tree_accept_sampled(torch.from_numpy(z).to(DEV), token, parent, 0, 1.0, 5, off)
        s = res["sampled"].cpu().numpy()
        assert s[2] == -1
        assert all(s[i] % 3 != 0 and 0 <= s[i] < 64 for i in (0, 1, 3))


def test_same_counter_same_draws():
    rng = np.random.default_rng(8)
    logits = torch.from_numpy(rng.standard_normal((64, 9000)).astype(np.float32)).to(DEV)
    parent = torch.from_numpy(synth.chain_tree(64)).to(DEV)
    token = torch.zeros(64, dtype=torch.int32, device=DEV)
    a = tvp.tree_accept_sampled(logits, token, parent, 0, 1.0, 11, 3)["sampled"].cpu()
    b = tvp.tree_accept_sampled(logits, token, parent, 0, 1.0, 11, 3)["sampled"].cpu()
    c = tvp.tree_accept_sampled(logits, token, parent, 0, 1.0, 11, 4)["sampled"].cpu()
    assert torch.equal(a, b) and not torch.equal(a, c)
