"""GPU parity of greedy acceptance and the re-root map (through the C ABI)
against the oracle, bit for bit: planted path lengths, random logits over the
128256-token vocabulary, duplicate sibling tokens, ties and NaNs, vocabularies
that defeat vector loads, and device-side validation."""
import numpy as np
import pytest
import torch

import oracle
from workloads import synth

tvp = pytest.importorskip("speculative_decoding_tree_masked_gb300")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
KEYS = ("am", "path", "out_tokens", "new_pos", "new_parent")


def _check(logits, token, parent, P, logits_dev=None):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ld = torch.from_numpy(np.ascontiguousarray(logits)).to(DEV) if logits_dev is None else logits_dev
    res = tvp.tree_accept(ld, torch.from_numpy(np.asarray(token, np.int32)).to(DEV),
                          torch.from_numpy(np.asarray(parent, np.int32)).to(DEV), P, status=status)
    want = oracle.tree_accept(logits, token, parent, P)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for key in KEYS:
        assert np.array_equal(res[key].cpu().numpy(), want[key]), key
    assert int(res["m"].item()) == want["m"]
    assert int(res["n_survivors"].item()) == want["n_survivors"]
    return want


@pytest.mark.parametrize("m", range(4))
def test_tiny_planted(m):
    w = synth.make_workload("tiny", seed=m, planted_m=m)
    assert _check(w.logits, w.token, w.parent, w.prefix)["m"] == m


@pytest.mark.parametrize("seed", range(9))
def test_full_step_planted(seed):
    w = synth.make_workload("full_step", seed=seed, planted_m=seed, layers=1)
    assert _check(w.logits, w.token, w.parent, w.prefix)["m"] == seed


def test_l3_8b_random_logits():
    w = synth.make_workload("l3_8b", seed=0)
    _check(w.logits, w.token, w.parent, w.prefix)


@pytest.mark.parametrize("seed", range(30))
def test_random_small_alphabet_trees(seed):
    rng = np.random.default_rng(seed)
    n = [1, 2, 5, 31, 32, 33, 64, 100, 127, 128][seed % 10]
    vocab = 3
    parent = synth.random_parent_tree(rng, n, max_depth=12)
    token = rng.integers(0, vocab, size=n).astype(np.int32)     # duplicates on purpose
    logits = rng.standard_normal((n, vocab)).astype(np.float32)
    _check(logits, token, parent, int(rng.integers(0, 5000)))


@pytest.mark.parametrize("vocab", [1, 3, 1001, 4097, 128256])
def test_ties_nans_and_odd_vocabularies(vocab):
    rng = np.random.default_rng(vocab)
    n = 40
    parent = synth.random_parent_tree(rng, n, max_depth=8)
    token = rng.integers(0, vocab, size=n).astype(np.int32)
    logits = np.round(rng.standard_normal((n, vocab)), 0).astype(np.float32)  # many ties
    logits[3, :] = 0.0
    logits[4, :] = -0.0
    logits[4, vocab // 2] = 0.0
    if vocab > 2:
        logits[5, 1] = np.nan
        logits[5, vocab - 1] = np.nan
        logits[6, :] = -np.inf
    logits[7, vocab - 1] = np.inf
    _check(logits, token, parent, 17)


def test_unaligned_logits_rows():
    # a view that starts one float into a buffer: rows are not 16-byte aligned
    rng = np.random.default_rng(9)
    n, vocab = 20, 4096
    parent = synth.random_parent_tree(rng, n, max_depth=6)
    token = rng.integers(0, vocab, size=n).astype(np.int32)
    logits = rng.standard_normal((n, vocab)).astype(np.float32)
    buf = torch.empty(n * vocab + 1, dtype=torch.float32, device=DEV)
    buf[1:] = torch.from_numpy(logits.reshape(-1)).to(DEV)
    _check(logits, token, parent, 3, logits_dev=buf[1:].view(n, vocab))


@pytest.mark.parametrize("parent,token", [
    ([0, 0, 1], [1, 2, 3]),          # root with a parent
    ([-1, 0, 2], [1, 2, 3]),         # self loop
    ([-1, 0, 1], [1, 2, 99]),        # token outside the vocabulary
])
def test_invalid_inputs_set_status(parent, token):
    logits = torch.zeros((3, 10), dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    res = tvp.tree_accept(logits, torch.tensor(token, dtype=torch.int32, device=DEV),
                          torch.tensor(parent, dtype=torch.int32, device=DEV), 5, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == tvp.TV_ERR_INVALID_TREE
    # the safe state: nothing accepted, nothing kept
    assert int(res["m"].item()) == 0 and int(res["n_survivors"].item()) == 0
    assert (res["new_pos"] == -1).all()
