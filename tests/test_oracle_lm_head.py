"""Pins of the LM-head oracle (oracle/lm_head.py): torch's fp64 matmul and
argmax, a hand-built case whose winning tokens and tie are known, and the
per-node selection."""
import numpy as np
import pytest
import torch

import oracle


def check_matches_torch(seed):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((7, 96))
    w = rng.standard_normal((500, 96))
    want = torch.argmax(torch.from_numpy(h) @ torch.from_numpy(w).T, dim=1).numpy()
    assert np.array_equal(oracle.lm_head_argmax(h, w), want)
    assert np.allclose(oracle.lm_head_logits(h, w), h @ w.T)


@pytest.mark.parametrize("seed", range(3))
def test_matches_torch(seed):
    check_matches_torch(seed)


def check_hand_built_winner_and_tie():
    # node 0's hidden state is e_2; the weight rows of tokens 5 and 9 are both
    # 3 e_2 (a tie: the lower id wins) and every other row is e_2; node 1's
    # hidden state is -e_0 and only token 11 has a negative first weight
    h = np.zeros((2, 4))
    h[0, 2] = 1.0
    h[1, 0] = -1.0
    w = np.zeros((12, 4))
    w[:, 2] = 1.0
    w[5, 2] = 3.0
    w[9, 2] = 3.0
    w[11, 0] = -2.0    # node 1: -1 * -2 = 2 beats every other row (0)
    assert oracle.lm_head_argmax(h, w).tolist() == [5, 11]


def test_hand_built_winner_and_tie():
    check_hand_built_winner_and_tie()


def test_node_subset():
    rng = np.random.default_rng(3)
    h = rng.standard_normal((10, 32))
    w = rng.standard_normal((200, 32))
    full = oracle.lm_head_argmax(h, w)
    assert oracle.lm_head_argmax(h, w, nodes=[7, 2]).tolist() == [full[7], full[2]]
