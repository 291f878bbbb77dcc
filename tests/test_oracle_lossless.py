"""Losslessness of the oracle's verification step (SwiftSpec review page,
"Core claim": speculative decoding emits exactly what the target would
decode greedily): speculative decoding of a toy one-layer target through the
oracle's tree attention, acceptance and KV compaction emits exactly the
tokens of the target's own autoregressive greedy decode, written out
independently in tests/toy_target.py.  This pins attention, the walk and
the compaction jointly: a wrong mask, a wrong bonus token or a row moved to
the wrong place changes a later step's context and so its tokens."""
import numpy as np
import pytest

import oracle
from tests.toy_target import ToyTarget, draft_tree


def speculative_decode(model: ToyTarget, prompt, n_new, reference, rng, n_nodes, plant):
    """Greedy tree verification with the oracle, step after step, until
    n_new tokens are emitted.  The draft plants the reference's continuation
    along one path with probability `plant` per node."""
    P = len(prompt) - 1                       # the last prompt token is the first root
    cap = len(prompt) + n_new + n_nodes + 4
    K = np.zeros((model.hkv, cap, model.dh))
    V = np.zeros((model.hkv, cap, model.dh))
    _, k, v = model.qkv(model.embed(prompt[:-1], range(P)))
    K[:, :P], V[:, :P] = k.transpose(1, 0, 2), v.transpose(1, 0, 2)
    root, emitted, accepted = int(prompt[-1]), [], []
    while len(emitted) < n_new:
        parent, token, depth = draft_tree(rng, root, reference[len(emitted):], model.vocab,
                                          n_nodes, plant)
        n = len(parent)
        x = model.embed(token, P + depth)
        q, k, v = model.qkv(x)
        K[:, P:P + n], V[:, P:P + n] = k.transpose(1, 0, 2), v.transpose(1, 0, 2)
        o = oracle.tree_attention(q, K, V, P, parent)
        z = model.logits(model.hidden(x, o))
        acc = oracle.tree_accept(z, token, parent, P)
        m = acc["m"]
        emitted += [int(t) for t in acc["out_tokens"][:m + 1]]
        accepted.append(m)
        K = oracle.kv_compact(K, P, acc["new_pos"])
        V = oracle.kv_compact(V, P, acc["new_pos"])
        P += m + 1
        root = emitted[-1]
    return emitted[:n_new], accepted


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("n_nodes,plant", [(1, 0.0), (8, 0.0), (8, 0.7), (15, 1.0), (12, 0.5)])
def test_speculative_equals_autoregressive(seed, n_nodes, plant):
    model = ToyTarget(seed)
    rng = np.random.default_rng(100 + seed)
    prompt = [int(t) for t in rng.integers(model.vocab, size=20)]
    n_new = 40
    reference, margins = model.greedy_decode(prompt, n_new)
    assert min(margins) > 1e-9                 # no exact ties to break
    got, accepted = speculative_decode(model, prompt, n_new, reference, rng, n_nodes, plant)
    assert got == reference
    if plant == 1.0:
        assert max(accepted) >= n_nodes - 2    # whole planted paths were accepted
    if n_nodes == 1:
        assert set(accepted) == {0}            # a lone root emits only the bonus token
