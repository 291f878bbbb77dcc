"""CPU oracle for the target's LM head fused with the argmax -- TEST
INFRASTRUCTURE.

Only the tests, the package's smoke check and the benchmark's CPU-baseline
leg may import this module; the product path never calls it.

The verification needs the target's argmax at every tree node (SwiftSpec
review page, "What carries the argument": the verified tokens are the
target's); the target produces it from the last hidden state of each node
through its LM head.  The plain definition: logits = H . W^T (hidden states H
[N][d_model], LM-head weights W [V][d_model]) and am[i] = argmax_v logits[i][v]
with ties to the lowest v.  Here in fp64 on the stored (rounded) values.
Pinned by tests/test_oracle_lm_head.py.
"""
from __future__ import annotations

import numpy as np

from .tree_verify import target_argmax


def lm_head_logits(hidden, weight) -> np.ndarray:
    """logits[i][v] = sum_k hidden[i][k] * weight[v][k], in fp64."""
    return np.asarray(hidden, dtype=np.float64) @ np.asarray(weight, dtype=np.float64).T


def lm_head_argmax(hidden, weight, nodes=None) -> np.ndarray:
    """The argmax of each node's logits (lowest token id on ties); only the
    listed nodes when `nodes` is given."""
    h = np.asarray(hidden, dtype=np.float64)
    if nodes is not None:
        h = h[list(nodes)]
    return target_argmax(lm_head_logits(h, weight))
