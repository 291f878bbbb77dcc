"""CPU oracle for sampling (stochastic) tree verification -- TEST
INFRASTRUCTURE.

Only the tests, the package's smoke check and the benchmark's CPU-baseline
leg may import this module.  The product path never calls it, and it shares
no code with that path.

The SwiftSpec review page verifies greedily ("What carries the argument":
verified tokens are the target's) and says nothing of sampling; this module
is the library's reading of the sampling case for the trees the draft grows
deterministically by maximum-likelihood expansion (review page, "Assumptions
& free parameters"):

  S1  At temperature T > 0 the target's distribution at tree node i is
      p_i = softmax(z_i / T) over the vocabulary.
  S2  One uniform u_i in (0, 1) per node comes from the counter-based
      generator Philox4x64-10 (Salmon, Moraes, Dror and Shaw, "Parallel
      random numbers: as easy as 1, 2, 3", SC 2011) with key (seed, 0) and
      counter (i, offset, 0, 0): u_i = (x0 >> 11 + 1/2) / 2^53 for the first
      output word x0.
  S3  The target's token at node i is drawn by inversion: the smallest v with
      p_i[0] + ... + p_i[v] > u_i.
  S4  The walk is the greedy walk with the drawn tokens in place of the
      argmax: from the root, follow the lowest-indexed child that carries
      the token drawn at the current node; the first draw that no child
      carries is the bonus token.  Every emitted token is then a draw from
      the target's own distribution at its context, which is what makes the
      scheme lossless.

Plain fp64 NumPy, the steps in order.  Pinned by tests/test_oracle_sample.py.
"""
from __future__ import annotations

from typing import Sequence

import numpy as np

from .tree_verify import accepted_tokens, greedy_walk, reroot

_MASK = (1 << 64) - 1
# Philox4x64 round multipliers and key increments (the published constants)
_M0, _M1 = 0xD2E7470EE14C6C93, 0xCA5A826395121157
_W0, _W1 = 0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B


def philox4x64_10(counter: Sequence[int], key: Sequence[int]) -> list[int]:
    """Ten Philox rounds on a 4 x 64-bit counter with a 2 x 64-bit key."""
    x0, x1, x2, x3 = (int(c) & _MASK for c in counter)
    k0, k1 = (int(k) & _MASK for k in key)
    for _ in range(10):
        p0 = _M0 * x0
        p1 = _M1 * x2
        x0, x1, x2, x3 = ((p1 >> 64) ^ x1 ^ k0) & _MASK, p1 & _MASK, \
            ((p0 >> 64) ^ x3 ^ k1) & _MASK, p0 & _MASK
        k0 = (k0 + _W0) & _MASK
        k1 = (k1 + _W1) & _MASK
    return [x0, x1, x2, x3]


def node_uniform(seed: int, offset: int, node: int) -> float:
    """u_i of reading S2, exactly representable in fp64."""
    x0 = philox4x64_10([node, offset, 0, 0], [seed, 0])[0]
    return ((x0 >> 11) + 0.5) / float(1 << 53)


def target_probs(logits, temperature: float) -> np.ndarray:
    """Reading S1 in fp64: softmax(z / T) per row."""
    if not temperature > 0:
        raise ValueError("temperature must be positive")
    z = np.asarray(logits, dtype=np.float64) / float(temperature)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def draw_by_inversion(probs_row, u: float) -> int:
    """Reading S3: the smallest v whose cumulative probability exceeds u (the
    last token with positive probability if rounding leaves u above it)."""
    c = np.cumsum(np.asarray(probs_row, dtype=np.float64))
    v = int(np.searchsorted(c, u, side="right"))
    if v >= len(c):
        v = int(np.flatnonzero(np.asarray(probs_row) > 0)[-1])
    return v


def sample_tokens(logits, temperature: float, seed: int, offset: int) -> np.ndarray:
    """The target's drawn token at every node (readings S1-S3)."""
    p = target_probs(logits, temperature)
    return np.array([draw_by_inversion(p[i], node_uniform(seed, offset, i))
                     for i in range(p.shape[0])], dtype=np.int32)


def tree_accept_sampled(logits, token: Sequence[int], parent: Sequence[int], prefix_len: int,
                        temperature: float, seed: int, offset: int) -> dict:
    """Sampling verification (reading S4) laid out like tree_accept's result,
    with the drawn tokens under "sampled"."""
    n = len(parent)
    s = sample_tokens(logits, temperature, seed, offset)
    path = greedy_walk(s, token, parent)
    toks = accepted_tokens(path, s, token)
    new_pos, new_parent, r = reroot(parent, path, prefix_len)
    path_out = np.full(n, -1, dtype=np.int32)
    path_out[:len(path)] = path
    tok_out = np.full(n + 1, -1, dtype=np.int32)
    tok_out[:len(toks)] = toks
    return {"sampled": s, "m": len(path) - 1, "path": path_out, "out_tokens": tok_out,
            "new_pos": new_pos, "new_parent": new_parent, "n_survivors": r}
