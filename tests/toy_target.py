"""A toy one-layer target model for the losslessness tests: seeded random
weights, a token embedding plus a position embedding, one GQA attention layer
with a residual connection, and an LM head.  Its autoregressive greedy decode
uses a plain causal softmax written out here; neither the oracle nor the CUDA
library is used, so a speculative decode through either can be compared with
it.

    x_p      = E[t_p] + Pos[p]                      (token t_p at position p)
    q, k, v  = x_p Wq, x_p Wk, x_p Wv               (Hq, Hkv, Hkv heads of dh)
    o_p[h]   = softmax_j<=p(q_p[h] . k_j[g(h)] / sqrt(dh)) . v_j[g(h)]
    h_p      = x_p + concat_h(o_p[h]) Wo
    z_p      = Wlm h_p                              (next-token logits)
"""
from __future__ import annotations

import numpy as np


class ToyTarget:
    def __init__(self, seed: int, vocab: int = 48, d_model: int = 32, hq: int = 4,
                 hkv: int = 2, dh: int = 16, max_pos: int = 256, lm_scale: float = 3.0):
        rng = np.random.default_rng(seed)
        self.vocab, self.d_model, self.hq, self.hkv, self.dh = vocab, d_model, hq, hkv, dh
        self.E = rng.standard_normal((vocab, d_model))
        self.Pos = 0.5 * rng.standard_normal((max_pos, d_model))
        self.Wq = rng.standard_normal((d_model, hq * dh)) / np.sqrt(d_model)
        self.Wk = rng.standard_normal((d_model, hkv * dh)) / np.sqrt(d_model)
        self.Wv = rng.standard_normal((d_model, hkv * dh)) / np.sqrt(d_model)
        self.Wo = rng.standard_normal((hq * dh, d_model)) / np.sqrt(hq * dh)
        self.Wlm = lm_scale * rng.standard_normal((vocab, d_model)) / np.sqrt(d_model)

    # per-token pieces, fp64 -------------------------------------------------
    def embed(self, tokens, positions) -> np.ndarray:
        return self.E[np.asarray(tokens)] + self.Pos[np.asarray(positions)]

    def qkv(self, x):
        x = np.atleast_2d(x)
        q = (x @ self.Wq).reshape(-1, self.hq, self.dh)
        k = (x @ self.Wk).reshape(-1, self.hkv, self.dh)
        v = (x @ self.Wv).reshape(-1, self.hkv, self.dh)
        return q, k, v

    def hidden(self, x, o) -> np.ndarray:
        """x [n][d_model], o [n][hq][dh] -> the final hidden states [n][d_model]."""
        return np.atleast_2d(x) + np.asarray(o).reshape(len(np.atleast_2d(x)), -1) @ self.Wo

    def logits(self, h) -> np.ndarray:
        return np.atleast_2d(h) @ self.Wlm.T

    # the reference -----------------------------------------------------------
    def greedy_decode(self, prompt, n_new: int):
        """Autoregressive greedy decoding: returns the n_new generated tokens
        and the margin (top minus second logit) of every choice."""
        toks = list(prompt)
        ks, vs = [], []
        x = self.embed(toks, range(len(toks)))
        _, k, v = self.qkv(x)
        ks.extend(k)
        vs.extend(v)
        out, margins = [], []
        g = self.hq // self.hkv
        for step in range(n_new):
            p = len(toks) - 1
            # the last token attends every position up to and including itself;
            # its own K/V are already in the lists
            q, _, _ = self.qkv(self.embed([toks[-1]], [p]))
            kk, vv = np.stack(ks), np.stack(vs)          # [p+1][hkv][dh]
            o = np.zeros((self.hq, self.dh))
            for h in range(self.hq):
                s = kk[:, h // g, :] @ q[0, h] / np.sqrt(self.dh)
                w = np.exp(s - s.max())
                o[h] = (w / w.sum()) @ vv[:, h // g, :]
            z = self.logits(self.hidden(self.embed([toks[-1]], [p]), o[None]))[0]
            nxt = int(np.argmax(z))
            srt = np.sort(z)
            margins.append(float(srt[-1] - srt[-2]))
            out.append(nxt)
            toks.append(nxt)
            _, k, v = self.qkv(self.embed([nxt], [len(toks) - 1]))
            ks.append(k[0])
            vs.append(v[0])
        return out, margins


def draft_tree(rng: np.random.Generator, root_token: int, continuation, vocab: int,
               n_nodes: int, plant: float):
    """A random draft tree of n_nodes rooted at root_token.  Along one path from
    the root each child carries the true next token of `continuation` with
    probability `plant` (else a random token); the other nodes hang off random
    earlier nodes with random tokens, sibling tokens distinct."""
    parent = [-1]
    token = [int(root_token)]
    depth = [0]
    u = 0
    for c in continuation:
        if len(parent) >= n_nodes:
            break
        t = int(c) if rng.random() < plant else int(rng.integers(vocab))
        parent.append(u)
        token.append(t)
        depth.append(depth[u] + 1)
        u = len(parent) - 1
    while len(parent) < n_nodes:
        p = int(rng.integers(len(parent)))
        used = {token[j] for j in range(len(parent)) if parent[j] == p}
        free = [t for t in range(vocab) if t not in used]
        parent.append(p)
        token.append(int(rng.choice(free)))
        depth.append(depth[p] + 1)
    return np.asarray(parent, dtype=np.int32), np.asarray(token, dtype=np.int32), \
        np.asarray(depth, dtype=np.int64)
