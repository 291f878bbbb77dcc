"""GPU parity of the draft side (through the C ABI) against the oracle:
maximum-likelihood expansion and draft re-rooting, then the draft cache's
compaction with the re-root map.

The expansion's selection is a discrete decision made on float32 scores by
the kernel and on float64 scores by the oracle.  What is unique is compared
exactly: the selected set wherever the oracle's w-th and (w+1)-th scores
differ by more than the float32 error bound, and the order wherever
consecutive selected scores do; elsewhere the GPU's picks must be a valid
top-w within that bound.  Re-rooting is integer work and bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from workloads import synth

tvp = pytest.importorskip("speculative_decoding_tree_masked_gb300")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
# float32 score error bound: a log-sum-exp over <= 5e5 terms plus a sum of
# three numbers of magnitude <= 40 stays far below this
TOL = 2e-4


def _check_expansion(logits, frontier, cum, w, got):
    nf, vocab = logits.shape
    flat = oracle.candidate_scores(logits, frontier, cum).ravel()
    order = np.lexsort((np.arange(flat.size), -flat))
    want = order[:w]
    pos = {int(u): f for f, u in enumerate(frontier)}
    gp = got["parent"].cpu().numpy()
    gt = got["token"].cpu().numpy()
    gs = got["score"].cpu().numpy().astype(np.float64)
    assert ((gt >= 0) & (gt < vocab)).all()
    gidx = np.array([pos[int(p)] * vocab + int(t) for p, t in zip(gp, gt)])
    assert len(set(gidx.tolist())) == w                      # distinct candidates
    assert np.abs(flat[gidx] - gs).max() <= TOL              # each pick's own score
    nxt = flat[order[w]] if w < flat.size else -np.inf
    if flat[want[-1]] - nxt > TOL:
        assert set(gidx.tolist()) == set(want.tolist())
    else:
        assert (flat[gidx] >= flat[want[-1]] - TOL).all()
    assert (np.diff(gs) <= TOL).all()                       # best first
    ws = flat[want]
    for k in range(w):                                       # order where unambiguous
        lo = ws[k - 1] - ws[k] > TOL if k > 0 else True
        hi = ws[k] - ws[k + 1] > TOL if k + 1 < w else True
        if lo and hi:
            assert gidx[k] == want[k]


@pytest.mark.parametrize("nf,vocab,w", [(1, 1000, 1), (1, 128256, 8), (8, 128256, 8),
                                        (3, 33, 16), (8, 4099, 64), (128, 997, 8),
                                        (16, 128256, 64), (5, 1, 5), (2, 524288, 16), (1, 131072, 64),
                                        # w = 1 over many slices per row (a chain draft)
                                        (1, 128256, 1), (8, 128256, 1), (64, 128256, 1),
                                        (3, 5000, 1), (128, 3000, 1),
                                        # merge clusters of 2, 5 and 8 CTAs
                                        (9, 20000, 8), (40, 4099, 8), (100, 128256, 4)])
@pytest.mark.parametrize("seed", [0, 1])
def test_expansion_matches_oracle(nf, vocab, w, seed):
    rng = np.random.default_rng(seed)
    logits = (rng.standard_normal((nf, vocab), dtype=np.float32) * 3).astype(np.float32)
    n_nodes = nf + 11
    frontier = rng.choice(n_nodes, size=nf, replace=False).astype(np.int32)
    cum = (-rng.uniform(0, 6, size=n_nodes)).astype(np.float32)
    got = tvp.tree_expand(torch.from_numpy(logits).to(DEV), torch.from_numpy(frontier).to(DEV),
                          torch.from_numpy(cum).to(DEV), w)
    torch.cuda.synchronize()
    _check_expansion(logits, frontier, cum, w, got)


def test_all_equal_scores_follow_the_tie_rule():
    nf, vocab, w = 3, 50, 20
    logits = torch.zeros((nf, vocab), dtype=torch.float32, device=DEV)
    frontier = torch.tensor([7, 2, 5], dtype=torch.int32, device=DEV)
    cum = torch.zeros(10, dtype=torch.float32, device=DEV)
    got = tvp.tree_expand(logits, frontier, cum, w)
    p, t, s = oracle.ml_expand(np.zeros((nf, vocab)), [7, 2, 5], np.zeros(10), w)
    assert got["parent"].cpu().tolist() == p.tolist()
    assert got["token"].cpu().tolist() == t.tolist()


@pytest.mark.parametrize("w", [1, 8, 64])
def test_ties_across_slices_and_rows_follow_the_tie_rule(w):
    # identical rows of 128256 logits with 40 equal maxima spread over the
    # vocabulary (so over many slices), equal path scores: every pick ties,
    # and the order is fixed by the frontier position, then the token id
    rng = np.random.default_rng(w)
    nf, vocab = 3, 128256
    row = np.full(vocab, -5.0, dtype=np.float32)
    row[rng.choice(vocab, size=40, replace=False)] = 2.0
    logits = np.tile(row, (nf, 1))
    frontier = np.array([9, 4, 6], dtype=np.int32)
    cum = np.full(12, -1.5, dtype=np.float32)
    got = tvp.tree_expand(torch.from_numpy(logits).to(DEV), torch.from_numpy(frontier).to(DEV),
                          torch.from_numpy(cum).to(DEV), w)
    p, t, _ = oracle.ml_expand(logits.astype(np.float64), frontier, cum.astype(np.float64), w)
    assert got["parent"].cpu().tolist() == p.tolist()
    assert got["token"].cpu().tolist() == t.tolist()
    sc = got["score"].cpu().numpy()
    assert (sc == sc[0]).all()                  # the same arithmetic on equal inputs


def test_unaligned_logits_rows():
    # a view that starts one float into a buffer: rows are not 16-byte aligned
    rng = np.random.default_rng(5)
    nf, vocab, w = 4, 4096, 8
    logits = (rng.standard_normal((nf, vocab)) * 3).astype(np.float32)
    buf = torch.empty(nf * vocab + 1, dtype=torch.float32, device=DEV)
    buf[1:] = torch.from_numpy(logits.reshape(-1)).to(DEV)
    frontier = np.array([3, 0, 7, 5], dtype=np.int32)
    cum = (-rng.uniform(0, 6, size=8)).astype(np.float32)
    got = tvp.tree_expand(buf[1:].view(nf, vocab), torch.from_numpy(frontier).to(DEV),
                          torch.from_numpy(cum).to(DEV), w)
    torch.cuda.synchronize()
    _check_expansion(logits, frontier, cum, w, got)


def test_masked_vocabulary_entries_are_never_preferred():
    rng = np.random.default_rng(3)
    nf, vocab, w = 4, 3000, 8
    logits = rng.standard_normal((nf, vocab)).astype(np.float32)
    logits[:, ::2] = -np.inf                    # even token ids excluded
    logits[1, :] = -np.inf                      # a row with nothing allowed
    frontier = np.arange(nf, dtype=np.int32)
    cum = np.zeros(nf, dtype=np.float32)
    got = tvp.tree_expand(torch.from_numpy(logits).to(DEV), torch.from_numpy(frontier).to(DEV),
                          torch.from_numpy(cum).to(DEV), w)
    assert (got["token"].cpu().numpy() % 2 == 1).all()
    assert (got["parent"].cpu().numpy() != 1).all()
    finite = np.isfinite(logits[[0, 2, 3]])
    assert finite.any()
    sub = logits[[0, 2, 3]]
    _check_expansion(sub, np.array([0, 2, 3], dtype=np.int32), cum, w,
                     {k: v for k, v in got.items()})


def test_bad_frontier_entry_is_reported():
    logits = torch.zeros((2, 100), dtype=torch.float32, device=DEV)
    frontier = torch.tensor([0, 12], dtype=torch.int32, device=DEV)
    cum = torch.zeros(5, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = tvp.tree_expand(logits, frontier, cum, 4, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == tvp.TV_ERR_INVALID_ARG
    assert (got["token"].cpu() == -1).all()


@pytest.mark.parametrize("bad_row", [3, 30, 39])
def test_bad_frontier_entry_in_any_merge_cta_is_reported(bad_row):
    # 40 rows: the merge runs as a cluster of 5 CTAs, row f held by CTA
    # (f / 8) % 5; a bad entry in any of them must reach CTA 0's check
    rng = np.random.default_rng(bad_row)
    nf, vocab = 40, 3000
    logits = torch.from_numpy(rng.standard_normal((nf, vocab), dtype=np.float32)).to(DEV)
    frontier = torch.arange(nf, dtype=torch.int32, device=DEV)
    frontier[bad_row] = nf + 7
    cum = torch.zeros(nf, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = tvp.tree_expand(logits, frontier, cum, 8, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == tvp.TV_ERR_INVALID_ARG
    assert (got["token"].cpu() == -1).all() and (got["parent"].cpu() == -1).all()


# ---------------------------------------------------------------- re-rooting

def _draft_case(seed, n_verified, n_draft, vocab=6):
    """A verified tree (the first n_verified nodes) that the draft has since
    grown to n_draft nodes, target logits that plant a random accepted path,
    and a bonus token that some later child of a_m may carry."""
    rng = np.random.default_rng(seed)
    parent = np.asarray(synth.uniform_parent_tree(rng, n_draft, max_depth=12, max_fanout=4),
                        dtype=np.int32)
    token = rng.integers(0, vocab, size=n_draft).astype(np.int32)
    cum = (-np.cumsum(rng.uniform(0.01, 1, size=n_draft))).astype(np.float32)
    cum[0] = 0.0
    logits = rng.standard_normal((n_verified, vocab)).astype(np.float32)
    return parent, token, cum, logits


@pytest.mark.parametrize("seed", range(12))
def test_draft_reroot_matches_oracle(seed):
    n0, n = [(8, 20), (64, 128), (30, 30), (1, 5)][seed % 4]
    parent, token, cum, logits = _draft_case(seed, n0, n)
    P = 77 + seed
    acc = tvp.tree_accept(torch.from_numpy(logits).to(DEV),
                          torch.from_numpy(token[:n0].copy()).to(DEV),
                          torch.from_numpy(parent[:n0].copy()).to(DEV), P)
    want_acc = oracle.tree_accept(logits, token[:n0], parent[:n0], P)
    m = want_acc["m"]
    path = want_acc["path"][:m + 1]
    bonus = int(want_acc["out_tokens"][m])
    want = oracle.draft_reroot(parent, token, cum.astype(np.float64), path, bonus, P)
    got = tvp.draft_reroot(torch.from_numpy(parent).to(DEV), torch.from_numpy(token).to(DEV),
                           torch.from_numpy(cum).to(DEV), acc, P)
    torch.cuda.synchronize()
    r = want["n_survivors"]
    assert int(got["n_survivors"].item()) == r
    assert got["new_pos"].cpu().tolist() == want["new_pos"].tolist()
    assert got["new_parent"].cpu().tolist() == want["new_parent"].tolist()
    assert got["new_token"].cpu().tolist() == want["new_token"].tolist()
    assert np.allclose(got["new_cum"].cpu().numpy(), want["new_cum"], atol=1e-6)


def test_bonus_child_survives_with_its_subtree():
    # the draft grew a child of a_m carrying the bonus token after the snapshot
    parent = np.array([-1, 0, 0, 1, 3, 3, 4, 5, 2], dtype=np.int32)
    token = np.array([0, 1, 2, 3, 4, 5, 6, 7, 8], dtype=np.int32)
    cum = np.array([0, -1, -2, -1.5, -2.5, -3, -3.5, -4, -4.5], dtype=np.float32)
    n0 = 3                                  # nodes 0..2 were verified
    logits = np.zeros((n0, 10), dtype=np.float32)
    logits[0, 1] = 5                        # root -> node 1 (token 1)
    logits[1, 3] = 5                        # node 1 -> bonus token 3 (node 3 is not verified)
    acc = tvp.tree_accept(torch.from_numpy(logits).to(DEV),
                          torch.from_numpy(token[:n0].copy()).to(DEV),
                          torch.from_numpy(parent[:n0].copy()).to(DEV), 40)
    got = tvp.draft_reroot(torch.from_numpy(parent).to(DEV), torch.from_numpy(token).to(DEV),
                           torch.from_numpy(cum).to(DEV), acc, 40)
    # path 0 1, bonus 3 -> b = node 3, subtree 3 4 5 6 7
    assert int(got["n_survivors"].item()) == 5
    assert got["new_pos"].cpu().tolist() == [40, 41, -1, 42, 43, 44, 45, 46, -1]
    assert got["new_parent"].cpu().tolist()[:5] == [-1, 0, 0, 1, 2]
    assert np.allclose(got["new_cum"].cpu().numpy()[:5], [0, -1, -1.5, -2, -2.5])


def test_invalid_path_is_reported():
    parent = torch.tensor([-1, 0, 1], dtype=torch.int32, device=DEV)
    token = torch.tensor([0, 1, 2], dtype=torch.int32, device=DEV)
    cum = torch.zeros(3, dtype=torch.float32, device=DEV)
    bad = {"path": torch.tensor([0, 2, -1], dtype=torch.int32, device=DEV),
           "m": torch.tensor([1], dtype=torch.int32, device=DEV),
           "out_tokens": torch.tensor([1, 2, -1, -1], dtype=torch.int32, device=DEV)}
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = tvp.draft_reroot(parent, token, cum, bad, 10, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == tvp.TV_ERR_INVALID_TREE
    assert (got["new_pos"].cpu() == -1).all()


@pytest.mark.parametrize("seed", range(4))
def test_draft_cache_compaction_with_reroot_map(seed):
    n0, n = 32, 96
    parent, token, cum, logits = _draft_case(100 + seed, n0, n)
    P, L, hkv, d = 50, 2, 4, 128
    cap = P + n + 3
    acc = tvp.tree_accept(torch.from_numpy(logits).to(DEV),
                          torch.from_numpy(token[:n0].copy()).to(DEV),
                          torch.from_numpy(parent[:n0].copy()).to(DEV), P)
    got = tvp.draft_reroot(torch.from_numpy(parent).to(DEV), torch.from_numpy(token).to(DEV),
                           torch.from_numpy(cum).to(DEV), acc, P)
    rng = np.random.default_rng(seed)
    k = torch.from_numpy(rng.standard_normal((L, hkv, cap, d), dtype=np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((L, hkv, cap, d), dtype=np.float32)).to(torch.bfloat16)
    kd, vd = k.to(DEV), v.to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tvp.kv_compact(kd, vd, P, n, got["new_pos"], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    new_pos = got["new_pos"].cpu().numpy()
    bits = lambda t: t.view(torch.int16).cpu().numpy()
    assert np.array_equal(bits(kd), oracle.kv_compact(bits(k), P, new_pos))
    assert np.array_equal(bits(vd), oracle.kv_compact(bits(v), P, new_pos))
