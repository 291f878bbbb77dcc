"""GPU parity of the batched acceptance and compaction (several requests'
trees packed into one pass, through the C ABI) against the oracle applied to
each request on its own, bit for bit: acceptance over packed logits, the
token-given walk, compaction of per-request caches and of one shared page
pool, the isolation of a bad request, and a whole batched verification step
(batched attention, acceptance and compaction) chained on the device."""
import numpy as np
import pytest
import torch

import oracle
from workloads import synth

tvp = pytest.importorskip("speculative_decoding_tree_masked_gb300")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
BF16_TOL = 2e-2
KEYS = ("path", "out_tokens", "new_pos", "new_parent")


def _requests(rng, ns, vocab, planted=True):
    """Per request: parent, token, logits (planted path length when the tree
    is deep enough, else random), prefix."""
    reqs = []
    for n in ns:
        parent = np.asarray(synth.uniform_parent_tree(rng, n, max_depth=8, max_fanout=8),
                            dtype=np.int32)
        token = np.asarray(synth.draft_tokens(rng, parent, vocab), dtype=np.int32)
        if planted:
            depth = synth.node_depths(parent)
            logits, _ = synth.planted_logits(rng, parent, token, vocab,
                                             int(rng.integers(0, depth.max() + 1)))
        else:
            logits = rng.standard_normal((n, vocab), dtype=np.float32)
        reqs.append((parent, token, logits, int(rng.integers(0, 9000))))
    return reqs


def _packed(reqs):
    cat = lambda i: torch.from_numpy(np.concatenate([r[i] for r in reqs])).to(DEV)
    return cat(0), cat(1), cat(2).contiguous()


def _assert_request(res, b, want):
    got = tvp.batched_request(res, b)
    for key in KEYS:
        assert np.array_equal(got[key].cpu().numpy(), want[key]), (b, key)
    if "am" in got:
        assert np.array_equal(got["am"].cpu().numpy(), want["am"]), (b, "am")
    assert int(got["m"].item()) == want["m"], b
    assert int(got["n_survivors"].item()) == want["n_survivors"], b


@pytest.mark.parametrize("ns,vocab", [
    ([64], 128256),
    ([64, 8, 128, 1, 33], 128256),
    ([int(x) for x in np.random.default_rng(1).integers(1, 129, 16)], 1000),
    ([128] * 16, 4097),
    ([1] * 16, 50),
])
def test_batched_accept_matches_oracle(ns, vocab):
    rng = np.random.default_rng(len(ns) * 7 + vocab)
    reqs = _requests(rng, ns, vocab)
    parent, token, logits = _packed(reqs)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    res = tvp.tree_accept_batched(logits, token, parent, ns, [r[3] for r in reqs], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for b, (par, tok, lg, P) in enumerate(reqs):
        _assert_request(res, b, oracle.tree_accept(lg, tok, par, P))


@pytest.mark.parametrize("seed", range(6))
def test_batched_accept_small_alphabet(seed):
    # duplicate sibling tokens and many ties: the lowest-index rules per request
    rng = np.random.default_rng(seed)
    ns = [int(x) for x in rng.integers(1, 129, int(rng.integers(2, 17)))]
    reqs = []
    for n in ns:
        parent = synth.random_parent_tree(rng, n, max_depth=12)
        token = rng.integers(0, 3, size=n).astype(np.int32)
        logits = np.round(rng.standard_normal((n, 3)), 0).astype(np.float32)
        reqs.append((parent, token, logits, int(rng.integers(0, 5000))))
    parent, token, logits = _packed(reqs)
    res = tvp.tree_accept_batched(logits, token, parent, ns, [r[3] for r in reqs])
    torch.cuda.synchronize()
    for b, (par, tok, lg, P) in enumerate(reqs):
        _assert_request(res, b, oracle.tree_accept(lg, tok, par, P))


def test_batched_accept_tokens_matches_oracle():
    rng = np.random.default_rng(11)
    ns = [64, 17, 128, 5, 64, 1, 90, 33]
    reqs = _requests(rng, ns, 32000)
    parent, token, logits = _packed(reqs)
    target = torch.from_numpy(np.concatenate([np.argmax(r[2], axis=1).astype(np.int32)
                                              for r in reqs])).to(DEV)
    res = tvp.tree_accept_tokens_batched(target, 32000, token, parent, ns, [r[3] for r in reqs])
    torch.cuda.synchronize()
    for b, (par, tok, lg, P) in enumerate(reqs):
        _assert_request(res, b, oracle.tree_accept(lg, tok, par, P))


def test_bad_request_is_reported_and_isolated():
    rng = np.random.default_rng(4)
    ns = [20, 12, 30]
    reqs = _requests(rng, ns, 500)
    bad = reqs[1][0].copy()
    bad[5] = 7                                   # parent after the node: not a tree
    reqs[1] = (bad,) + reqs[1][1:]
    parent, token, logits = _packed(reqs)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    res = tvp.tree_accept_batched(logits, token, parent, ns, [r[3] for r in reqs], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == tvp.TV_ERR_INVALID_TREE
    got = tvp.batched_request(res, 1)
    assert int(got["m"].item()) == 0 and int(got["n_survivors"].item()) == 0
    assert (got["new_pos"] == -1).all() and (got["out_tokens"] == -1).all()
    for b in (0, 2):
        par, tok, lg, P = reqs[b]
        _assert_request(res, b, oracle.tree_accept(lg, tok, par, P))


@pytest.mark.parametrize("seed", range(3))
def test_batched_sampling_equals_single_calls_and_oracle(seed):
    # every request has its own temperature, seed and offset; its draws and
    # walk must be exactly those of the single-request call with them, and
    # the draws the oracle's wherever the uniform is not within 1e-5 of a
    # cumulative-probability boundary
    rng = np.random.default_rng(70 + seed)
    ns = [[64, 1, 17], [int(x) for x in rng.integers(1, 129, 16)], [128, 64]][seed]
    vocab = [128256, 1000, 33][seed]
    reqs = []
    for n in ns:
        parent = np.asarray(synth.uniform_parent_tree(rng, n, max_depth=8, max_fanout=8),
                            dtype=np.int32)
        token = rng.integers(0, vocab, size=n).astype(np.int32)
        logits = (rng.standard_normal((n, vocab)) * 3).astype(np.float32)
        reqs.append((parent, token, logits, int(rng.integers(0, 5000))))
    temps = [float(t) for t in rng.uniform(0.3, 2.0, len(ns))]
    seeds = [int(x) for x in rng.integers(0, 2**63, len(ns))]
    offs = [int(x) for x in rng.integers(0, 1000, len(ns))]
    parent, token, logits = _packed(reqs)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    res = tvp.tree_accept_sampled_batched(logits, token, parent, ns, [r[3] for r in reqs], temps,
                                          seeds, offs, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for b, (par, tok, lg, P) in enumerate(reqs):
        one = tvp.tree_accept_sampled(torch.from_numpy(lg).to(DEV), torch.from_numpy(tok).to(DEV),
                                      torch.from_numpy(par).to(DEV), P, temps[b], seeds[b],
                                      offs[b])
        got = tvp.batched_request(res, b)
        torch.cuda.synchronize()
        for key in ("sampled", "m", "path", "out_tokens", "new_pos", "new_parent",
                    "n_survivors"):
            assert torch.equal(got[key], one[key]), (b, key)
        s = got["sampled"].cpu().numpy()
        p = oracle.target_probs(lg.astype(np.float64), temps[b])
        for i in range(len(par)):
            u = oracle.node_uniform(seeds[b], offs[b], i)
            want = oracle.draw_by_inversion(p[i], u)
            g = int(s[i])
            if g != want:
                c = np.cumsum(p[i])
                lo = c[g - 1] if g > 0 else 0.0
                assert lo - 1e-5 <= u < c[g] + 1e-5, (b, i, g, want)


def _bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32).cpu().numpy()


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64)])
@pytest.mark.parametrize("seed", range(3))
def test_batched_compaction_matches_oracle(dtype, d, seed):
    rng = np.random.default_rng(50 + seed)
    ns = [[64, 1, 128, 9], [int(x) for x in rng.integers(1, 129, 16)], [33, 64]][seed]
    layers, hkv = 3, 2
    reqs = [(p, t, lg, int(rng.integers(0, 3000))) for p, t, lg, _ in _requests(rng, ns, 300)]
    parent, token, logits = _packed(reqs)
    acc = tvp.tree_accept_batched(logits, token, parent, ns, [r[3] for r in reqs])
    caps = [r[3] + n + int(rng.integers(0, 20)) for r, n in zip(reqs, ns)]
    ks = [torch.from_numpy(rng.standard_normal((layers, hkv, c, d), dtype=np.float32)).to(dtype)
          for c in caps]
    vs = [torch.from_numpy(rng.standard_normal((layers, hkv, c, d), dtype=np.float32)).to(dtype)
          for c in caps]
    kd, vd = [k.to(DEV) for k in ks], [v.to(DEV) for v in vs]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tvp.kv_compact_batched(kd, vd, [r[3] for r in reqs], ns, acc["new_pos"], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for b, (par, tok, lg, P) in enumerate(reqs):
        new_pos = oracle.tree_accept(lg, tok, par, P)["new_pos"]
        assert np.array_equal(_bits(kd[b]), oracle.kv_compact(_bits(ks[b]), P, new_pos)), b
        assert np.array_equal(_bits(vd[b]), oracle.kv_compact(_bits(vs[b]), P, new_pos)), b


def test_batched_compaction_reports_one_bad_new_pos():
    rng = np.random.default_rng(8)
    n, P, cap, d = 6, 10, 30, 64
    ks = [torch.from_numpy(rng.standard_normal((1, 1, cap, d), dtype=np.float32))
          .to(torch.bfloat16) for _ in range(2)]
    kd = [k.to(DEV) for k in ks]
    vd = [k.clone().to(DEV) for k in ks]
    good = np.array([10, 11, -1, 12, -1, 13], dtype=np.int32)
    bad = np.array([10, 11, 25, 9, 11, -1], dtype=np.int32)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tvp.kv_compact_batched(kd, vd, [P, P], [n, n],
                           [torch.from_numpy(good).to(DEV), torch.from_numpy(bad).to(DEV)],
                           status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == tvp.TV_ERR_INVALID_ARG
    assert np.array_equal(_bits(kd[0]), oracle.kv_compact(_bits(ks[0]), P, good))
    got, ref = _bits(kd[1]), _bits(ks[1])
    assert np.array_equal(got[..., :P, :], ref[..., :P, :])
    assert np.array_equal(got[..., P + n:, :], ref[..., P + n:, :])


def _logical(pool, table):
    """[L, num_pages, Hkv, ps, d] -> [L, Hkv, T * ps, d] in table order."""
    g = pool[:, torch.as_tensor(table, dtype=torch.long)]       # [L, T, Hkv, ps, d]
    g = g.movedim(1, 2)                                         # [L, Hkv, T, ps, d]
    return g.reshape(g.shape[0], g.shape[1], -1, g.shape[-1])


@pytest.mark.parametrize("page_size", [16, 64, 100])
def test_batched_paged_compaction_matches_oracle(page_size):
    rng = np.random.default_rng(page_size)
    ns = [64, 3, 128, 40, 1]
    layers, hkv, d = 2, 4, 128
    reqs = _requests(rng, ns, 200)
    reqs = [(p, t, lg, int(rng.integers(0, 700))) for p, t, lg, _ in reqs]
    parent, token, logits = _packed(reqs)
    acc = tvp.tree_accept_batched(logits, token, parent, ns, [r[3] for r in reqs])
    counts = [-(-(r[3] + n) // page_size) for r, n in zip(reqs, ns)]
    total = sum(counts)
    perm = rng.permutation(total + 6).astype(np.int32)
    tables, at = [], 0
    for c in counts:
        tables.append(perm[at:at + c])
        at += c
    shape = (layers, total + 6, hkv, page_size, d)
    kp = torch.from_numpy(rng.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)
    vp = torch.from_numpy(rng.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)
    kd, vd = kp.to(DEV), vp.to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tvp.kv_compact_batched_paged(kd, vd, [torch.from_numpy(t).to(DEV) for t in tables],
                                 [r[3] for r in reqs], ns, acc["new_pos"], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    bits = lambda t: t.view(torch.int16).cpu()
    for pool, dev_pool in ((kp, kd), (vp, vd)):
        for (par, tok, lg, P), table in zip(reqs, tables):
            new_pos = oracle.tree_accept(lg, tok, par, P)["new_pos"]
            want = oracle.kv_compact(_logical(pool.view(torch.int16), table).numpy(), P, new_pos)
            assert np.array_equal(_logical(bits(dev_pool), table).numpy(), want)
        spare = perm[total:]
        assert torch.equal(bits(dev_pool)[:, spare], pool.view(torch.int16)[:, spare])


def test_batched_verification_step():
    """Eight ragged requests: batched attention, packed acceptance and the
    batched compaction, chained on the device without a host round trip;
    each request checked against the oracle."""
    rng = np.random.default_rng(2024)
    hq, hkv, d, vocab = 64, 8, 128, 128256
    ns = [64, 64, 32, 64, 17, 64, 8, 64]
    prefixes = [1024, 4096, 333, 8000, 64, 2048, 0, 5000]
    reqs = _requests(rng, ns, vocab)
    reqs = [(p, t, lg, P) for (p, t, lg, _), P in zip(reqs, prefixes)]
    f = lambda *s: torch.from_numpy(rng.standard_normal(s, dtype=np.float32)).to(torch.bfloat16)
    qs = [f(n, hq, d) for n in ns]
    ks = [f(hkv, P + n + 4, d) for P, n in zip(prefixes, ns)]
    vs = [f(hkv, P + n + 4, d) for P, n in zip(prefixes, ns)]
    kd, vd = [k.to(DEV) for k in ks], [v.to(DEV) for v in vs]
    parent, token, logits = _packed(reqs)
    pars = [torch.from_numpy(r[0]).to(DEV) for r in reqs]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = tvp.tree_attn_verify_batched([q.to(DEV) for q in qs], kd, vd, prefixes, pars,
                                        status=st)
    acc = tvp.tree_accept_batched(logits, token, parent, ns, prefixes, status=st)
    tvp.kv_compact_batched(kd, vd, prefixes, ns, acc["new_pos"], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for b, (par, tok, lg, P) in enumerate(reqs):
        nodes = sorted({0, ns[b] // 2, ns[b] - 1})
        ref = oracle.tree_attention(qs[b].float().numpy(), ks[b].float().numpy(),
                                    vs[b].float().numpy(), P, par, nodes=nodes)
        assert float(np.abs(outs[b].float().cpu().numpy()[nodes] - ref).max()) <= BF16_TOL
        want = oracle.tree_accept(lg, tok, par, P)
        _assert_request(acc, b, want)
        assert np.array_equal(_bits(kd[b]), oracle.kv_compact(_bits(ks[b]), P, want["new_pos"]))
        assert np.array_equal(_bits(vd[b]), oracle.kv_compact(_bits(vs[b]), P, want["new_pos"]))
