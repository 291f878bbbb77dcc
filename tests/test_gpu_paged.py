"""Paged K/V caches through the C ABI.  A page pool holds the rows of every
request in shuffled pages; the logical cache of a request is its pages
gathered in table order.  Paged attention must equal the contiguous kernel
on that logical cache bit for bit (the same plan and arithmetic; rows past
P + N hold large finite values and are weighted by exactly zero) and the
oracle within 2e-2; paged compaction must move the logical rows exactly as
the oracle's compaction does and touch nothing else."""
import numpy as np
import pytest
import torch

import oracle
from workloads import synth

tvp = pytest.importorskip("speculative_decoding_tree_masked_gb300")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
BF16_TOL = 2e-2


def _pool_case(seed, prefix, n, hkv, d, page_size, spare_pages=5, layers=None):
    """Random K and V pools (CPU, bf16) holding one request's logical cache
    [Hkv][T * page_size][d] in shuffled pages among spare ones, and the
    request's page table."""
    rng = np.random.default_rng(seed)
    t = -(-(prefix + n) // page_size)
    num_pages = t + spare_pages
    shape = (num_pages, hkv, page_size, d) if layers is None else \
        (layers, num_pages, hkv, page_size, d)
    kp = torch.from_numpy(rng.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)
    vp = torch.from_numpy(rng.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)
    table = rng.permutation(num_pages)[:t].astype(np.int32)
    # rows of the request's last page past P + N: large but finite
    last, tail = table[-1], (prefix + n) - (t - 1) * page_size
    if tail < page_size:
        kp[..., last, :, tail:, :] = 3.0e4
        vp[..., last, :, tail:, :] = -3.0e4
    return kp, vp, table


def _logical(pool, table):
    """[..., num_pages, Hkv, ps, d] -> [..., Hkv, T * ps, d] in table order."""
    g = pool[..., torch.as_tensor(table, dtype=torch.long), :, :, :]
    g = g.movedim(-4, -3)                       # [..., Hkv, T, ps, d]
    return g.reshape(*g.shape[:-3], g.shape[-3] * g.shape[-2], g.shape[-1])


@pytest.mark.parametrize("prefix,n,page_size,d", [
    (4096, 64, 64, 128), (4096, 64, 128, 128), (1000, 15, 64, 64), (8192, 64, 256, 128),
    (0, 1, 64, 128), (32768, 8, 64, 128), (2047, 128, 192, 64), (300, 33, 64, 128)])
def test_paged_attention_equals_contiguous_and_oracle(prefix, n, page_size, d):
    hq, hkv = 64, 8
    rng = np.random.default_rng(prefix + n)
    parent = np.asarray(synth.uniform_parent_tree(rng, n, max_depth=8, max_fanout=8),
                        dtype=np.int32)
    kp, vp, table = _pool_case(7, prefix, n, hkv, d, page_size)
    q = torch.from_numpy(rng.standard_normal((n, hq, d), dtype=np.float32)).to(torch.bfloat16)
    par = torch.from_numpy(parent).to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = tvp.tree_attn_verify_paged(q.to(DEV), kp.to(DEV), vp.to(DEV),
                                     torch.from_numpy(table).to(DEV), prefix, par, status=st)
    kl, vl = _logical(kp, table), _logical(vp, table)
    cont = tvp.tree_attn_verify(q.to(DEV), kl.to(DEV).contiguous(), vl.to(DEV).contiguous(),
                                prefix, par)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(got.view(torch.int16), cont.view(torch.int16))
    nodes = list(range(n)) if n <= 16 else sorted(set([0, n - 1] + list(rng.choice(n, 6))))
    ref = oracle.tree_attention(q.float().numpy(), kl.float().numpy(), vl.float().numpy(),
                                prefix, parent, nodes=nodes)
    assert float(np.abs(got.float().cpu().numpy()[nodes] - ref).max()) <= BF16_TOL


def test_batched_paged_equals_batched_contiguous():
    hq, hkv, d, page_size = 64, 8, 128, 64
    rng = np.random.default_rng(3)
    prefixes = [1024, 4096, 333, 8000, 64]
    ns = [64, 32, 17, 64, 8]
    # one pool holding every request's pages, shuffled together
    tables, total = [], 0
    for p, n in zip(prefixes, ns):
        t = -(-(p + n) // page_size)
        tables.append(np.arange(total, total + t))
        total += t
    perm = rng.permutation(total + 7).astype(np.int32)
    tables = [perm[t] for t in tables]
    shape = (total + 7, hkv, page_size, d)
    kp = torch.from_numpy(rng.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)
    vp = torch.from_numpy(rng.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)
    qs, pars = [], []
    for n in ns:
        qs.append(torch.from_numpy(rng.standard_normal((n, hq, d), dtype=np.float32))
                  .to(torch.bfloat16).to(DEV))
        pars.append(torch.from_numpy(np.asarray(
            synth.uniform_parent_tree(rng, n, max_depth=8, max_fanout=8), dtype=np.int32)).to(DEV))
    kpd, vpd = kp.to(DEV), vp.to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = tvp.tree_attn_verify_batched_paged(qs, kpd, vpd,
                                             [torch.from_numpy(t).to(DEV) for t in tables],
                                             prefixes, pars, status=st)
    kls = [_logical(kp, t).to(DEV).contiguous() for t in tables]
    vls = [_logical(vp, t).to(DEV).contiguous() for t in tables]
    want = tvp.tree_attn_verify_batched(qs, kls, vls, prefixes, pars)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for g, w in zip(got, want):
        assert torch.equal(g.view(torch.int16), w.view(torch.int16))


def test_bad_page_entry_is_reported():
    prefix, n, hkv, d, page_size = 500, 16, 8, 128, 64
    kp, vp, table = _pool_case(1, prefix, n, hkv, d, page_size)
    table = table.copy()
    table[2] = kp.shape[0] + 3                  # outside the pool
    q = torch.zeros((n, 64, d), dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tvp.tree_attn_verify_paged(q, kp.to(DEV), vp.to(DEV), torch.from_numpy(table).to(DEV),
                               prefix, torch.from_numpy(synth.chain_tree(n).astype(np.int32))
                               .to(DEV), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == tvp.TV_ERR_INVALID_ARG


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("page_size", [16, 64, 100])
def test_paged_compaction_matches_oracle(seed, page_size):
    layers, hkv, d, prefix, n = 3, 4, 128, 250 + seed * 37, 64
    rng = np.random.default_rng(seed)
    parent = np.asarray(synth.uniform_parent_tree(rng, n, max_depth=8, max_fanout=8),
                        dtype=np.int32)
    token = np.asarray(synth.draft_tokens(rng, parent, 50), dtype=np.int32)
    depth = synth.node_depths(parent)
    logits, _ = synth.planted_logits(rng, parent, token, 50, int(rng.integers(0, depth.max() + 1)))
    acc = oracle.tree_accept(logits, token, parent, prefix)
    kp, vp, table = _pool_case(seed, prefix, n, hkv, d, page_size, layers=layers)
    kd, vd = kp.to(DEV), vp.to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    new_pos = torch.from_numpy(acc["new_pos"].astype(np.int32)).to(DEV)
    tvp.kv_compact_paged(kd, vd, torch.from_numpy(table).to(DEV), prefix, n, new_pos, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    bits = lambda t: t.view(torch.int16).cpu()
    for pool, dev_pool in ((kp, kd), (vp, vd)):
        want = oracle.kv_compact(_logical(pool, table).view(torch.int16).numpy(), prefix,
                                 acc["new_pos"])
        assert np.array_equal(_logical(bits(dev_pool), table).numpy(), want)
        # pages outside the table are untouched
        spare = np.setdiff1d(np.arange(pool.shape[1]), table)
        assert torch.equal(bits(dev_pool)[:, spare], pool.view(torch.int16)[:, spare])


def test_paged_compaction_skips_rows_of_bad_pages():
    layers, hkv, d, prefix, n, page_size = 1, 2, 64, 60, 8, 16
    kp, vp, table = _pool_case(0, prefix, n, hkv, d, page_size, layers=layers)
    table = table.copy()
    table[-1] = -5                               # the page of rows 64..67
    new_pos = torch.tensor([60, 61, -1, -1, 62, -1, -1, 63], dtype=torch.int32, device=DEV)
    kd, vd = kp.to(DEV), vp.to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tvp.kv_compact_paged(kd, vd, torch.from_numpy(table).to(DEV), prefix, n, new_pos, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == tvp.TV_ERR_INVALID_ARG
    # node 7 (row 67, on the bad page) did not move; node 4 (row 64) neither
    kl = _logical(kd.cpu(), table[:-1])
    assert torch.equal(kl[0, :, 63].view(torch.int16),
                       _logical(kp, table[:-1])[0, :, 63].view(torch.int16))
