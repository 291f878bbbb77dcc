"""The checked build on the GPU.  The same sources compiled with -DTV_CHECKED=1
test the index ranges of their guarded accesses and record TV_ERR_BOUNDS
instead of touching memory out of range.  Run on valid inputs across the
product's launch shapes (the full-step attention with two tiles per CTA, a
short tree with one tile and double-buffered scores, a batch of requests,
paged K/V, greedy and sampled acceptance, compaction, expansion), no guard
may fire and every output must equal the normal build's bit for bit: the
guards only test indices, they change no arithmetic."""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_tree_masked_gb300 import _build, _lib
from workloads import synth

tvp = pytest.importorskip("speculative_decoding_tree_masked_gb300")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def checked(tmp_path_factory):
    d = tmp_path_factory.mktemp("checked")
    path = _build.build(extra_flags=["-DTV_CHECKED=1"], build_dir=str(d / "objs"),
                        lib_path=str(d / "libtreeverify_checked.so"))
    lib = ctypes.CDLL(path)
    for name, (res, args) in _lib.SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    assert lib.tv_checked_build() == 1
    return lib


def _both(checked, run):
    """run(status) under the normal library, then under the checked one;
    returns both results and both device status words."""
    normal = _lib.load()
    assert normal.tv_checked_build() == 0
    out = []
    for lib in (normal, checked):
        saved = _lib._lib
        _lib._lib = lib
        try:
            st = torch.zeros(1, dtype=torch.int32, device=DEV)
            res = run(st)
            torch.cuda.synchronize()
            out.append((res, int(st.item())))
        finally:
            _lib._lib = saved
    return out


def _same(a, b):
    if isinstance(a, dict):
        return a.keys() == b.keys() and all(_same(a[k], b[k]) for k in a)
    if isinstance(a, (list, tuple)):
        return len(a) == len(b) and all(_same(x, y) for x, y in zip(a, b))
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b)


def _qkv(rng, n, hq, hkv, d, cap):
    q = torch.from_numpy(rng.standard_normal((n, hq, d), dtype=np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(rng.standard_normal((hkv, cap, d), dtype=np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((hkv, cap, d), dtype=np.float32)).to(torch.bfloat16)
    return q.to(DEV), k.to(DEV), v.to(DEV)


@pytest.mark.parametrize("prefix,n", [(4096, 64), (8192, 8), (1000, 33), (0, 1)])
def test_checked_attention(checked, prefix, n):
    rng = np.random.default_rng(prefix + n)
    parent = torch.from_numpy(synth.random_parent_tree(rng, n, max_depth=8)).to(DEV)
    q, k, v = _qkv(rng, n, 64, 8, 128, prefix + n)
    (a, sa), (b, sb) = _both(checked, lambda st: tvp.tree_attn_verify(q, k, v, prefix, parent,
                                                                       status=st))
    assert sa == 0 and sb == 0
    assert _same(a, b)


def test_checked_batched_and_paged_attention(checked):
    rng = np.random.default_rng(11)
    prefixes, ns = [1024, 4096, 333], [64, 17, 8]
    qs, ks, vs, pars = [], [], [], []
    for p, n in zip(prefixes, ns):
        q, k, v = _qkv(rng, n, 64, 8, 128, p + n)
        qs.append(q)
        ks.append(k)
        vs.append(v)
        pars.append(torch.from_numpy(synth.random_parent_tree(rng, n, max_depth=8)).to(DEV))
    (a, sa), (b, sb) = _both(checked, lambda st: tvp.tree_attn_verify_batched(
        qs, ks, vs, prefixes, pars, status=st))
    assert sa == 0 and sb == 0
    assert _same(a, b)
    # one request's cache in shuffled 64-row pages of a pool
    prefix, n, ps = 4096, 64, 64
    t = -(-(prefix + n) // ps)
    pool_k = torch.from_numpy(rng.standard_normal((t + 3, 8, ps, 128), dtype=np.float32)).to(
        torch.bfloat16).to(DEV)
    pool_v = torch.from_numpy(rng.standard_normal((t + 3, 8, ps, 128), dtype=np.float32)).to(
        torch.bfloat16).to(DEV)
    table = torch.from_numpy(rng.permutation(t + 3)[:t].astype(np.int32)).to(DEV)
    q = qs[0].new_empty((n, 64, 128)).copy_(
        torch.from_numpy(rng.standard_normal((n, 64, 128), dtype=np.float32)))
    par = pars[0]
    (a, sa), (b, sb) = _both(checked, lambda st: tvp.tree_attn_verify_paged(
        q, pool_k, pool_v, table, prefix, par, status=st))
    assert sa == 0 and sb == 0
    assert _same(a, b)


def test_checked_acceptance_compaction_and_expansion(checked):
    w = synth.make_workload("l3_8b", seed=5)
    logits = torch.from_numpy(w.logits).to(DEV)
    token = torch.from_numpy(w.token).to(DEV)
    parent = torch.from_numpy(w.parent).to(DEV)
    n = w.n
    (a, sa), (b, sb) = _both(checked, lambda st: tvp.tree_accept(logits, token, parent, w.prefix,
                                                                 status=st))
    assert sa == 0 and sb == 0
    assert _same(a, b)
    (a2, sa), (b2, sb) = _both(checked, lambda st: tvp.tree_accept_sampled(
        logits, token, parent, w.prefix, 1.0, 1234, 7, status=st))
    assert sa == 0 and sb == 0
    assert _same(a2, b2)
    new_pos = a["new_pos"]
    rng = np.random.default_rng(5)
    k0 = torch.from_numpy(rng.standard_normal((2, 8, w.prefix + n, 128), dtype=np.float32)).to(
        torch.bfloat16).to(DEV)
    v0 = torch.from_numpy(rng.standard_normal((2, 8, w.prefix + n, 128), dtype=np.float32)).to(
        torch.bfloat16).to(DEV)

    def compact(st):
        k, v = k0.clone(), v0.clone()
        tvp.kv_compact(k, v, w.prefix, n, new_pos, status=st)
        return k, v

    (a3, sa), (b3, sb) = _both(checked, compact)
    assert sa == 0 and sb == 0
    assert _same(a3, b3)
    frontier = torch.arange(8, dtype=torch.int32, device=DEV)
    cum = torch.from_numpy(rng.standard_normal(n).astype(np.float32)).to(DEV)
    rows = logits[:8].contiguous()
    (a4, sa), (b4, sb) = _both(checked, lambda st: tvp.tree_expand(rows, frontier, cum, 8,
                                                                   status=st))
    assert sa == 0 and sb == 0
    assert _same(a4, b4)
