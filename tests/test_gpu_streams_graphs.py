"""Streams and graphs.  The library keeps no state between calls other than
the static-scratch entry point's array (tested on its own), so calls on
different streams with their own workspaces run independently: issued on two
streams at once they must give exactly what they give one after the other.
Every kernel is launched under programmatic serialization, so the batched
attention and the batched acceptance are also captured into a CUDA graph and
replayed, and must give exactly the eager results."""
import numpy as np
import pytest
import torch

from workloads import synth

tvp = pytest.importorskip("speculative_decoding_tree_masked_gb300")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _layer(rng, n, P, hq=64, hkv=8, d=128):
    f = lambda *s: torch.from_numpy(rng.standard_normal(s, dtype=np.float32)).to(
        torch.bfloat16).to(DEV)
    parent = torch.from_numpy(synth.random_parent_tree(rng, n, max_depth=8)).to(DEV)
    return f(n, hq, d), f(hkv, P + n, d), f(hkv, P + n, d), parent


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


def test_two_streams_equal_sequential():
    rng = np.random.default_rng(41)
    cases = [(64, 4096), (8, 16384)]          # two tiles per CTA; one tile, 19 splits
    layers = [_layer(rng, n, P) for n, P in cases]
    ws = [tvp.attn_workspace(n, 64, 8, 128, torch.bfloat16, P, DEV) for n, P in cases]
    st = [torch.zeros(1, dtype=torch.int32, device=DEV) for _ in cases]
    seq = [tvp.tree_attn_verify(q, k, v, P, par, workspace=w, status=s)
           for (q, k, v, par), (n, P), w, s in zip(layers, cases, ws, st)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(DEV) for _ in cases]
    outs = [torch.empty_like(q) for q, _, _, _ in layers]
    for _ in range(3):
        for (q, k, v, par), (n, P), w, s, o, strm in zip(layers, cases, ws, st, outs, streams):
            with torch.cuda.stream(strm):
                tvp.tree_attn_verify(q, k, v, P, par, out=o, workspace=w, status=s, stream=strm)
        torch.cuda.synchronize()
        for a, b in zip(seq, outs):
            assert torch.equal(_bits(a), _bits(b))
    assert all(int(s.item()) == 0 for s in st)


def test_batched_attention_and_acceptance_in_a_graph():
    rng = np.random.default_rng(43)
    shapes = [(64, 2048), (17, 300), (64, 8000)]
    reqs = [_layer(rng, n, P) for n, P in shapes]
    qs, ks, vs, pars = ([r[i] for r in reqs] for i in range(4))
    prefixes = [P for _, P in shapes]
    ns = [n for n, _ in shapes]
    total, vocab = sum(ns), 4096
    logits = torch.from_numpy(rng.standard_normal((total, vocab), dtype=np.float32)).to(DEV)
    token = torch.from_numpy(rng.integers(0, vocab, size=total).astype(np.int32)).to(DEV)
    parent = torch.cat(pars)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    eager_att = tvp.tree_attn_verify_batched(qs, ks, vs, prefixes, pars, status=st)
    eager_acc = tvp.tree_accept_batched(logits, token, parent, ns, prefixes, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    outs = [torch.empty_like(q) for q in qs]
    ws = torch.zeros(tvp.attn_batched_workspace_size(ns, 64, 8, 128, torch.bfloat16),
                     dtype=torch.uint8, device=DEV)
    tensors = [k for k, v in eager_acc.items() if isinstance(v, torch.Tensor)]
    acc = {k: torch.empty_like(eager_acc[k]) for k in tensors}
    stream = torch.cuda.Stream(DEV)

    def step():
        tvp.tree_attn_verify_batched(qs, ks, vs, prefixes, pars, outs=outs, workspace=ws,
                                     status=st, stream=stream)
        tvp.tree_accept_batched(logits, token, parent, ns, prefixes, outs=acc, status=st,
                                stream=stream)

    with torch.cuda.stream(stream):
        step()                                # first calls outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for _ in range(2):
        for o in outs:
            o.zero_()
        for k in tensors:
            acc[k].fill_(-7)
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        for a, b in zip(eager_att, outs):
            assert torch.equal(_bits(a), _bits(b))
        for k in tensors:
            assert torch.equal(eager_acc[k], acc[k]), k
