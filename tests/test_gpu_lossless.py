"""Losslessness through the CUDA library: speculative decoding of a toy
one-layer target (tests/toy_target.py) with the GPU's tree attention,
acceptance (the argmax kernel on fp32 logits, or the fused LM-head argmax
on bf16 hidden states) and in-place KV compaction emits exactly the tokens
of the target's own autoregressive greedy decode in fp64 on the CPU.

Every emitted token is decided on the accepted path, whose contexts are the
true ones, so a decision can differ from the fp64 one only where the GPU's
rounding reaches the margin between the two best logits.  The fp32 path errs
by ~1e-6, far below every margin here (checked).  For the bf16 path the
seeds are chosen, deterministically, among those whose smallest margin is at
least five times the largest logit deviation of a bf16 simulation of the
same decode (Q, K, V, the unnormalised softmax weights, the attention
output, the hidden state and the LM head rounded to bf16), so a flipped
decision means a wrong kernel, not rounding."""
import numpy as np
import pytest
import torch

from tests.toy_target import ToyTarget, draft_tree

tvp = pytest.importorskip("speculative_decoding_tree_masked_gb300")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
N_NEW = 24


def _bf(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def _bf16_deviation(model, prompt, reference):
    """Largest |logit| deviation of a bf16 simulation along the reference."""
    toks = list(prompt) + list(reference)
    x = model.embed(toks, range(len(toks)))
    q, k, v = model.qkv(x)
    qb, kb, vb = _bf(q), _bf(k), _bf(v)
    g, sc = model.hq // model.hkv, 1.0 / np.sqrt(model.dh)
    worst = 0.0
    for p in range(len(prompt) - 1, len(toks) - 1):
        ob, oe = np.zeros((model.hq, model.dh)), np.zeros((model.hq, model.dh))
        for h in range(model.hq):
            s = kb[:p + 1, h // g] @ qb[p, h] * sc
            e = np.exp(s - s.max())
            ob[h] = (_bf(e) @ vb[:p + 1, h // g]) / e.sum()
            s = k[:p + 1, h // g] @ q[p, h] * sc
            e = np.exp(s - s.max())
            oe[h] = (e @ v[:p + 1, h // g]) / e.sum()
        zb = _bf(model.hidden(x[p:p + 1], _bf(ob)[None])) @ _bf(model.Wlm).T
        ze = model.hidden(x[p:p + 1], oe[None]) @ model.Wlm.T
        worst = max(worst, float(np.abs(zb - ze).max()))
    return worst


def _case(seed):
    model = ToyTarget(seed, dh=64)
    rng = np.random.default_rng(100 + seed)
    prompt = [int(t) for t in rng.integers(model.vocab, size=20)]
    reference, margins = model.greedy_decode(prompt, N_NEW)
    return model, prompt, reference, margins, rng


def _robust_bf16_seeds(count=3, ratio=5.0, limit=300):
    seeds = []
    for seed in range(limit):
        model, prompt, reference, margins, _ = _case(seed)
        if min(margins) >= ratio * _bf16_deviation(model, prompt, reference):
            seeds.append(seed)
            if len(seeds) == count:
                break
    assert len(seeds) == count
    return seeds


def gpu_speculative_decode(model, prompt, reference, rng, n_nodes, plant, bf16):
    dt = torch.bfloat16 if bf16 else torch.float32
    P = len(prompt) - 1
    cap = len(prompt) + N_NEW + n_nodes + 4
    K = torch.zeros((1, model.hkv, cap, model.dh), dtype=dt, device=DEV)
    V = torch.zeros_like(K)
    _, k, v = model.qkv(model.embed(prompt[:-1], range(P)))
    K[0, :, :P] = torch.from_numpy(k.transpose(1, 0, 2).copy()).to(DEV, dt)
    V[0, :, :P] = torch.from_numpy(v.transpose(1, 0, 2).copy()).to(DEV, dt)
    wo = torch.from_numpy(model.Wo).to(DEV, torch.float32)
    wlm = torch.from_numpy(model.Wlm).to(DEV, torch.float32)
    wlm_bf = wlm.to(torch.bfloat16).contiguous()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    root, emitted, accepted = int(prompt[-1]), [], []
    while len(emitted) < N_NEW:
        parent, token, depth = draft_tree(rng, root, reference[len(emitted):], model.vocab,
                                          n_nodes, plant)
        n = len(parent)
        x = model.embed(token, P + depth)
        q, k, v = model.qkv(x)
        K[0, :, P:P + n] = torch.from_numpy(k.transpose(1, 0, 2).copy()).to(DEV, dt)
        V[0, :, P:P + n] = torch.from_numpy(v.transpose(1, 0, 2).copy()).to(DEV, dt)
        par = torch.from_numpy(parent).to(DEV)
        tok = torch.from_numpy(token).to(DEV)
        o = tvp.tree_attn_verify(torch.from_numpy(q).to(DEV, dt).contiguous(), K[0], V[0], P,
                                 par, status=status)
        h = torch.from_numpy(x).to(DEV, torch.float32) + o.float().reshape(n, -1) @ wo
        if bf16:
            res = tvp.lm_head_argmax(h.to(torch.bfloat16).contiguous(), wlm_bf, status=status)
            acc = tvp.tree_accept_tokens(res["am"], model.vocab, tok, par, P, status=status)
        else:
            acc = tvp.tree_accept((h @ wlm.T).contiguous(), tok, par, P, status=status)
        m = int(acc["m"].item())
        emitted += [int(t) for t in acc["out_tokens"][:m + 1].tolist()]
        accepted.append(m)
        tvp.kv_compact(K, V, P, n, acc["new_pos"], status=status)
        P += m + 1
        root = emitted[-1]
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return emitted[:N_NEW], accepted


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("n_nodes,plant", [(1, 0.0), (8, 0.7), (15, 1.0), (64, 0.5)])
def test_fp32_speculative_equals_autoregressive(seed, n_nodes, plant):
    model, prompt, reference, margins, rng = _case(seed)
    assert min(margins) > 1e-4
    got, accepted = gpu_speculative_decode(model, prompt, reference, rng, n_nodes, plant,
                                           bf16=False)
    assert got == reference
    if plant == 1.0:
        assert max(accepted) >= 10


_BF16_SEEDS = None


@pytest.mark.parametrize("which", range(3))
@pytest.mark.parametrize("n_nodes,plant", [(8, 0.7), (15, 1.0), (64, 0.5)])
def test_bf16_speculative_equals_autoregressive(which, n_nodes, plant):
    global _BF16_SEEDS
    if _BF16_SEEDS is None:
        _BF16_SEEDS = _robust_bf16_seeds()
    model, prompt, reference, _, rng = _case(_BF16_SEEDS[which])
    got, _ = gpu_speculative_decode(model, prompt, reference, rng, n_nodes, plant, bf16=True)
    assert got == reference
