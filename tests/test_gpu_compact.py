"""GPU parity of in-place KV compaction (through the C ABI) against the
oracle's out-of-place copy, byte for byte, with canary rows around the tree
region; plus the full verify step (attention, acceptance, compaction of
every layer) and the re-rooting invariant on the GPU."""
import numpy as np
import pytest
import torch

import oracle
from workloads import synth

tvp = pytest.importorskip("speculative_decoding_tree_masked_gb300")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32).cpu().numpy()


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.bfloat16, 64),
                                     (torch.float32, 128), (torch.float32, 64)])
@pytest.mark.parametrize("seed", range(4))
def test_compaction_matches_oracle(dtype, d, seed):
    rng = np.random.default_rng(seed)
    n = [5, 33, 64, 128][seed]
    P, L, hkv = 50 + seed, 3, 2
    cap = P + n + 7
    parent = synth.random_parent_tree(rng, n, max_depth=10)
    token = rng.integers(0, 4, size=n).astype(np.int32)
    logits = rng.standard_normal((n, 4)).astype(np.float32)
    want = oracle.tree_accept(logits, token, parent, P)
    k = torch.from_numpy(rng.standard_normal((L, hkv, cap, d), dtype=np.float32)).to(dtype)
    v = torch.from_numpy(rng.standard_normal((L, hkv, cap, d), dtype=np.float32)).to(dtype)
    kd, vd = k.to(DEV), v.to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tvp.kv_compact(kd, vd, P, n, torch.from_numpy(want["new_pos"]).to(DEV), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(_bits(kd), oracle.kv_compact(_bits(k), P, want["new_pos"]))
    assert np.array_equal(_bits(vd), oracle.kv_compact(_bits(v), P, want["new_pos"]))


def test_invalid_new_pos_is_reported_and_nothing_outside_is_written():
    rng = np.random.default_rng(0)
    n, P, cap, d = 6, 10, 30, 64
    k = torch.from_numpy(rng.standard_normal((1, 1, cap, d), dtype=np.float32)).to(torch.bfloat16)
    kd, vd = k.to(DEV), k.clone().to(DEV)
    bad = torch.tensor([10, 11, 25, 9, 11, -1], dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tvp.kv_compact(kd, vd, P, n, bad, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == tvp.TV_ERR_INVALID_ARG
    got = _bits(kd)
    ref = _bits(k)
    assert np.array_equal(got[..., :P, :], ref[..., :P, :])
    assert np.array_equal(got[..., P + n:, :], ref[..., P + n:, :])


def test_full_verify_step_all_layers():
    # the benchmark's step at 8 layers: attention every layer, accept, compact
    w = synth.make_workload("full_step", seed=4, layers=8)
    q, k, v = synth.make_qkv(w)
    kd, vd = k.to(DEV), v.to(DEV)
    parent = torch.from_numpy(w.parent).to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    nodes = [0, 17, 63]
    for layer in range(w.layers):
        out = tvp.tree_attn_verify(q[layer].to(DEV), kd[layer], vd[layer], w.prefix, parent,
                                   status=st)
        if layer in (0, w.layers - 1):
            ref = oracle.tree_attention(q[layer].float().numpy(), k[layer].float().numpy(),
                                        v[layer].float().numpy(), w.prefix, w.parent, nodes=nodes)
            assert float(np.abs(out.float().cpu().numpy()[nodes] - ref).max()) <= 2e-2
    res = tvp.tree_accept(torch.from_numpy(w.logits).to(DEV), torch.from_numpy(w.token).to(DEV),
                          parent, w.prefix, status=st)
    tvp.kv_compact(kd, vd, w.prefix, w.n, res["new_pos"], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    want = oracle.tree_accept(w.logits, w.token, w.parent, w.prefix)
    assert int(res["m"].item()) == want["m"] == len(w.planted_path) - 1
    assert np.array_equal(res["out_tokens"].cpu().numpy(), want["out_tokens"])
    assert np.array_equal(_bits(kd), oracle.kv_compact(_bits(k), w.prefix, want["new_pos"]))
    assert np.array_equal(_bits(vd), oracle.kv_compact(_bits(v), w.prefix, want["new_pos"]))


@pytest.mark.parametrize("seed", range(6))
def test_reroot_preserves_survivor_attention_on_gpu(seed):
    rng = np.random.default_rng(seed)
    n, P, hq, hkv, d = 64, 300, 8, 2, 128
    while True:  # draw until some subtree survives
        parent = synth.random_parent_tree(rng, n, max_depth=10)
        token = rng.integers(0, 2, size=n).astype(np.int32)
        logits = rng.standard_normal((n, 2)).astype(np.float32)
        want = oracle.tree_accept(logits, token, parent, P)
        m, r = want["m"], want["n_survivors"]
        if r > 0:
            break
    f = lambda *s: torch.from_numpy(rng.standard_normal(s, dtype=np.float32)).to(torch.bfloat16)
    q, k, v = f(n, hq, d), f(hkv, P + n, d), f(hkv, P + n, d)
    kd, vd = k.to(DEV), v.to(DEV)
    before = tvp.tree_attn_verify(q.to(DEV), kd, vd, P, torch.from_numpy(parent).to(DEV)).cpu()
    tvp.kv_compact(kd, vd, P, n, torch.from_numpy(want["new_pos"]).to(DEV))
    surv = [i for i in range(n) if want["new_pos"][i] >= P + m + 1]
    after = tvp.tree_attn_verify(q[surv].contiguous().to(DEV), kd, vd, P + m + 1,
                                 torch.from_numpy(want["new_parent"][:r].copy()).to(DEV)).cpu()
    assert float((after.float() - before[surv].float()).abs().max()) <= 2e-2
