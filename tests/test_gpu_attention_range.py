"""GPU parity of tree-masked attention at large magnitudes, against the fp64
oracle.

The target's mask attention has to give the model's own attention for any
finite bf16 cache (SwiftSpec review page, "What carries the argument"), so
the split-KV path may not narrow the range of what it carries between the
splits and their merge.  These tests scale V far past float16's largest
value (65504), and K so that the exact scores reach about 1e4, at a shape
the planner cuts into several key splits (the full verify step's layer) and
at one it keeps in a single split, and through the batched call whose
partials pass through the workspace.

The bound is relative to the largest |V| of the cache: 2e-2 * max|V|
element-wise (for N(0,1) values this is the 2e-2 of the other tests), and
no output may be inf or NaN."""
import numpy as np
import pytest
import torch

import oracle
from workloads import synth

tvp = pytest.importorskip("speculative_decoding_tree_masked_gb300")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
REL_TOL = 2e-2


def _normal(rng, *shape):
    return torch.from_numpy(rng.standard_normal(shape, dtype=np.float32))


def _integer_qk(rng, n, hq, hkv, d, cap, k_scale):
    """Q and K with entries in {-2..2} (K times a power of two): every score
    is an integer multiple of k_scale below 2^24, so the tensor cores and
    the oracle compute the same scores exactly."""
    q = torch.from_numpy(rng.integers(-2, 3, (n, hq, d)).astype(np.float32))
    k = torch.from_numpy(rng.integers(-2, 3, (hkv, cap, d)).astype(np.float32)) * k_scale
    return q.to(torch.bfloat16), k.to(torch.bfloat16)


def _check(out, q, k, v, P, parent, nodes):
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all(), "inf or NaN in the output"
    ref = oracle.tree_attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), P,
                                parent, nodes=nodes)
    vmax = float(v.float().abs().max())
    err = float(np.abs(got[nodes] - ref).max())
    assert err <= REL_TOL * vmax, f"max error {err:.3e} against max|V| {vmax:.3e}"


# (label, hq, hkv, d, P, n): the full step's layer is cut into 9 key splits
# on a 152-SM GB300; the small one fits one split
SHAPES = [("full_step_layer", 64, 8, 128, 4096, 64), ("one_split", 8, 2, 128, 100, 16)]


def _splits(hq, hkv, d, P, n):
    return tvp.attn_plan(n, hq, hkv, d, torch.bfloat16, P)["splits"]


def test_shapes_cover_one_and_several_splits():
    assert _splits(*SHAPES[0][1:]) > 1
    assert _splits(*SHAPES[1][1:]) == 1


@pytest.mark.parametrize("v_scale", [1e5, 1e30])
@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
def test_large_values(shape, v_scale):
    _, hq, hkv, d, P, n = shape
    rng = np.random.default_rng(31)
    parent = synth.ml_expansion_tree(rng, n) if n == 64 else synth.random_parent_tree(rng, n)
    q = _normal(rng, n, hq, d).to(torch.bfloat16)
    k = _normal(rng, hkv, P + n, d).to(torch.bfloat16)
    v = (_normal(rng, hkv, P + n, d) * v_scale).to(torch.bfloat16)
    out = tvp.tree_attn_verify(q.to(DEV), k.to(DEV), v.to(DEV), P,
                               torch.from_numpy(parent).to(DEV))
    nodes = sorted({0, 1, n // 2, n - 1})
    _check(out, q, k, v, P, parent, nodes)


@pytest.mark.parametrize("v_scale", [1.0, 1e30])
@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
def test_large_scores(shape, v_scale):
    # K entries up to 2 * 4096: |q.k| reaches about 1e5, the scaled scores
    # about 1e4, so the softmax of a row is nearly one-hot and the splits'
    # log-sum-exps differ by thousands
    _, hq, hkv, d, P, n = shape
    rng = np.random.default_rng(47)
    parent = synth.random_parent_tree(rng, n, max_depth=12)
    q, k = _integer_qk(rng, n, hq, hkv, d, P + n, 4096.0)
    v = (_normal(rng, hkv, P + n, d) * v_scale).to(torch.bfloat16)
    scores = torch.einsum("nhd,gkd->nhgk", q[:2].float(), k.float()).abs().max()
    assert float(scores) / np.sqrt(d) > 5e3
    out = tvp.tree_attn_verify(q.to(DEV), k.to(DEV), v.to(DEV), P,
                               torch.from_numpy(parent).to(DEV))
    nodes = sorted({0, 1, n // 2, n - 1})
    _check(out, q, k, v, P, parent, nodes)


def test_batched_large_values_and_scores():
    rng = np.random.default_rng(53)
    hq, hkv, d = 64, 8, 128
    reqs = []
    for n, P, v_scale, big_scores in [(64, 4096, 1e30, False), (16, 2000, 1e5, True),
                                      (40, 700, 1e30, True)]:
        parent = synth.random_parent_tree(rng, n, max_depth=12)
        if big_scores:
            q, k = _integer_qk(rng, n, hq, hkv, d, P + n, 4096.0)
        else:
            q = _normal(rng, n, hq, d).to(torch.bfloat16)
            k = _normal(rng, hkv, P + n, d).to(torch.bfloat16)
        v = (_normal(rng, hkv, P + n, d) * v_scale).to(torch.bfloat16)
        reqs.append((q, k, v, P, parent))
    outs = tvp.tree_attn_verify_batched([r[0].to(DEV) for r in reqs], [r[1].to(DEV) for r in reqs],
                                        [r[2].to(DEV) for r in reqs], [r[3] for r in reqs],
                                        [torch.from_numpy(r[4]).to(DEV) for r in reqs])
    torch.cuda.synchronize()
    for (q, k, v, P, parent), out in zip(reqs, outs):
        n = q.shape[0]
        _check(out, q, k, v, P, parent, sorted({0, n // 2, n - 1}))
