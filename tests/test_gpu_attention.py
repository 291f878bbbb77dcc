"""GPU parity of tree-masked attention (through the C ABI) against the fp64
oracle: every workload shape, random trees of every size class around the
32-node mask words and the 128-key blocks, a sampled full-size layer, the
masking invariant bit for bit, and device-side tree validation."""
import numpy as np
import pytest
import torch

import oracle
from workloads import synth

tvp = pytest.importorskip("speculative_decoding_tree_masked_gb300")

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2   # max-abs, bf16 inputs with fp32 accumulation
F32_TOL = 1e-4    # max-abs, fp32 inputs and fp32 arithmetic

DEV = "cuda:0"


def _run(q, k, v, P, parent, scale=0.0, status=None):
    par = torch.as_tensor(np.asarray(parent, dtype=np.int32)).to(DEV)
    return tvp.tree_attn_verify(q.to(DEV), k.to(DEV), v.to(DEV), P, par, scale=scale,
                                status=status)


def _ref(q, k, v, P, parent, scale=None, nodes=None):
    return oracle.tree_attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), P,
                                 parent, scale=scale, nodes=nodes)


def _err(out, ref, nodes=None):
    got = out.float().cpu().numpy()
    if nodes is not None:
        got = got[nodes]
    return float(np.abs(got - ref).max())


def _qkv(rng, n, hq, hkv, d, cap, dtype):
    f = lambda *s: torch.from_numpy(rng.standard_normal(s, dtype=np.float32)).to(dtype)
    return f(n, hq, d), f(hkv, cap, d), f(hkv, cap, d)


def test_tiny_workload_fp32():
    w = synth.make_workload("tiny", seed=0)
    q, k, v = synth.make_qkv(w, layer=0)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(q, k, v, w.prefix, w.parent, status=st)
    assert _err(out, _ref(q, k, v, w.prefix, w.parent)) <= F32_TOL
    assert int(st.item()) == 0


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_l3_8b_workload(seed):
    w = synth.make_workload("l3_8b", seed=seed, with_logits=False)
    q, k, v = synth.make_qkv(w, layer=0)
    out = _run(q, k, v, w.prefix, w.parent)
    assert _err(out, _ref(q, k, v, w.prefix, w.parent)) <= BF16_TOL


def test_l3_70b_workload_sampled_nodes():
    w = synth.make_workload("l3_70b", seed=0, layers=1)
    q, k, v = synth.make_qkv(w, layer=0)
    out = _run(q, k, v, w.prefix, w.parent)
    nodes = [0, 1, 7, 20, 33, 50, 63]
    assert _err(out, _ref(q, k, v, w.prefix, w.parent, nodes=nodes), nodes) <= BF16_TOL


@pytest.mark.parametrize("n", [1, 2, 3, 15, 31, 32, 33, 64, 127, 128])
def test_random_trees_every_size(n):
    rng = np.random.default_rng(100 + n)
    P = [0, 1, 127, 128, 129, 300][n % 6]
    hq, hkv, d = 8, 2, 128
    parent = synth.random_parent_tree(rng, n, max_depth=16)
    q, k, v = _qkv(rng, n, hq, hkv, d, P + n, torch.bfloat16)
    out = _run(q, k, v, P, parent)
    assert _err(out, _ref(q, k, v, P, parent)) <= BF16_TOL


@pytest.mark.parametrize("hq,hkv,d,dtype", [
    (4, 4, 64, torch.bfloat16), (6, 2, 64, torch.bfloat16), (7, 1, 128, torch.bfloat16),
    (16, 2, 128, torch.bfloat16), (8, 1, 128, torch.float32), (2, 2, 64, torch.float32)])
def test_head_layouts(hq, hkv, d, dtype):
    rng = np.random.default_rng(hq * 100 + hkv * 10 + d)
    n, P = 37, 515
    parent = synth.random_parent_tree(rng, n, max_depth=9)
    q, k, v = _qkv(rng, n, hq, hkv, d, P + n + 5, dtype)
    out = _run(q, k, v, P, parent)
    tol = BF16_TOL if dtype == torch.bfloat16 else F32_TOL
    assert _err(out, _ref(q, k, v, P, parent)) <= tol


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_explicit_scale_and_forest(dtype):
    rng = np.random.default_rng(3)
    n, P, hq, hkv, d = 20, 64, 4, 2, 64
    parent = np.array([-1, 0, 1, -1, 3, 3, 0, -1] + list(range(7, 19)), dtype=np.int32)
    q, k, v = _qkv(rng, n, hq, hkv, d, P + n, dtype)
    out = _run(q, k, v, P, parent, scale=0.05)
    tol = BF16_TOL if dtype == torch.bfloat16 else F32_TOL
    assert _err(out, _ref(q, k, v, P, parent, scale=0.05)) <= tol


def test_full_step_layer_sampled():
    # the benchmark's layer shape: 64/8 heads, d128, P=4096, 64 nodes
    w = synth.make_workload("full_step", seed=1, layers=1)
    q, k, v = synth.make_qkv(w, layer=0)
    out = _run(q, k, v, w.prefix, w.parent)
    nodes = [0, 5, 31, 32, 63]
    assert _err(out, _ref(q, k, v, w.prefix, w.parent, nodes=nodes), nodes) <= BF16_TOL


@pytest.mark.parametrize("P", [1024, 16384])
@pytest.mark.parametrize("n", [8, 128])
def test_sweep_corners_sampled(P, n):
    w = synth.make_workload("q2_72b", seed=P + n, prefix=P, n=n)
    q, k, v = synth.make_qkv(w, layer=0)
    out = _run(q, k, v, w.prefix, w.parent)
    nodes = sorted({0, n // 2, n - 1})
    assert _err(out, _ref(q, k, v, w.prefix, w.parent, nodes=nodes), nodes) <= BF16_TOL


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_masked_rows_do_not_change_the_output_bits(dtype):
    rng = np.random.default_rng(11)
    n, P, hq, hkv, d = 48, 200, 8, 2, 128
    parent = synth.random_parent_tree(rng, n, max_depth=6)
    cap = P + n + 40
    q, k, v = _qkv(rng, n, hq, hkv, d, cap, dtype)
    base = _run(q, k, v, P, parent).cpu()
    target = n - 1
    anc = set(oracle.ancestors_inclusive(parent, target))
    k2, v2 = k.clone(), v.clone()
    for j in range(n):
        if j not in anc:
            k2[:, P + j] *= 1000
            v2[:, P + j] *= -1000
    k2[:, P + n:] = float("nan")   # rows past the tree are never read
    v2[:, P + n:] = float("nan")
    pert = _run(q, k2, v2, P, parent).cpu()
    assert torch.equal(pert[target], base[target])


def test_chain_tree_is_causal_on_gpu():
    rng = np.random.default_rng(4)
    n, P, hq, hkv, d = 40, 77, 8, 8, 64
    q, k, v = _qkv(rng, n, hq, hkv, d, P + n, torch.bfloat16)
    out = _run(q, k, v, P, synth.chain_tree(n))
    assert _err(out, _ref(q, k, v, P, synth.chain_tree(n))) <= BF16_TOL


def test_runs_are_bitwise_reproducible():
    w = synth.make_workload("l3_8b", seed=5, with_logits=False)
    q, k, v = synth.make_qkv(w, layer=0)
    a = _run(q, k, v, w.prefix, w.parent).cpu()
    b = _run(q, k, v, w.prefix, w.parent).cpu()
    assert torch.equal(a, b)


@pytest.mark.parametrize("bad", [[-1, 1, 0], [-1, 0, 5], [-1, -3, 0]])
def test_invalid_tree_sets_device_status(bad):
    rng = np.random.default_rng(0)
    q, k, v = _qkv(rng, 3, 4, 1, 64, 40, torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    _run(q, k, v, 30, bad, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == tvp.TV_ERR_INVALID_TREE


def test_host_side_errors():
    rng = np.random.default_rng(0)
    q, k, v = _qkv(rng, 3, 4, 1, 64, 40, torch.bfloat16)
    with pytest.raises(tvp.TreeVerifyError) as e:
        _run(q, k, v, 38, [-1, 0, 1])       # P + N > cap
    assert e.value.status == tvp.TV_ERR_CAPACITY
    q2, k2, v2 = _qkv(rng, 3, 4, 1, 96, 40, torch.bfloat16)
    with pytest.raises(tvp.TreeVerifyError) as e:
        _run(q2, k2, v2, 10, [-1, 0, 1])    # d = 96
    assert e.value.status == tvp.TV_ERR_UNSUPPORTED
    par = torch.tensor([-1, 0, 1], dtype=torch.int32, device=DEV)
    small = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(tvp.TreeVerifyError) as e:
        tvp.tree_attn_verify(q.to(DEV), k.to(DEV), v.to(DEV), 10, par, workspace=small)
    assert e.value.status == tvp.TV_ERR_CAPACITY


@pytest.mark.parametrize("n", [1, 31, 32, 33, 64, 96, 128])
def test_tree_mask_words_match_oracle(n):
    rng = np.random.default_rng(n)
    parent = synth.random_parent_tree(rng, n, max_depth=16)
    words = tvp.tree_mask(torch.from_numpy(parent).to(DEV)).cpu().numpy().view(np.uint32)
    assert np.array_equal(words, oracle.ancestor_bitmask(parent))


@pytest.mark.parametrize("grow", [0.0, 3.0])
def test_single_tile_with_late_maxima(grow):
    # G * N <= 128 rows per KV head: one row tile per CTA, whose scores are
    # double-buffered.  Key norms growing along the prefix make later blocks
    # raise the running maximum, which rescales O while the previous PV may
    # still be in flight.
    rng = np.random.default_rng(7)
    n, P, hq, hkv, d = 8, 8192, 64, 8, 128
    parent = synth.random_parent_tree(rng, n, max_depth=4)
    q, k, v = _qkv(rng, n, hq, hkv, d, P + n, torch.bfloat16)
    ramp = torch.from_numpy((1.0 + grow * np.arange(P + n) / (P + n)).astype(np.float32))
    k = (k.float() * ramp[None, :, None]).to(torch.bfloat16)
    out = _run(q, k, v, P, parent)
    nodes = [0, 3, 7]
    assert _err(out, _ref(q, k, v, P, parent, nodes=nodes), nodes) <= BF16_TOL


@pytest.mark.parametrize("hq,hkv,n,P,lo,hi", [
    (64, 8, 64, 4096, 2, 12),      # per-count combine (9 splits at the full step's layer)
    (64, 8, 8, 8192, 13, 32),      # lane-parallel combine: 17 splits of a short tree
    (8, 1, 8, 8192, 33, 10 ** 6),  # one KV head: more than 32 splits, the loop
])
def test_each_combine_path(hq, hkv, n, P, lo, hi):
    splits = tvp.attn_plan(n, hq, hkv, 128, torch.bfloat16, P)["splits"]
    assert lo <= splits <= hi, splits
    rng = np.random.default_rng(900 + splits)
    parent = synth.random_parent_tree(rng, n, max_depth=8)
    q, k, v = _qkv(rng, n, hq, hkv, 128, P + n, torch.bfloat16)
    out = _run(q, k, v, P, parent)
    nodes = sorted({0, n // 2, n - 1})
    assert _err(out, _ref(q, k, v, P, parent, nodes=nodes), nodes) <= BF16_TOL


# Key blocks per CTA: with two tiles per CTA (N 64) V(j) and K(j+1) share a
# barrier except K(2); with one tile (N 32, N 8) the K slot release is read
# from the score barrier.  Each case pins the split plan so that CTAs hold 1 to
# 8 key blocks (the last split often fewer), covering every pairing edge.
@pytest.mark.parametrize("n,P,per", [
    (64, 500, 1), (64, 1500, 2), (64, 3000, 3), (64, 5000, 5), (64, 6000, 6),
    (32, 1200, 2), (32, 2500, 3), (32, 3500, 4), (32, 9000, 8), (8, 2500, 2), (8, 9000, 4),
])
def test_blocks_per_cta(n, P, per):
    plan = tvp.attn_plan(n, 64, 8, 128, torch.bfloat16, P)
    assert plan["keys_per_split"] // 128 == per, plan
    rng = np.random.default_rng(700 + n + P)
    parent = synth.random_parent_tree(rng, n, max_depth=8)
    q, k, v = _qkv(rng, n, 64, 8, 128, P + n, torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(q, k, v, P, parent, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    nodes = sorted({0, n // 3, n - 1})
    assert _err(out, _ref(q, k, v, P, parent, nodes=nodes), nodes) <= BF16_TOL


# The d 64 instantiation of the tensor-core kernel at the full step's head
# layout: two tiles per CTA (N 64) and one (N 32, N 8), several key blocks each.
@pytest.mark.parametrize("n,P", [(64, 3000), (64, 600), (32, 2500), (8, 9000)])
def test_head_dim_64_tile_paths(n, P):
    rng = np.random.default_rng(1100 + n + P)
    parent = synth.random_parent_tree(rng, n, max_depth=8)
    q, k, v = _qkv(rng, n, 64, 8, 64, P + n, torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(q, k, v, P, parent, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    nodes = sorted({0, n // 2, n - 1})
    assert _err(out, _ref(q, k, v, P, parent, nodes=nodes), nodes) <= BF16_TOL
