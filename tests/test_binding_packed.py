"""Host logic of the packed (batched) acceptance layout, without a GPU: the
offsets, the slicing of a packed result back into one request's results,
and the per-request views of a packed new_pos.  The packed dict is built here
from the oracle's per-request results following the layout the C header
documents (request b's nodes from off[b], its out_tokens from off[b] + b),
so the binding's unpacking is checked against that layout."""
import numpy as np
import pytest
import torch

import oracle
from workloads import synth

tvp = pytest.importorskip("speculative_decoding_tree_masked_gb300")


def test_node_offsets():
    assert tvp.node_offsets([]) == [0]
    assert tvp.node_offsets([3, 1, 2]) == [0, 3, 4, 6]
    assert tvp.node_offsets([128] * 16)[-1] == 2048


def _pack(results, ns):
    off = tvp.node_offsets(ns)
    total, batch = off[-1], len(ns)
    packed = {k: np.full(total, -7, np.int32) for k in ("am", "path", "new_pos", "new_parent")}
    packed["out_tokens"] = np.full(total + batch, -7, np.int32)
    packed["m"] = np.zeros(batch, np.int32)
    packed["n_survivors"] = np.zeros(batch, np.int32)
    for b, r in enumerate(results):
        for k in ("am", "path", "new_pos", "new_parent"):
            packed[k][off[b]:off[b + 1]] = r[k]
        packed["out_tokens"][off[b] + b:off[b + 1] + b + 1] = r["out_tokens"]
        packed["m"][b] = r["m"]
        packed["n_survivors"][b] = r["n_survivors"]
    out = {k: torch.from_numpy(v) for k, v in packed.items()}
    out["node_offset"] = off
    return out


@pytest.mark.parametrize("seed", range(4))
def test_batched_request_unpacks_the_documented_layout(seed):
    rng = np.random.default_rng(seed)
    ns = [int(x) for x in rng.integers(1, 129, int(rng.integers(1, 17)))]
    results = []
    for n in ns:
        parent = synth.random_parent_tree(rng, n, max_depth=10)
        token = rng.integers(0, 4, size=n).astype(np.int32)
        logits = rng.standard_normal((n, 4)).astype(np.float32)
        results.append(oracle.tree_accept(logits, token, parent, int(rng.integers(0, 999))))
    packed = _pack(results, ns)
    # every packed entry is claimed by exactly one request: no -7 survives
    for k in ("am", "path", "new_pos", "new_parent", "out_tokens"):
        assert (packed[k] != -7).all()
    for b, want in enumerate(results):
        got = tvp.batched_request(packed, b)
        for k in ("am", "path", "new_pos", "new_parent", "out_tokens"):
            assert np.array_equal(got[k].numpy(), want[k]), (b, k)
        assert int(got["m"].item()) == want["m"]
        assert int(got["n_survivors"].item()) == want["n_survivors"]


def test_per_request_new_pos_views():
    packed = torch.arange(10, dtype=torch.int32)
    views = tvp._per_request_new_pos(packed, [3, 1, 6])
    assert [v.tolist() for v in views] == [[0, 1, 2], [3], [4, 5, 6, 7, 8, 9]]
    assert all(v.is_contiguous() for v in views)
    with pytest.raises(ValueError):
        tvp._per_request_new_pos(packed, [3, 1, 5])             # sizes do not add up
    with pytest.raises(ValueError):
        tvp._per_request_new_pos([packed[:3]], [3, 7])           # one tensor per request
    with pytest.raises(ValueError):
        tvp._per_request_new_pos([packed[:3].long()], [3])       # int32 only


def test_batched_calls_reject_host_tensors():
    cpu = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(ValueError):
        tvp.tree_accept_batched(torch.zeros((4, 10)), cpu, cpu, [4], [0])
    with pytest.raises(ValueError):
        tvp.kv_compact_batched([torch.zeros((1, 8, 16))], [torch.zeros((1, 8, 16))], [0], [4],
                               cpu)
