"""GPU parity of batched tree attention (several requests with their own
prefixes, trees and caches in one launch, through the C ABI) against the
oracle per request, against the single-request call, and the masking
invariant per request."""
import numpy as np
import pytest
import torch

import oracle
from workloads import synth

tvp = pytest.importorskip("speculative_decoding_tree_masked_gb300")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
BF16_TOL = 2e-2


def _request(rng, n, P, hq, hkv, d, extra=3):
    parent = synth.random_parent_tree(rng, n, max_depth=12)
    f = lambda *s: torch.from_numpy(rng.standard_normal(s, dtype=np.float32)).to(torch.bfloat16)
    return f(n, hq, d), f(hkv, P + n + extra, d), f(hkv, P + n + extra, d), parent


def _oracle(q, k, v, P, parent, nodes=None):
    return oracle.tree_attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), P,
                                 parent, nodes=nodes)


@pytest.mark.parametrize("case", range(4))
def test_ragged_batch_matches_oracle(case):
    rng = np.random.default_rng(200 + case)
    hq, hkv, d = [(64, 8, 128), (32, 8, 128), (16, 2, 64), (64, 8, 128)][case]
    shapes = [[(64, 4096), (8, 300), (128, 1000), (33, 0)],
              [(64, 2048), (64, 2048), (16, 7000)],
              [(7, 129), (100, 50), (1, 0), (128, 513), (40, 2000)],
              [(8, 16384), (64, 1024)]][case]
    reqs = [_request(rng, n, P, hq, hkv, d) for n, P in shapes]
    outs = tvp.tree_attn_verify_batched([r[0].to(DEV) for r in reqs],
                                        [r[1].to(DEV) for r in reqs],
                                        [r[2].to(DEV) for r in reqs],
                                        [P for _, P in shapes],
                                        [torch.from_numpy(r[3]).to(DEV) for r in reqs])
    torch.cuda.synchronize()
    for (n, P), (q, k, v, parent), out in zip(shapes, reqs, outs):
        nodes = sorted({0, n // 2, n - 1})
        ref = _oracle(q, k, v, P, parent, nodes=nodes)
        assert float(np.abs(out.float().cpu().numpy()[nodes] - ref).max()) <= BF16_TOL


def test_sixteen_requests_agree_with_single_calls():
    rng = np.random.default_rng(5)
    hq, hkv, d = 32, 8, 128
    shapes = [(int(rng.integers(1, 129)), int(rng.integers(0, 3000))) for _ in range(16)]
    reqs = [_request(rng, n, P, hq, hkv, d) for n, P in shapes]
    dev = [(q.to(DEV), k.to(DEV), v.to(DEV), torch.from_numpy(p).to(DEV)) for q, k, v, p in reqs]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = tvp.tree_attn_verify_batched([x[0] for x in dev], [x[1] for x in dev],
                                        [x[2] for x in dev], [P for _, P in shapes],
                                        [x[3] for x in dev], status=st)
    for (n, P), x, out in zip(shapes, dev, outs):
        single = tvp.tree_attn_verify(x[0], x[1], x[2], P, x[3])
        torch.cuda.synchronize()
        assert float((out.float() - single.float()).abs().max()) <= BF16_TOL
    assert int(st.item()) == 0


def test_masked_rows_do_not_change_batched_outputs():
    rng = np.random.default_rng(9)
    hq, hkv, d = 16, 4, 128
    shapes = [(20, 130), (9, 0), (64, 700)]
    reqs = [_request(rng, n, P, hq, hkv, d, extra=50) for n, P in shapes]

    def run(reqs):
        outs = tvp.tree_attn_verify_batched([r[0].to(DEV) for r in reqs],
                                            [r[1].to(DEV) for r in reqs],
                                            [r[2].to(DEV) for r in reqs],
                                            [P for _, P in shapes],
                                            [torch.from_numpy(r[3]).to(DEV) for r in reqs])
        torch.cuda.synchronize()
        return [o.view(torch.int16).cpu() for o in outs]
    a = run(reqs)
    # rows past each request's tree hold NaN; rows of non-ancestors grow x1000
    poisoned = []
    for (n, P), (q, k, v, parent) in zip(shapes, reqs):
        k2, v2 = k.clone(), v.clone()
        k2[:, P + n:, :] = float("nan")
        v2[:, P + n:, :] = float("nan")
        poisoned.append((q, k2, v2, parent))
    b = run(poisoned)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
