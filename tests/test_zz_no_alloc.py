"""The allocation-free attention entry point, tv_tree_attn_verify_static.

Some callers cannot allocate device memory: a serving framework whose caching
allocator owns the whole GPU, a plug-in that is only handed its buffers, a
latency-critical loop where cudaMalloc/cudaFree would synchronise the device.
For them the library keeps its split partials in one fixed device array.
These tests call that entry point through the C ABI and compare it with the
workspace-taking entry point on the same inputs, twice in a row (the second
call reuses the array the first one left behind).  This file is collected
last so that a run stopping at its first failure has run everything else."""
import ctypes

import numpy as np
import pytest
import torch

from workloads import synth

tvp = pytest.importorskip("speculative_decoding_tree_masked_gb300")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
BF16_TOL = 2e-2
F32_TOL = 1e-4


def _static(q, k, v, P, parent, out):
    lib = tvp.lib()
    n, hq, d = q.shape
    hkv, cap, _ = k.shape
    return lib.tv_tree_attn_verify_static(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), cap, P, n, parent.data_ptr(), out.data_ptr(),
        hq, hkv, d, tvp.TV_BF16 if q.dtype == torch.bfloat16 else tvp.TV_F32,
        ctypes.c_float(0.0), None, torch.cuda.current_stream().cuda_stream)


def _case(name, **kw):
    w = synth.make_workload(name, seed=7, with_logits=False, **kw)
    q, k, v = synth.make_qkv(w, layer=0)
    return (q.to(DEV), k.to(DEV), v.to(DEV), w.prefix,
            torch.from_numpy(w.parent).to(DEV))


def test_static_scratch_matches_workspace_entry_point_twice():
    cases = [_case("full_step", layers=1), _case("l3_8b"), _case("tiny")]
    for q, k, v, P, parent in cases + cases[:1]:
        want = tvp.tree_attn_verify(q, k, v, P, parent)
        got = torch.empty_like(q)
        assert _static(q, k, v, P, parent, got) == tvp.TV_OK
        torch.cuda.synchronize()
        tol = BF16_TOL if q.dtype == torch.bfloat16 else F32_TOL
        assert float((got.float() - want.float()).abs().max()) <= tol


def test_oversized_problem_is_rejected_before_launch():
    # 1024 query heads over 8 KV heads and 128 nodes need about 34 MB of
    # partials, more than the 16 MiB array: rejected, nothing launched
    q = torch.zeros((128, 1024, 128), dtype=torch.bfloat16, device=DEV)
    k = torch.zeros((8, 4096 + 128, 128), dtype=torch.bfloat16, device=DEV)
    parent = torch.from_numpy(synth.chain_tree(128)).to(DEV)
    out = torch.empty_like(q)
    assert tvp.lib().tv_attn_workspace_size(128, 1024, 8, 128, tvp.TV_BF16, 4096) > (16 << 20)
    assert _static(q, k, k, 4096, parent, out) == tvp.TV_ERR_CAPACITY
