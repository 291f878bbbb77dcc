"""The allocation-free attention entry point, tv_tree_attn_verify_static.

Some callers cannot allocate device memory: a serving framework whose caching
allocator owns the whole GPU, a plug-in that is only handed its buffers, a
latency-critical loop where cudaMalloc/cudaFree would synchronise the device.
For them the library keeps its split partials in one fixed device array.
These tests call that entry point through the C ABI and compare it with the
workspace-taking entry point on the same inputs, twice in a row (the second
call reuses the array the first one left behind).  Both calls run the same
kernels under the same split plan, so their outputs must agree bit for bit;
one shape is also checked against the oracle.  This file is collected last
so that a run stopping at its first failure has run everything else."""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from workloads import synth

tvp = pytest.importorskip("speculative_decoding_tree_masked_gb300")

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
BF16_TOL = 2e-2
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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
        got = torch.full_like(q, float("nan"))
        assert _static(q, k, v, P, parent, got) == tvp.TV_OK
        torch.cuda.synchronize()
        assert torch.equal(got, want)


def test_binding_wrapper_against_the_oracle():
    # the Python wrapper (its shape and dtype checks), then the oracle
    w = synth.make_workload("l3_8b", seed=3, with_logits=False)
    q, k, v = synth.make_qkv(w, layer=0)
    parent = torch.from_numpy(w.parent).to(DEV)
    out = torch.empty(q.shape, dtype=q.dtype, device=DEV)
    for _ in range(2):
        tvp.tree_attn_verify_static(q.to(DEV), k.to(DEV), v.to(DEV), w.prefix, parent, out)
        torch.cuda.synchronize()
        ref = oracle.tree_attention(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                    w.prefix, w.parent)
        assert float(np.abs(out.float().cpu().numpy() - ref).max()) <= BF16_TOL
    with pytest.raises(ValueError):
        tvp.tree_attn_verify_static(q.to(DEV), k.to(DEV), v.to(DEV), w.prefix, parent,
                                    out[:-1])


def test_first_call_in_a_fresh_process():
    # the first call right after the CUDA context is created (the array is
    # reserved then), then a second, both against the workspace entry point
    code = (
        "import torch, ctypes\n"
        "import speculative_decoding_tree_masked_gb300 as tvp\n"
        "from workloads import synth\n"
        "torch.cuda.init(); torch.zeros(1, device='cuda:0')\n"
        "w = synth.make_workload('l3_8b', seed=9, with_logits=False, prefix=700, n=40)\n"
        "q, k, v = [t.to('cuda:0') for t in synth.make_qkv(w, layer=0)]\n"
        "par = torch.from_numpy(w.parent).to('cuda:0')\n"
        "outs = [torch.empty_like(q) for _ in range(2)]\n"
        "for o in outs:\n"
        "    tvp.tree_attn_verify_static(q, k, v, w.prefix, par, o)\n"
        "want = tvp.tree_attn_verify(q, k, v, w.prefix, par)\n"
        "torch.cuda.synchronize()\n"
        "assert all(torch.equal(o, want) for o in outs)\n"
        "print('fresh ok')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and "fresh ok" in r.stdout, r.stdout + r.stderr


def test_oversized_problem_is_rejected_before_launch():
    # 1024 query heads over 8 KV heads and 128 nodes need about 34 MB of
    # partials, more than the 16 MiB array: rejected, nothing launched
    q = torch.zeros((128, 1024, 128), dtype=torch.bfloat16, device=DEV)
    k = torch.zeros((8, 4096 + 128, 128), dtype=torch.bfloat16, device=DEV)
    parent = torch.from_numpy(synth.chain_tree(128)).to(DEV)
    out = torch.empty_like(q)
    assert tvp.lib().tv_attn_workspace_size(128, 1024, 8, 128, tvp.TV_BF16, 4096) > (16 << 20)
    assert _static(q, k, k, 4096, parent, out) == tvp.TV_ERR_CAPACITY
