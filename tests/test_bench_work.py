"""The algorithmic work bench.py divides by: bytes, flops and visible
(row, key) pairs of one tree-attention call, checked against counts made by
hand for trees whose ancestor sets are known in closed form, and the lower
bounds derived from them."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from workloads import synth  # noqa: E402


def test_chain_tree_counts():
    # node i of a chain sees the whole prefix and nodes 0..i: i + 1 tree keys
    n, P, hq, hkv, d = 10, 100, 8, 2, 64
    parent = synth.chain_tree(n)
    anc = n * (n + 1) // 2
    nbytes, flops = bench._algorithmic_work(parent, P, n, hq, hkv, d)
    assert nbytes == 2 * hkv * (P + n) * d * 2 + 2 * n * hq * d * 2
    assert flops == 4 * hq * d * (n * P + anc)
    assert bench._visible_pairs(parent, P, hq) == hq * (n * P + anc)


def test_star_tree_counts():
    # every non-root node's only strict ancestor is the root: 2 tree keys
    n, P, hq = 9, 7, 4
    parent = np.array([-1] + [0] * (n - 1), dtype=np.int32)
    assert bench._visible_pairs(parent, P, hq) == hq * (n * P + 1 + 2 * (n - 1))


def test_bounds_scale_with_their_peaks():
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0, "sm_max_mhz": 1000.0}
    b = bench._bounds_us(2e9, 3e12, 152 * 16 * 1e9, peaks)
    assert abs(b["hbm"] - 2000.0) < 1e-9
    assert abs(b["tensor"] - 30000.0) < 1e-9
    assert abs(b["exp"] - 1e6) < 1e-6
