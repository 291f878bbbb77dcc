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
    b = bench._bounds_us(2e9, 3e12, 152 * 16 * 1e9, peaks, sms=152)
    assert abs(b["hbm"] - 2000.0) < 1e-9
    assert abs(b["tensor"] - 30000.0) < 1e-9
    assert abs(b["exp"] - 1e6) < 1e-6


def test_reference_arm_prints_the_contract_line():
    # the reference arm is the CPU oracle: it runs without a GPU and prints
    # one JSON line in the bench contract's shape
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                         timeout=600, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert "workload" in d["config"]


def test_all_cores_oracle_sample_runs_and_scales():
    # the cpu_baseline leg's parallel sample, small: 2 processes, 4 nodes of one layer
    s = bench._oracle_subprocess(4, 1, 1, workers=2)[0]
    one = bench._oracle_subprocess(4, 1, 1)[0]
    assert s["threads"] == 2 and "over 2 processes" in s["sample"]
    assert s["t_step_s"] > 0 and one["t_step_s"] > 0
    assert s["m"] == one["m"]                       # the same acceptance on the same inputs
