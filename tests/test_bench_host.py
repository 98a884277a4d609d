"""Host-side pieces of the benchmark contract (no GPU): the algorithmic bytes
of a pass, the traffic table's keys, the reference arm's line shape."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth import workloads as W  # noqa: E402


def test_algorithmic_bytes_of_the_qwen3_layer():
    w = W.get_workload("qwen3_8b_layer")
    score_b, move_b = bench.algorithmic_bytes(w, 8 * 8000)
    assert score_b == 8 * 32768 * 256                     # every fp16 key row read once
    assert move_b == 8 * 8000 * (2 * 256 + 2 * 256 + 8)   # read + write of K, V and pos
    w8 = W.get_workload("q8_0")
    s8, _ = bench.algorithmic_bytes(w8, 0)
    assert s8 == 8 * 65536 * (128 + 8)                    # q8_0 codes + fp16 block scales


def test_traffic_table_names_known_workloads_and_kernels():
    for (name, kernel), val in bench.TRAFFIC.items():
        assert name in W.WORKLOADS and kernel in ("k_score", "k_move", "k_pass")
        assert isinstance(val, int) and val > 0


def test_reference_arm_prints_one_line_on_the_host():
    """--impl reference runs the oracle on the host cores (tiny workload, one
    short step): one JSON line with the contract's keys."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "tiny", "--steps", "1", "--warmup", "1"], capture_output=True, text=True, env=env,
                         timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0


def test_both_arms_describe_the_workload_with_the_same_config():
    """The reference arm's config is the one the GPU arm reports (same keys and
    values), so the two lines compare the same workload."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "tiny", "--steps", "1", "--warmup", "1"], capture_output=True, text=True, env=env,
                         timeout=300)
    d = json.loads([ln for ln in res.stdout.splitlines() if ln.startswith("{")][0])
    assert d["config"] == json.loads(json.dumps(bench.config_of(W.get_workload("tiny"), 1)))


def test_default_workload_is_the_whole_batched_model():
    args = bench.parse([])
    assert args.workload == "batched_long" and args.layers == 0
    assert W.get_workload(args.workload).n_layers == 48
