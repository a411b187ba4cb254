"""The bench's byte accounting (measurement, not the method) against hand counts."""
import numpy as np

import bench
import workloads as W


def test_dense_bytes_count_each_active_slot_once():
    """Two slots of rank 8 and 16 used by 3 tokens, one token without an adapter and
    one on a rank-0 slot; k = 64, slices 32 + 16 (d = 48)."""
    slot_ids = np.array([0, 1, 0, -1, 2], np.int32)
    ranks = np.array([8, 16, 0], np.int32)
    k, widths = 64, [32, 16]
    weights = 2 * 8 * (2 * 64 + 48) + 2 * 16 * (2 * 64 + 48)   # A and B of slots 0 and 1, bf16
    rows = 2 * 64 * 3 + 4 * 48 * 3                               # x read, y read and written: 3 tokens
    assert bench.algorithmic_bytes(slot_ids, ranks, k, widths) == weights + rows
    assert bench.algorithmic_bytes(slot_ids, ranks, k, widths, wbytes=1) == weights // 2 + rows


def test_moe_bytes_count_each_used_expert_pair_once():
    """3 tokens, K = 2, E = 4, adapters of rank 8: token 0 (adapter 0) on experts 1, 2;
    token 1 (adapter 0) on experts 2, 3; token 2 without an adapter.  Three distinct
    (adapter, expert) pairs are used, by four pairs."""
    wl = W.generate_moe(name="acct", seed=1, T=3, K=2, E=4, n_adapters=1, rank=8,
                        modules=[{"name": "up", "k": 64, "slices": [32], "x_per_token": True},
                                 {"name": "down", "k": 32, "slices": [64], "x_per_token": False}])
    wl.slot_ids = np.array([0, 0, -1], np.int32)
    wl.expert_ids = np.array([[1, 2], [2, 3], [0, 1]], np.int32)
    up = 3 * 2 * 8 * (64 + 32) + 2 * 64 * 2 + 4 * 32 * 4       # 3 expert pairs, x per token (2), y of 4 pairs
    down = 3 * 2 * 8 * (32 + 64) + 2 * 32 * 4 + 4 * 64 * 4     # x per pair (4)
    assert bench.moe_algorithmic_bytes(wl, 0) == up
    assert bench.moe_algorithmic_bytes(wl, 1) == down


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference (the oracle on the host cores) prints one JSON line
    with the keys the driver reads, on a config small enough for a unit test."""
    import json
    import subprocess
    import sys
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny", "--steps", "2",
                          "--warmup", "1"], cwd=root, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-500:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
