"""The CPU arms of bench.py: `--impl reference` and the threaded oracle baseline.

Both time the unchanged oracle on host threads that fold disjoint rows. This
checks, without a GPU, that the reference arm prints one JSON line with the
contract's keys, and that the threaded timing returns rows from every thread.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_prints_contract_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "4", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["steps"] == 4 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["unit"] == "rows/s"
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == d["value"] and cpu["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "rows/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    import bench
    from gather_lora_gb300 import workloads as W
    wl = W.by_name(bench.HEADLINE)
    assert d["config"] == bench.workload_config(wl, bench.algorithmic_bytes(wl))
    assert d["config"]["workload"] == "moe_down_fold" and d["config"]["windows"] == 4
    assert cpu["cpu_model"]


@pytest.mark.parametrize("name", ["moe_down_fold", "decode_qproj_bgmv"])
def test_threaded_oracle_baseline_counts_every_thread(name):
    import bench
    import oracle
    from gather_lora_gb300 import workloads as W
    oracle.load()
    wl = W.by_name(name)
    rows_per_s, rows, secs = bench.oracle_rows_per_s(wl, 0.0, rows_per_call=2, threads=3)
    # a zero budget still lets each thread fold one call's rows
    assert rows == 3 * 2 and secs > 0 and rows_per_s > 0
    base = bench.cpu_baseline(wl, 0.0)
    assert base["cores"] == bench.host_threads() and base["kind"] == "oracle"
    assert base["single_thread"]["cores"] == 1 and base["single_thread"]["value"] > 0


def test_moe_oracle_sample_equals_the_window_fold():
    """The baseline folds sorted rows [lo, hi) as the same problem on fewer rows;
    its results must be the rows the oracle gives over the whole window."""
    import numpy as np
    import oracle
    from gather_lora_gb300 import workloads as W
    from gpu_util import oracle_moe
    oracle.load()
    wl = W.make_moe("sample_eq", num_tokens=96, top_k=4, num_experts=12, k_in=64, n_out=48,
                    max_loras=3, max_rank=8, rank=8, alpha=16.0, adapter_base_frac=0.2, cap=384,
                    seed=12)
    full, _, _ = oracle_moe(wl, wl.windows())
    lo, hi = 37, 211
    offs = np.clip(wl.expert_offsets.astype(np.int64) - lo, 0, hi - lo).astype(np.int32)
    out = wl.out_buf[lo:hi].copy()
    oracle.lora_moe_grouped_fold(wl.x[lo:hi], wl.k_in, out, wl.n_out, offs,
                                 wl.sorted_token_ids[lo:hi], wl.row_adapter, wl.num_tokens, 0,
                                 hi - lo, wl.a_list(), wl.b_list(), wl.scale, wl.max_rank, wl.k_in,
                                 wl.n_out)
    assert np.array_equal(out, full[lo:hi])


def test_one_launch_moe_workload_is_the_same_problem():
    import numpy as np
    import bench
    from gather_lora_gb300 import workloads as W
    a = W.by_name("moe_down_fold")
    b = W.by_name("moe_down_fold_one_launch")
    assert b.name == "moe_down_fold_one_launch" and b.cap == b.te == a.te
    assert b.windows() == [(0, a.te)] and len(a.windows()) == 4
    for f in ("x", "out_buf", "expert_offsets", "sorted_token_ids", "row_adapter", "present",
              "a_pool", "b_pool", "scale"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    ba, bb = bench.algorithmic_bytes(a), bench.algorithmic_bytes(b)
    # same routed rows; an (adapter, expert) pair split by a window boundary is counted once
    assert ba["routed_rows"] == bb["routed_rows"] and bb["adapters"] <= ba["adapters"]
    assert bb["bytes"] < ba["bytes"]
    assert "moe_down_fold_one_launch" in bench.SIDE_WORKLOADS


def test_threaded_oracle_baseline_propagates_a_thread_failure(monkeypatch):
    import pytest
    import bench
    from gather_lora_gb300 import workloads as W
    wl = W.by_name("tiny_bgmv")

    def boom(wl, idx):
        raise RuntimeError("oracle call failed")

    monkeypatch.setattr(bench, "oracle_fold", boom)
    with pytest.raises(RuntimeError, match="oracle call failed"):
        bench.oracle_rows_per_s(wl, 0.0, rows_per_call=1, threads=2)
