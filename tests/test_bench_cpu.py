"""Host-side logic of bench.py that needs no GPU: the step-4 walk policy of the
timed round, the workload's byte and flop model, and the DRAM-traffic table
lookup (reported only while the kernel's sources match the capture)."""
import os

import bench
from diffusion_draft_tree_gb300 import workloads as wl


def test_walk_policy():
    bench.WALK = "auto"
    want = {"tiny": "full", "8b_single": "full", "budget_sweep_n32": "full",
            "budget_sweep_n64": "full", "budget_sweep_n128": "path",
            "budget_sweep_n512": "path", "ragged_serving": "path", "long_context_70b": "path"}
    for name, walk in want.items():
        assert bench.walk_for(wl.CONFIGS[name]) == walk, name
    for forced in ("full", "path"):
        bench.WALK = forced
        assert bench.walk_for(wl.CONFIGS["8b_single"]) == forced
    bench.WALK = "auto"


def test_config_names_the_walk():
    bench.WALK = "auto"
    c = bench.config_of(wl.CONFIGS["ragged_serving"], None)
    assert c["workload"] == "ragged_serving" and c["walk"] == "path"


def test_work_model_8b():
    w = wl.CONFIGS["8b_single"]
    m = bench.work_model(w, 0)
    # top-K reads every draft row once; the full walk every tree row once
    assert m["topk"]["bytes"] >= w.B * w.L * w.V * w.esize
    assert m["accept"]["bytes"] == w.B * (w.N + 1) * w.V * w.esize
    # tree attention: K/V prefix + tree K/V + Q in + O out, in bf16
    P = w.P[0]
    expect = (4 * w.Hkv * w.D * P + 4 * w.Hkv * w.D * w.B * (w.N + 1)
              + 4 * w.Hq * w.D * w.B * (w.N + 1))
    assert m["tree_attn"]["bytes"] == expect


def test_traffic_lookup_follows_the_sources(tmp_path, monkeypatch):
    got = bench.measured_traffic("tree_attn", "8b_single")
    assert got is None or got > 9_000_000
    assert bench.measured_traffic("tree_attn", "no_such_workload") is None
