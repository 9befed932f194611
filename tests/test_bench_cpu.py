"""Host-side logic of bench.py that needs no GPU: the step-4 walk policy of the
timed round, the workload's byte and flop model, and the DRAM-traffic table
lookup (reported only while the kernel's sources match the capture), and the
`--impl reference` arm (the oracle timed on the host)."""
import os

import bench
from diffusion_draft_tree_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_walk_policy():
    bench.WALK = "auto"
    want = {"tiny": "full", "8b_single": "path", "budget_sweep_n32": "path",
            "budget_sweep_n64": "path", "budget_sweep_n128": "path",
            "budget_sweep_n512": "path", "ragged_serving": "path", "long_context_70b": "path"}
    for name, walk in want.items():
        assert bench.walk_for(wl.CONFIGS[name]) == walk, name
    for forced in ("full", "path"):
        bench.WALK = forced
        assert bench.walk_for(wl.CONFIGS["8b_single"]) == forced
    bench.WALK = "auto"


def test_config_names_the_walk():
    bench.WALK = "auto"
    c = bench.config_of(wl.CONFIGS["ragged_serving"])
    assert c["workload"] == "ragged_serving" and c["walk"] == "path"
    # both arms print this same dict: nothing in it depends on the arm
    assert c == bench.config_of(wl.CONFIGS["ragged_serving"]) and "l2" in c


def test_oracle_attention_sample():
    """Small layers run in full as (sequence, KV head) units; large ones as a
    seeded sample of node rows within the per-core budget, at least one row per
    core, never past a sequence's tree."""
    w = wl.CONFIGS["8b_single"]
    tasks, done, total = bench.oracle_attn_tasks(w, [w.N], 8)
    assert done == total and len(tasks) == w.Hkv and all(t[2:] == (0, w.N + 1) for t in tasks)
    w = wl.CONFIGS["long_context_70b"]
    n = [200, 256, 10, 0]
    tasks, done, total = bench.oracle_attn_tasks(w, n, 4)
    assert 4 <= len(tasks) and done <= 4 * bench.ORACLE_ROWS_PER_CORE + 8 * (131072 + 257)
    assert total == sum(8 * (n[b] + 1) * 8 * (131072 + n[b] + 1) for b in range(4))
    assert len(set(tasks)) == len(tasks)
    for b, g, lo, hi in tasks:
        assert 0 <= g < 8 and hi == lo + 1 and 0 <= lo <= n[b]
    assert tasks == bench.oracle_attn_tasks(w, n, 4)[0]  # seeded


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


def _run_bench(args, env_extra=None):
    import json
    import subprocess
    import sys
    env = dict(os.environ, **(env_extra or {}))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True,
                       text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    return [json.loads(l) for l in lines]


def test_reference_arm_line():
    """`--impl reference` times the oracle on the host and prints one line with
    the GPU arm's metric, unit and direction, its own cpu_baseline and an e2e
    equal to its value with no host-device traffic."""
    (line,) = _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "2",
                          "--warmup", "1"])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC
    assert line["unit"] == "rounds/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["steps"] == 2 and line["warmup"] == 1
    assert line["config"] == bench.config_of(wl.CONFIGS["tiny"])
    # value and ms_per_step are the measured steps
    assert abs(line["value"] * line["ms_per_step"] / 1e3 - 1) < 1e-9  # B = 1
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == bench.host_cores() and cb["sample"]
    assert cb["value"] == line["value"]
    assert line["full_round_extrapolated"]["rounds_per_s"] > 0
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_print_nothing():
    assert _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "1",
                       "--warmup", "0", "--gpus", "2"],
                      {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []
