"""Throughput of one DDTree round on GB300: top-K -> heap build -> tree
attention (one target layer) -> acceptance walk, through libddtree.so.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gb300|reference]

Prints ONE JSON line (rank 0).  `value` is sequence-rounds per second with all
inputs resident in HBM; a "step" is one round over one batch.  The default
workload is the largest single-GPU one (long_context_70b).  The round's four
C-ABI calls are captured in CUDA graphs; to keep the 129 MB L2 from serving a
step's inputs, steps rotate over copies of every per-step input (together
> 3x L2).  Each call is also timed alone (graphs of back-to-back launches) for
the per-call rates and the roofline.  `e2e` repeats the measurement through the
public API from pinned host buffers (inputs copied in and results copied out
every step).  `--impl reference` times the CPU oracle on the host cores
instead (a reported baseline; on the large workloads each step computes the
tree attention of a seeded sample of node rows).  Multi-GPU runs are
independent replicas (sequences are independent units).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from diffusion_draft_tree_gb300 import workloads as wl  # noqa: E402

L2_BYTES = 129 * 2**20
X36 = 36  # layers of the 8B-class target (Qwen3-8B)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="long_context_70b", choices=sorted(wl.CONFIGS),
                    help="default: the largest single-GPU workload (B = 4, P = 131072, "
                         "N = 256, 64/8 heads)")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-x36", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--walk", default="auto", choices=["auto", "full", "path"],
                    help="step 4: the full-tree walk (ddtree_accept), the path-only walk "
                         "(ddtree_accept_path), or auto: the path-only walk once the batch "
                         "has >= 32 tree rows, B (N + 1)")
    ap.add_argument("--acceptance-stats", type=int, default=0, metavar="ROUNDS",
                    help="instead of timing: run ROUNDS independent synthetic rounds per node "
                         "budget (and the K = 1 chain) and report acceptance lengths")
    ap.add_argument("--profile-rounds", type=int, default=0,
                    help="only run this many eager rounds (rotating input copies) and exit; "
                         "for kernel profilers")
    ap.add_argument("--profile-call", default=None,
                    choices=["topk", "build", "tree_attn", "accept", "accept_path"],
                    help="only run this one call of the round 3 times on the workload's inputs "
                         "and exit; for kernel profilers (capture the second launch)")
    ap.add_argument("--batch", type=int, default=None,
                    help="with --profile-call: use the first BATCH sequences of the workload")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# algorithmic work per launch (bytes that must move, flops that must run)
# ---------------------------------------------------------------------------

def work_model(w, tree_anc_total: int) -> dict:
    R = w.N + 1
    es = w.esize
    topk_bytes = w.B * w.L * (w.V * es + w.K * 8 + 4)
    kv_prefix = 4 * w.Hkv * w.D * sum(w.P)               # K + V, bf16
    kv_tree = 4 * w.Hkv * w.D * R * w.B
    qo = 4 * w.Hq * w.D * R * w.B                         # Q read + O written, bf16
    attn_bytes = kv_prefix + kv_tree + qo
    attn_flops = 4 * w.Hq * w.D * (R * sum(w.P)) + 4 * w.Hq * w.D * tree_anc_total
    accept_bytes = w.B * R * w.V * es
    build_bytes = w.B * (w.L * w.K * 8 + R * (7 * 4 + ((R + 31) // 32) * 4))
    return {"topk": {"bytes": topk_bytes}, "build": {"bytes": build_bytes},
            "tree_attn": {"bytes": attn_bytes, "flops": attn_flops},
            "accept": {"bytes": accept_bytes}}


# Kernels one round launches: top-K partials and row merge, tree build, tree
# attention, accept.
LAUNCHES_PER_ROUND = 5
# the headline metric, the same string on both arms
METRIC = "draft-tree rounds/sec (topK+build+tree-attn+accept); tree-attn % roofline"
# Sources a kernel's DRAM traffic depends on (its own file and shared headers).
KERNEL_SOURCES = {"tree_attn": ["tree_attn.cu", "sm100.cuh", "common.cuh"]}


def kernel_source_hash(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "diffusion_draft_tree_gb300",
                        "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) that an
    ncu capture recorded in profiles/traffic.json for this kernel and workload,
    or None if there is none or the kernel's sources changed since."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        entries = json.load(f).get("entries", [])
    want = kernel_source_hash(kernel)
    for e in entries:
        if e.get("kernel") == kernel and e.get("workload") == workload and \
                e.get("sources_sha16") == want:
            return int(e["bytes_per_launch"])
    return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def to_dev_logits(a, dtype, dev):
    import torch
    if dtype == wl.BF16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)


class Round:
    """Device buffers and calls for one round over one copy of the inputs."""

    def __init__(self, ops, w, inputs, dev, ws, layers=1):
        import torch
        self.ops, self.w = ops, w
        self.inp = inputs
        B, L, K, N = w.B, w.L, w.K, w.N
        self.topk_idx = torch.empty((B * L, K), dtype=torch.int32, device=dev)
        self.topk_lp = torch.empty((B * L, K), dtype=torch.float32, device=dev)
        self.lse = torch.empty((B * L,), dtype=torch.float32, device=dev)
        self.tree = ops.tree_buffers(B, N, dev)
        self.out = [torch.empty_like(inputs["q"][0]) for _ in range(layers)]
        self.acc = ops.accept_buffers(B, L, N, dev)
        self.ws = ws
        self.walk = walk_for(w)

    def run(self, layers=1):
        ops, w, x = self.ops, self.w, self.inp
        ops.ddtree_topk(x["draft"], w.K, self.topk_idx, self.topk_lp, self.lse, self.ws["topk"])
        ops.ddtree_build(self.topk_lp.view(w.B, w.L, w.K), self.topk_idx.view(w.B, w.L, w.K),
                         x["bonus"], x["prefix_len"], w.N, self.tree)
        for l in range(layers):
            ops.ddtree_tree_attn(x["q"][l], x["k_cache"][l], x["v_cache"][l], x["k_tree"][l],
                                 x["v_tree"][l], x["prefix_len"], self.tree["n_nodes"],
                                 self.tree["anc_mask"], self.out[l], None, None,
                                 self.ws["attn"])
        self.accept()

    def accept(self):
        ops, w, x = self.ops, self.w, self.inp
        if self.walk == "path":
            ops.ddtree_accept_path(x["target"], self.tree["parent"], self.tree["token"],
                                   self.tree["n_nodes"], w.L, self.acc, w.T, wl.philox_seed(w), 0)
        else:
            ops.ddtree_accept(x["target"], self.tree["parent"], self.tree["token"],
                              self.tree["n_nodes"], w.L, self.acc, w.T, wl.philox_seed(w), 0,
                              self.ws["accept"])

    def stages(self):
        """The four calls as separate closures (for per-kernel event timing)."""
        ops, w, x = self.ops, self.w, self.inp
        return [
            lambda: ops.ddtree_topk(x["draft"], w.K, self.topk_idx, self.topk_lp, self.lse,
                                    self.ws["topk"]),
            lambda: ops.ddtree_build(self.topk_lp.view(w.B, w.L, w.K),
                                     self.topk_idx.view(w.B, w.L, w.K), x["bonus"],
                                     x["prefix_len"], w.N, self.tree),
            lambda: ops.ddtree_tree_attn(x["q"][0], x["k_cache"][0], x["v_cache"][0],
                                         x["k_tree"][0], x["v_tree"][0], x["prefix_len"],
                                         self.tree["n_nodes"], self.tree["anc_mask"],
                                         self.out[0], None, None, self.ws["attn"]),
            self.accept,
        ]


def host_inputs(w):
    return {"draft": wl.draft_logits(w).reshape(w.B * w.L, w.V), "bonus": wl.bonus_tokens(w),
            "prefix_len": wl.prefix_lengths(w), "q": wl.queries(w), "k_cache": wl.kv_cache(w, 0),
            "v_cache": wl.kv_cache(w, 1), "k_tree": wl.kv_tree(w, 0), "v_tree": wl.kv_tree(w, 1)}


STAGE_METHOD = ("each call alone: a captured graph of M back-to-back launches over rotating "
                "copies of its own inputs (together > 3x the L2), CUDA events around the whole "
                "replay on the launching stream, per launch = total / M; no event between "
                "launches, so no per-launch event latency")


def stage_times(ops, w, base, copies, rounds, ws, dev, stream, steps):
    """Per-launch time (ms) of each call of the round and of the two calls after
    it, each timed alone (see STAGE_METHOD)."""
    import torch

    r0 = rounds[0]
    t_budget_ms = 60.0  # device time per replay

    def n_copies(nbytes):
        return int(max(2, min(64, np.ceil(3 * L2_BYTES / max(1, nbytes)))))

    def grow(key, n):  # n device copies of one per-step input (list-valued keys: layer 0)
        have = [c[key][0] if isinstance(c[key], list) else c[key] for c in copies]
        while len(have) < n:
            have.append(have[len(have) % len(copies)].clone())
        return have[:n]

    def time_graph(make, n, est_ms):
        M = n * max(1, int(min(64, max(4, t_budget_ms / max(est_ms, 1e-3))) // n))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(M):
                make(i % n)
        with torch.cuda.stream(stream):
            for _ in range(2):
                g.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            reps = []
            for _ in range(3):
                e0.record(stream)
                g.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                reps.append(e0.elapsed_time(e1) / M)
        ops.ddtree_device_check()
        del g
        return {"ms": float(np.median(reps)), "launches": M, "input_copies": n}

    def nb(t):
        return t.numel() * t.element_size()

    out = {}
    # step 1: top-K over copies of the draft logits
    drafts = grow("draft", n_copies(nb(base["draft"])))
    out["topk"] = time_graph(lambda i: ops.ddtree_topk(drafts[i], w.K, r0.topk_idx, r0.topk_lp,
                                                       r0.lse, ws["topk"]), len(drafts), 0.02)
    # restore the round's top-K outputs (same draft logits: identical)
    ops.ddtree_topk(base["draft"], w.K, r0.topk_idx, r0.topk_lp, r0.lse, ws["topk"])
    # step 2: the build reads the (small) top-K outputs, as in the round
    out["build"] = time_graph(lambda i: ops.ddtree_build(
        r0.topk_lp.view(w.B, w.L, w.K), r0.topk_idx.view(w.B, w.L, w.K), base["bonus"],
        base["prefix_len"], w.N, r0.tree), 1, 0.02)
    # step 3: tree attention over copies of q, the KV cache and the tree K/V
    kv_keys = ("q", "k_cache", "v_cache", "k_tree", "v_tree")
    n_a = n_copies(sum(nb(base[k][0]) for k in kv_keys))
    kv = {k: grow(k, n_a) for k in kv_keys}
    est = 1e-3 * sum(nb(base[k][0]) for k in kv_keys) / 2e3  # ~2 TB/s guess
    out["tree_attn"] = time_graph(lambda i: ops.ddtree_tree_attn(
        kv["q"][i], kv["k_cache"][i], kv["v_cache"][i], kv["k_tree"][i], kv["v_tree"][i],
        base["prefix_len"], r0.tree["n_nodes"], r0.tree["anc_mask"], r0.out[0], None, None,
        ws["attn"]), n_a, est)
    del kv
    # step 4, both walks, over copies of the target logits
    targets = grow("target", n_copies(nb(base["target"])))
    accs = {"path": ops.accept_buffers(w.B, w.L, w.N, dev),
            "full": ops.accept_buffers(w.B, w.L, w.N, dev)}
    seed = wl.philox_seed(w)
    est = 1e-3 * nb(base["target"]) / 3e3
    out["accept_path"] = time_graph(lambda i: ops.ddtree_accept_path(
        targets[i], r0.tree["parent"], r0.tree["token"], r0.tree["n_nodes"], w.L, accs["path"],
        w.T, seed, 0), len(targets), 0.02)
    out["accept_full"] = time_graph(lambda i: ops.ddtree_accept(
        targets[i], r0.tree["parent"], r0.tree["token"], r0.tree["n_nodes"], w.L, accs["full"],
        w.T, seed, 0, ws["accept"]), len(targets), est)
    out["same_tokens"] = bool(torch.equal(accs["path"]["out_tokens"], accs["full"]["out_tokens"]))
    out["path_rows"] = int(accs["path"]["accept_len"].sum().item()) + w.B
    out["accept"] = dict(out["accept_" + walk_for(w)])
    del targets, drafts
    # after the round: commit the accepted path (prefix lengths restored before each)
    try:
        cap2 = w.P_cap + w.L + 1
        kc2 = torch.empty((w.B, w.Hkv, cap2, w.D), dtype=torch.bfloat16, device=dev)
        vc2 = torch.empty_like(kc2)
        plen0 = base["prefix_len"]
        plen = plen0.clone()

        def commit(i):
            plen.copy_(plen0)
            ops.ddtree_commit(kc2, vc2, base["k_tree"][0], base["v_tree"][0],
                              accs["path"]["accept_len"], accs["path"]["accepted_nodes"], plen)

        out["commit"] = time_graph(commit, 1, 0.01)
        out["commit"]["note"] = ("includes a 4-byte-per-sequence copy restoring the prefix "
                                 "lengths before each launch")
        out["commit_rows"] = out["path_rows"]
        del kc2, vc2
    except Exception as e:  # noqa: BLE001
        out["commit"] = {"unavailable": repr(e)}
    return out


def gpu_arm(args, rank, world, dev):
    import torch
    from diffusion_draft_tree_gb300 import ops

    w = wl.CONFIGS[args.workload]
    torch.cuda.set_device(dev)
    h = host_inputs(w)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(
        torch.bfloat16)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
    ws = {"topk": ops.alloc_workspace(ops.workspace_size(ops.OP_TOPK, B=w.B, L=w.L, V=w.V,
                                                         K=w.K, dtype=w.dtype), dev),
          "attn": ops.alloc_workspace(ops.workspace_size(ops.OP_TREE_ATTN, B=w.B, N=w.N,
                                                         Hq=w.Hq, Hkv=w.Hkv, D=w.D,
                                                         cache_cap=w.P_cap), dev),
          "accept": ops.alloc_workspace(ops.workspace_size(ops.OP_ACCEPT, B=w.B, N=w.N, V=w.V,
                                                           dtype=w.dtype), dev)}
    base = {"draft": to_dev_logits(h["draft"], w.dtype, dev), "bonus": i32(h["bonus"]),
            "prefix_len": i32(h["prefix_len"]), "q": [bf(h["q"])], "k_cache": [bf(h["k_cache"])],
            "v_cache": [bf(h["v_cache"])], "k_tree": [bf(h["k_tree"])],
            "v_tree": [bf(h["v_tree"])]}
    # target logits come from the tree the GPU builds for these draft logits
    probe = Round(ops, w, dict(base, target=None), dev, ws)
    probe.stages()[0]()
    probe.stages()[1]()
    depth = probe.tree["depth"].cpu().numpy()
    h["target"] = wl.target_logits(w, wl.draft_logits(w), depth)
    base["target"] = to_dev_logits(h["target"], w.dtype, dev)
    torch.cuda.synchronize()

    per_copy = sum(t.numel() * t.element_size() for k, t in base.items()
                   if k in ("draft", "target")) + sum(
        t[0].numel() * t[0].element_size() for k, t in base.items()
        if k in ("q", "k_cache", "v_cache", "k_tree", "v_tree"))
    R = max(2, min(64, int(np.ceil(3 * L2_BYTES / per_copy))))  # > 3x the L2 together

    def clone(src):
        return {k: ([t.clone() for t in v] if isinstance(v, list) else v.clone())
                for k, v in src.items()}

    copies = [base] + [clone(base) for _ in range(R - 1)]
    rounds = [Round(ops, w, c, dev, ws) for c in copies]
    for r in rounds:  # eager warm-up outside capture (sets function attributes)
        r.run()
    torch.cuda.synchronize()
    ops.ddtree_device_check()
    if args.profile_rounds:
        for i in range(args.profile_rounds):
            rounds[i % R].run()
        torch.cuda.synchronize()
        ops.ddtree_device_check()
        return {"profile_only": True, "w": w, "R": R}

    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    g_all = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_all, stream=stream):
        for r in rounds:
            r.run()
    g_one = []
    for r in rounds:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            r.run()
        g_one.append(g)

    def replay(n):
        for _ in range(n // R):
            g_all.replay()
        for c in range(n % R):
            g_one[c].replay()

    replay(max(args.warmup, 3) * 1)
    torch.cuda.synchronize()
    # sustained pre-run so that the clock samples see the GPU under this load
    sampler = ClockSampler(torch.cuda.current_device() if dev.index is None else dev.index)
    with sampler:
        t_end = time.time() + 1.5
        while time.time() < t_end:
            replay(R * 16)
            torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        replay(args.steps)
        e1.record()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    ms_total = e0.elapsed_time(e1)
    clocks = sampler.summary()

    # Every call of the round, and the calls outside it, timed alone: a captured
    # graph of M back-to-back launches of that call over rotating copies of its
    # own inputs (together > 3x the L2), CUDA events around the whole replay,
    # per launch = total / M.  As in the round, programmatic dependent launch
    # lets a launch's set-up overlap the previous launch's tail, and no event
    # sits between launches to add its latency.
    stage = {}
    try:
        stage = stage_times(ops, w, base, copies, rounds, ws, dev, stream, args.steps)
    except Exception as e:  # noqa: BLE001
        stage = {"unavailable": repr(e)}

    # 36-layer round: 36 tree-attention launches, each on its own KV cache
    x36 = None
    if not args.no_x36:
        layers = X36
        cache_bytes = 2 * base["k_cache"][0].numel() * 2
        if cache_bytes * layers < 40 * 2**30:
            lay = dict(base)
            for k in ("q", "k_cache", "v_cache", "k_tree", "v_tree"):
                lay[k] = [base[k][0]] + [base[k][0].clone() for _ in range(layers - 1)]
            r36 = Round(ops, w, lay, dev, ws, layers=layers)
            r36.run(layers)
            torch.cuda.synchronize()
            g36 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g36, stream=stream):
                r36.run(layers)
            for _ in range(3):
                g36.replay()
            torch.cuda.synchronize()
            n36 = max(10, min(200, args.steps // 10))
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record()
            for _ in range(n36):
                g36.replay()
            a1.record()
            torch.cuda.synchronize()
            ms36 = a0.elapsed_time(a1) / n36
            x36 = {"rounds_per_s": w.B * 1000.0 / ms36, "ms_per_round": ms36, "steps": n36,
                   "layers": layers}
            del r36, lay

    # end to end through the public API, inputs from pinned host memory
    e2e = None
    if not args.no_e2e:
        def host_t(a):
            a = np.ascontiguousarray(a)
            return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).pin_memory()

        pin = {k: host_t(h[k]) for k in ("draft", "target", "q", "k_tree", "v_tree", "bonus",
                                         "prefix_len")}
        # two input sets: step s+1's inputs are copied on a second stream while
        # step s computes; the host reads every step's outputs, and reuses a
        # pinned output buffer only after it has read the previous step's
        sets = [copies[0], copies[1]]
        out_pin = [{k: torch.empty(rounds[0].acc[k].shape, dtype=torch.int32).pin_memory()
                    for k in ("accept_len", "out_tokens", "next_bonus")} for _ in range(2)]
        cps = torch.cuda.Stream(device=dev)
        comp_cap = torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        used = [False, False]
        got = []

        def h2d(dst_t, src):
            d = dst_t.view(torch.int16) if dst_t.dtype == torch.bfloat16 else dst_t
            d.copy_(src.view(d.shape), non_blocking=True)

        h2d_bytes = sum(t.numel() * t.element_size() for t in pin.values())
        d2h_bytes = sum(t.numel() * t.element_size() for t in out_pin[0].values())

        # every step's work captured once per input set: the copies in (on the
        # copy stream) and the round with its outputs copied out (on the compute
        # stream), so that a step costs the host a few calls
        g_copy, g_round = [], []
        for i in range(2):
            gc = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gc, stream=cps):
                for k in ("draft", "target", "bonus", "prefix_len"):
                    h2d(sets[i][k], pin[k])
                for k in ("q", "k_tree", "v_tree"):
                    h2d(sets[i][k][0], pin[k])
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=comp_cap):
                rounds[i].run()
                for k, t in out_pin[i].items():
                    t.copy_(rounds[i].acc[k], non_blocking=True)
            g_copy.append(gc)
            g_round.append(gr)
        torch.cuda.synchronize()

        def e2e_step(step):
            i = step & 1
            if used[i]:
                ev_out[i].synchronize()  # this set's previous outputs are on the host
                got.append(int(out_pin[i]["accept_len"][0]))
                cps.wait_event(ev_out[i])  # ... and the round that read its inputs is done
            with torch.cuda.stream(cps):
                g_copy[i].replay()
                ev_in[i].record(cps)
            with torch.cuda.stream(comp_cap):
                comp_cap.wait_event(ev_in[i])
                g_round[i].replay()
                ev_out[i].record(comp_cap)
            used[i] = True

        def drain():
            for i in range(2):
                if used[i]:
                    ev_out[i].synchronize()
                    got.append(int(out_pin[i]["accept_len"][0]))
                    used[i] = False

        for st in range(max(4, args.warmup // 4)):
            e2e_step(st)
        drain()
        n_e2e = max(20, min(500, args.steps // 4))
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for st in range(n_e2e):
            e2e_step(st)
        drain()
        t1 = time.perf_counter()
        assert len(set(got)) == 1, "every step reads the same inputs, so the same result"
        e2e = {"value": w.B * n_e2e / (t1 - t0), "unit": "rounds/s",
               "h2d_bytes_per_step": int(h2d_bytes), "d2h_bytes_per_step": int(d2h_bytes),
               "steps": n_e2e,
               "note": "public Python API (ops.*) over the C ABI; every step copies its inputs "
                       "in from pinned host memory (on a second stream, overlapping the "
                       "previous step's round) and its accept outputs out, which the host "
                       "reads; the KV cache is device-resident state"}

    ops.ddtree_device_check()
    tree_anc = int(np.sum([bin(int(x)).count("1") for x in
                           rounds[0].tree["anc_mask"].cpu().numpy().view(np.uint32).ravel()]))
    return {"w": w, "ms_total": ms_total, "R": R, "per_copy": per_copy, "clocks": clocks,
            "stage": stage, "x36": x36, "e2e": e2e, "tree_anc": tree_anc}


# ---------------------------------------------------------------------------
# the CPU oracle (reported baseline; also the `--impl reference` arm)
# ---------------------------------------------------------------------------

# Key-head rows of fp64 tree attention one host core is given per oracle step
# (one key row against one query head: ~0.2-0.3 us on the hosts measured), so
# a step's attention takes about a second on every core.
ORACLE_ROWS_PER_CORE = 1 << 22


def host_cores() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def oracle_setup(w):
    import oracle
    h = host_inputs(w)
    draft = wl.draft_logits(w)
    idx, _, lp32, _ = oracle.topk(draft, w.dtype, w.K)
    tree = oracle.build_tree(lp32, idx, h["bonus"], h["prefix_len"], w.N)
    h["target"] = wl.target_logits(w, draft, tree["depth"])
    return oracle, h, tree


def oracle_attn_tasks(w, n_nodes, cores):
    """The tree-attention work of one oracle step, as (b, kv_head, u_lo, u_hi)
    tasks, with its size and the full layer's size in key-head rows (one key
    against one query head).  The whole layer when it fits the per-core budget,
    else a seeded uniform sample of single node rows (b, g, u) that does."""
    G = w.Hq // w.Hkv
    row_cost = [G * (w.P[b] + int(n_nodes[b]) + 1) for b in range(w.B)]
    total = sum(w.Hkv * (int(n_nodes[b]) + 1) * row_cost[b] for b in range(w.B))
    budget = cores * ORACLE_ROWS_PER_CORE
    if total <= budget:
        return [(b, g, 0, w.N + 1) for b in range(w.B) for g in range(w.Hkv)], total, total
    rows = [(b, g, u) for b in range(w.B) for g in range(w.Hkv) for u in range(int(n_nodes[b]) + 1)]
    order = np.random.default_rng(0x0AC1E).permutation(len(rows))
    tasks, done = [], 0
    for i in order:
        b, g, u = rows[i]
        if done + row_cost[b] > budget and len(tasks) >= cores:
            break
        tasks.append((b, g, u, u + 1))
        done += row_cost[b]
    return tasks, done, total


def oracle_step(o, w, h, tasks, cores):
    """One round of the oracle: top-K, heap and walk over the whole batch, tree
    attention on `tasks` spread over `cores` host threads.  Returns the four
    stage times (s)."""
    t0 = time.perf_counter()
    idx, _, lp32, _ = o.topk(h["draft"].reshape(w.B, w.L, w.V), w.dtype, w.K)
    t1 = time.perf_counter()
    tree = o.build_tree(lp32, idx, h["bonus"], h["prefix_len"], w.N)
    t2 = time.perf_counter()
    o.tree_attn_tasks(h["q"], h["k_cache"], h["v_cache"], h["k_tree"], h["v_tree"],
                      h["prefix_len"], tree["n_nodes"], tree["anc_mask"], tasks, threads=cores)
    t3 = time.perf_counter()
    o.accept(h["target"], w.dtype, tree, w.L, temperature=w.T, seed=wl.philox_seed(w))
    t4 = time.perf_counter()
    return np.array([t1 - t0, t2 - t1, t3 - t2, t4 - t3])


def oracle_summary(w, stage_s, done_rows, total_rows, cores, steps):
    """The measured oracle step and, separately, a full round extrapolated from
    it (attention time scaled by the unsampled share of its key-head rows)."""
    per = stage_s.mean(axis=0)
    step_s = float(per.sum())
    full_s = float(per[0] + per[1] + per[2] * total_rows / done_rows + per[3])
    frac = done_rows / total_rows
    if done_rows == total_rows:
        sample = (f"{steps} full rounds of '{w.name}' (all B = {w.B} sequences): top-K, heap and "
                  f"walk on 1 core, tree attention over (sequence, KV head) units on {cores} "
                  f"host threads")
    else:
        sample = (f"{steps} rounds of '{w.name}' (all B = {w.B} sequences): top-K, heap and walk "
                  f"in full on 1 core; tree attention on a seeded sample of node rows "
                  f"({100 * frac:.3g} % of the layer's key-head rows) on {cores} host threads; "
                  f"value counts these sampled rounds")
    return {"value": w.B / step_s, "unit": "rounds/s", "cores": cores, "kind": "oracle",
            "sample": sample, "seconds_per_step": step_s,
            "stage_seconds": {k: float(v) for k, v in zip(("topk", "build", "tree_attn", "accept"),
                                                          per)},
            "attn_fraction_of_layer": frac,
            "full_round_extrapolated": {"seconds": full_s, "rounds_per_s": w.B / full_s,
                                        "method": "attention time x (layer's key-head rows / "
                                                  "sampled ones); other stages as measured"}}


def cpu_baseline(w, seconds, steps=None):
    o, h, tree = oracle_setup(w)
    cores = host_cores()
    tasks, done, total = oracle_attn_tasks(w, tree["n_nodes"], cores)
    times = []
    t_start = time.perf_counter()
    while True:
        times.append(oracle_step(o, w, h, tasks, cores))
        if steps is not None and len(times) >= steps:
            break
        if steps is None and (time.perf_counter() - t_start > seconds or len(times) >= 50):
            break
    return oracle_summary(w, np.array(times), done, total, cores, len(times))


def reference_arm(args, rank, world):
    """`--impl reference`: the oracle, as it stands, timed on the host cores on
    the GPU arm's workload, metric, unit and direction.  Each step is one
    oracle round (sampled attention on the large shapes); `ms_per_step` and
    `value` are those measured steps; a full round's extrapolated time is in
    its own field."""
    w = wl.CONFIGS[args.workload]
    if rank != 0:
        return
    o, h, tree = oracle_setup(w)
    cores = host_cores()
    tasks, done, total = oracle_attn_tasks(w, tree["n_nodes"], cores)
    for _ in range(args.warmup):
        oracle_step(o, w, h, tasks, cores)
    t0 = time.perf_counter()
    st = np.array([oracle_step(o, w, h, tasks, cores) for _ in range(args.steps)])
    wall = time.perf_counter() - t0
    summ = oracle_summary(w, st, done, total, cores, args.steps)
    ms_step = wall * 1e3 / args.steps
    value = w.B * args.steps / wall
    summ["value"] = value
    line = {"impl": "reference", "metric": METRIC,
            "value": value, "unit": "rounds/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w), "cpu_baseline": summ,
            "full_round_extrapolated": summ["full_round_extrapolated"],
            "e2e": {"value": value, "unit": "rounds/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def aggregate_replicas(ms_local: float, world: int, B: int, steps: int, device):
    """Replicas: every rank ran `steps` rounds of B sequences on its own GPU.
    The job's time is the slowest rank's; its throughput counts every rank's
    sequences.  Returns (max milliseconds over ranks, sequence-rounds per second)."""
    ms = ms_local
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * B * steps / (ms / 1e3)


# How the timed steps keep the L2 from serving their inputs (both arms print
# the same config; the GPU arm's number of input copies is in `input_copies`).
L2_POLICY = ("per-step inputs rotated over copies that together exceed 3x the 129 MB L2, "
             "so no step reads its inputs from L2")


def config_of(w):
    return {"workload": w.name, "B": w.B, "L": w.L, "V": w.V, "K": w.K, "N": w.N,
            "P": list(w.P) if len(set(w.P)) > 1 else w.P[0], "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
            "temperature": w.T, "layers": 1, "walk": walk_for(w), "l2": L2_POLICY}


def acceptance_stats(rounds: int) -> dict:
    """Acceptance length against the node budget on the budget-sweep shape
    (L = 16, V = 151936, bf16, greedy), plus the vanilla chain (K = 1, N = L):
    a synthetic analogue of the pages' acceptance-vs-budget study (§5).  Every
    round draws fresh draft logits (3 N(0,1) + a +6 spike per position) and
    target rows (the draft row at the node's depth + N(0,1)) on the device and
    runs top-K -> build -> accept through the library.  Also reports the
    surrogate of §4.2, sum over drafted nodes of exp(score): the expected
    accepted length if the target followed the factorised draft exactly."""
    import torch
    from diffusion_draft_tree_gb300 import ops

    dev = torch.device("cuda", 0)
    base = wl.CONFIGS["budget_sweep_n512"]
    L, V = base.L, base.V
    out = {"metric": "acceptance length (accepted draft tokens per round)", "rounds": rounds,
           "shape": {"L": L, "V": V, "draft": "3*N(0,1) + 6 spike", "target": "draft row at "
                     "depth + N(0,1)", "temperature": 0.0}, "budgets": {}}
    for label, K, N in [("chain K=1 N=16", 1, 16), ("N=32", 16, 32), ("N=64", 16, 64),
                        ("N=128", 16, 128), ("N=256", 16, 256), ("N=512", 16, 512),
                        ("N=1024", 16, 1024)]:
        g = torch.Generator(device=dev)
        g.manual_seed(0xACC + 7919 * K + N)
        lens, surr = [], []
        bonus = torch.zeros(1, dtype=torch.int32, device=dev)
        plen = torch.zeros(1, dtype=torch.int32, device=dev)
        for _ in range(rounds):
            d32 = torch.randn((L, V), generator=g, device=dev) * 3.0
            spike = torch.randint(0, V, (L,), generator=g, device=dev)
            d32[torch.arange(L, device=dev), spike] += 6.0
            draft = d32.to(torch.bfloat16)
            idx, lp, _ = ops.topk(draft, K)
            tree = ops.build(lp.view(1, L, K), idx.view(1, L, K), bonus, plen, N)
            depth = tree["depth"][0].long()
            rows = draft.float()[depth.clamp(min=0).clamp(max=L - 1)]
            noise = torch.randn(rows.shape, generator=g, device=dev)
            target = (rows + noise).to(torch.bfloat16)[None]
            acc = ops.accept(target, tree, L)
            lens.append(int(acc["accept_len"][0].item()))
            n = int(tree["n_nodes"][0].item())
            surr.append(float(torch.exp(tree["score"][0, 1:n + 1].double()).sum().item()))
        ops.ddtree_device_check()
        a = np.array(lens)
        entry = {"K": K, "N": N, "mean_accept_len": float(a.mean()),
                 "tokens_per_round": float(a.mean() + 1), "std": float(a.std()),
                 "surrogate_mean": float(np.mean(surr))}
        if N in (512, 16):
            entry["histogram"] = [int((a == k).sum()) for k in range(L + 1)]
        out["budgets"][label] = entry
    return out


def profile_call(call: str, workload: str, batch=None) -> dict:
    """Runs one call of the round three times on the workload's inputs (the
    tree from the library's own top-K and build), for a kernel profiler."""
    import torch
    from diffusion_draft_tree_gb300 import ops

    w = wl.CONFIGS[workload]
    if batch is not None:
        w = w.with_(B=batch, P=tuple(w.P[:batch]))
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(
        torch.bfloat16)
    draft = wl.draft_logits(w)
    d = to_dev_logits(draft.reshape(w.B * w.L, w.V), w.dtype, dev)
    idx, lp, _ = ops.topk(d, w.K)
    bonus, plen = i32(wl.bonus_tokens(w)), i32(wl.prefix_lengths(w))
    tree = ops.build(lp.view(w.B, w.L, w.K), idx.view(w.B, w.L, w.K), bonus, plen, w.N)
    torch.cuda.synchronize()
    if call == "topk":
        ws = ops.alloc_workspace(ops.workspace_size(ops.OP_TOPK, B=w.B, L=w.L, V=w.V, K=w.K,
                                                    dtype=w.dtype), dev)
        run = lambda: ops.topk(d, w.K, workspace=ws)
    elif call == "build":
        run = lambda: ops.build(lp.view(w.B, w.L, w.K), idx.view(w.B, w.L, w.K), bonus, plen, w.N)
    elif call == "tree_attn":
        q, kc, vc = bf(wl.queries(w)), bf(wl.kv_cache(w, 0)), bf(wl.kv_cache(w, 1))
        kt, vt = bf(wl.kv_tree(w, 0)), bf(wl.kv_tree(w, 1))
        ws = ops.alloc_workspace(ops.workspace_size(ops.OP_TREE_ATTN, B=w.B, N=w.N, Hq=w.Hq,
                                                    Hkv=w.Hkv, D=w.D, cache_cap=w.P_cap), dev)
        run = lambda: ops.tree_attn(q, kc, vc, kt, vt, plen, tree["n_nodes"], tree["anc_mask"],
                                    workspace=ws)
    else:
        tgt = to_dev_logits(wl.target_logits(w, draft, tree["depth"].cpu().numpy()), w.dtype, dev)
        ws = ops.alloc_workspace(ops.workspace_size(ops.OP_ACCEPT, B=w.B, N=w.N, V=w.V,
                                                    dtype=w.dtype), dev)
        if call == "accept":
            run = lambda: ops.accept(tgt, tree, w.L, temperature=w.T, seed=wl.philox_seed(w),
                                     workspace=ws)
        else:
            run = lambda: ops.accept_path(tgt, tree, w.L, temperature=w.T, seed=wl.philox_seed(w))
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    ops.ddtree_device_check()
    return {"profile_call": call, "workload": w.name, "B": w.B}


WALK = "auto"  # step 4 of the timed round (--walk)


def walk_for(w) -> str:
    """The walk the round uses: measured on the workloads, the path-only walk
    (a dependent chain of rows) gives the faster round once the batch's trees
    hold 32 rows or more (8b_single 44.2 -> 40.4 us a round, N = 32 55.5 ->
    50.5 us, N = 64 65.7 -> 59.2 us; larger trees gain more); the full-tree
    walk (every row at once) only for the tiniest trees, where it is also the
    faster call alone."""
    if WALK != "auto":
        return WALK
    return "path" if w.B * (w.N + 1) >= 32 else "full"


def kernel_report(w, model, stage, peaks):
    """Per-call achieved rates from the stage times, and the roofline object of
    the dominant call (tree attention), its bound chosen from its arithmetic
    intensity against the measured peaks."""
    kernels = {}
    if "unavailable" in stage:
        return {"unavailable": stage["unavailable"]}, None
    path_bytes = stage["path_rows"] * w.V * w.esize
    full_bytes = w.B * (w.N + 1) * w.V * w.esize
    if walk_for(w) == "path":  # the round's step 4 reads the path's rows only
        model = dict(model, accept={"bytes": path_bytes})
    model = dict(model, accept_path={"bytes": path_bytes}, accept_full={"bytes": full_bytes},
                 commit={"bytes": 8 * stage.get("commit_rows", 0) * w.Hkv * w.D})
    notes = {"accept": f"step 4 of the round: the {walk_for(w)} walk",
             "accept_path": "step 4 reading only the accepted path's rows (bytes = "
                            "(accept_len + 1) x V x elem per sequence); outside the round",
             "accept_full": "step 4 resolving every tree row (bytes = (N + 1) x V x elem per "
                            "sequence); outside the round",
             "commit": "after the round, not in its metric: the accepted path's K/V rows "
                       "into the cache"}
    for n in ("topk", "build", "tree_attn", "accept", "accept_path", "accept_full", "commit"):
        st = stage.get(n) or {}
        if "ms" not in st:
            kernels[n] = st
            continue
        ms = st["ms"]
        k = {"ms": ms, "launches_timed": st["launches"], "input_copies": st["input_copies"]}
        if "bytes" in model[n]:
            k["bytes"] = model[n]["bytes"]
            k["GBps"] = model[n]["bytes"] / (ms * 1e-3) / 1e9
            k["hbm_frac"] = k["GBps"] / peaks["hbm_gbs"]
        if "flops" in model[n]:
            k["flops"] = model[n]["flops"]
            k["TFLOPps"] = model[n]["flops"] / (ms * 1e-3) / 1e12
            k["tensor_frac"] = k["TFLOPps"] / peaks["bf16_tflops"]
        if n in notes:
            k["note"] = notes[n]
        if n.startswith("accept_"):
            k["same_tokens_as_other_walk"] = stage.get("same_tokens")
        kernels[n] = k
    a = model["tree_attn"]
    ams = kernels["tree_attn"]["ms"]
    t_hbm = a["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = a["flops"] / (peaks["bf16_tflops"] * 1e12)
    if t_tc >= t_hbm:
        roof = {"kernel": "tree_attn", "bound": "tensor",
                "achieved": a["flops"] / (ams * 1e-3) / 1e12, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    else:
        roof = {"kernel": "tree_attn", "bound": "hbm", "achieved": a["bytes"] / (ams * 1e-3) / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = measured_traffic("tree_attn", w.name)
    roof["peak_source"] = f"{peaks['source']} (MEASURED_PEAKS.json burst figure), of measured"
    roof["algorithmic_bytes"] = a["bytes"]
    roof["algorithmic_flops"] = a["flops"]
    roof["duration_ms"] = ams
    return kernels, roof


def main():
    global WALK
    args = parse()
    WALK = args.walk
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
    if world > 1 and "RANK" not in os.environ:
        world = 1
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return
    if args.acceptance_stats:
        if rank == 0:
            print(json.dumps(acceptance_stats(args.acceptance_stats)), flush=True)
        return
    if args.profile_call:
        print(json.dumps(profile_call(args.profile_call, args.workload, args.batch)), flush=True)
        return
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        local = int(os.environ.get("LOCAL_RANK", rank))
        dev = torch.device("cuda", local)
    else:
        dev = torch.device("cuda", 0)
    res = gpu_arm(args, rank, world, dev)
    w = res["w"]
    if res.get("profile_only"):
        if rank == 0:
            print(json.dumps({"profile_rounds": args.profile_rounds, "workload": w.name,
                              "copies": res["R"]}), flush=True)
        return
    ms_total, value = aggregate_replicas(res["ms_total"], world, w.B, args.steps, dev)
    ms_step = ms_total / args.steps
    peaks = load_peaks()
    model = work_model(w, res["tree_anc"])
    kernels, roof = kernel_report(w, model, res["stage"], peaks)
    ms_sum = sum(kernels[n]["ms"] for n in ("topk", "build", "tree_attn", "accept")
                 if "ms" in kernels.get(n, {}))
    line = {"metric": METRIC,
            "value": value, "unit": "rounds/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(w), "roofline": roof, "kernels": kernels,
            "kernel_timing": STAGE_METHOD, "round_calls_ms_sum": ms_sum,
            "input_copies": res["R"], "gpu_launches": LAUNCHES_PER_ROUND * args.steps,
            "clocks": res["clocks"], "e2e": res["e2e"]}
    if res["x36"]:
        line["rounds_per_s_x36_layers"] = res["x36"]["rounds_per_s"] * world
        line["x36"] = res["x36"]
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
