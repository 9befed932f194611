"""Throughput of one DDTree round on GB300: top-K -> heap build -> tree
attention (one target layer) -> acceptance walk, through libddtree.so.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gb300|reference]

Prints ONE JSON line (rank 0).  `value` is sequence-rounds per second with all
inputs resident in HBM; a "step" is one round over one batch.  The round's four
C-ABI calls are captured in CUDA graphs; to keep the 129 MB L2 from serving a
step's inputs, steps rotate over R copies of every per-step input (R copies
> 2x L2).  `e2e` repeats the measurement through the public API from pinned
host buffers (inputs copied in and results copied out every step).
`--impl reference` times the CPU oracle on the host cores instead (a reported
baseline; it runs a bounded sample of the same workload per step).
Multi-GPU runs are independent replicas (sequences are independent units).
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
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="8b_single", choices=sorted(wl.CONFIGS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-x36", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--walk", default="auto", choices=["auto", "full", "path"],
                    help="step 4: the full-tree walk (ddtree_accept), the path-only walk "
                         "(ddtree_accept_path), or auto: the path-only walk once the batch "
                         "has >= 128 tree rows, B (N + 1)")
    ap.add_argument("--acceptance-stats", type=int, default=0, metavar="ROUNDS",
                    help="instead of timing: run ROUNDS independent synthetic rounds per node "
                         "budget (and the K = 1 chain) and report acceptance lengths")
    ap.add_argument("--profile-rounds", type=int, default=0,
                    help="only run this many eager rounds (rotating input copies) and exit; "
                         "for kernel profilers")
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
    ncu capture recorded in profiles/traffic.md for this kernel and workload, or
    None if there is none or the kernel's sources changed since."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(kernel)
    for line in open(path):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) >= 4 and cells[0] == kernel and cells[1] == workload and cells[3] == want:
            try:
                return int(cells[2])
            except ValueError:
                return None
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
    R = max(2, min(64, int(np.ceil(3 * L2_BYTES / per_copy))))

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

    # per-kernel durations: external event nodes inside a captured graph
    kern = {}
    try:
        evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(5)]
               for _ in range(R)]
        g_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_ev, stream=stream):
            for r, ev in zip(rounds, evs):
                st = r.stages()
                for i in range(4):
                    ev[i].record()
                    st[i]()
                ev[4].record()
        acc = np.zeros(4)
        reps = max(4, min(200, args.steps // R))
        for _ in range(reps):
            g_ev.replay()
            torch.cuda.synchronize()
            for ev in evs:
                acc += [ev[i].elapsed_time(ev[i + 1]) for i in range(4)]
        kern_ms = acc / (reps * R)
        kern_method = "external CUDA events between the four kernels inside the graph"
    except Exception as e:  # noqa: BLE001
        kern_ms = np.full(4, np.nan)
        kern_method = f"unavailable: {e!r}"

    # the step after the round: commit the accepted path to the KV cache (not
    # part of the round's metric; timed alone, prefix lengths restored first)
    commit = None
    try:
        r0 = rounds[0]
        cap2 = w.P_cap + w.L + 1
        kc2 = torch.empty((w.B, w.Hkv, cap2, w.D), dtype=torch.bfloat16, device=dev)
        vc2 = torch.empty_like(kc2)
        plen0 = base["prefix_len"]
        plen = plen0.clone()
        n_c = 20
        c_ev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
                for _ in range(n_c)]

        def commit_once(ev):
            plen.copy_(plen0)
            ev[0].record()
            ops.ddtree_commit(kc2, vc2, base["k_tree"][0], base["v_tree"][0],
                              r0.acc["accept_len"], r0.acc["accepted_nodes"], plen)
            ev[1].record()

        commit_once(c_ev[0])
        torch.cuda.synchronize()
        g_c = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_c, stream=stream):
            for ev in c_ev:
                commit_once(ev)
        t_c = 0.0
        for _ in range(5):
            g_c.replay()
            torch.cuda.synchronize()
            t_c += sum(ev[0].elapsed_time(ev[1]) for ev in c_ev)
        n_c *= 5
        ops.ddtree_device_check()
        rows = int(r0.acc["accept_len"].sum().item()) + w.B
        commit = {"ms": t_c / n_c, "bytes": 8 * rows * w.Hkv * w.D}
        del kc2, vc2
    except Exception as e:  # noqa: BLE001
        commit = {"unavailable": repr(e)}

    # the path-only walk on the same round's tree and target rows (an alternative
    # to the full-tree accept; timed alone, not in the round's metric)
    # both step-4 walks timed alone on the same round's tree and target rows
    # (whichever the round uses), and their emitted tokens compared
    walks = {}
    try:
        r0 = rounds[0]
        outs = {"path": ops.accept_buffers(w.B, w.L, w.N, dev),
                "full": ops.accept_buffers(w.B, w.L, w.N, dev)}

        def run_walk(kind):
            if kind == "path":
                ops.ddtree_accept_path(r0.inp["target"], r0.tree["parent"], r0.tree["token"],
                                       r0.tree["n_nodes"], w.L, outs[kind], w.T,
                                       wl.philox_seed(w), 0)
            else:
                ops.ddtree_accept(r0.inp["target"], r0.tree["parent"], r0.tree["token"],
                                  r0.tree["n_nodes"], w.L, outs[kind], w.T, wl.philox_seed(w), 0,
                                  ws["accept"])

        for kind in ("path", "full"):
            n_p = 20
            p_ev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
                    for _ in range(n_p)]

            def once(ev):
                ev[0].record()
                run_walk(kind)
                ev[1].record()

            once(p_ev[0])
            torch.cuda.synchronize()
            g_p = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_p, stream=stream):
                for ev in p_ev:
                    once(ev)
            t_p = 0.0
            for _ in range(5):
                g_p.replay()
                torch.cuda.synchronize()
                t_p += sum(ev[0].elapsed_time(ev[1]) for ev in p_ev)
            ops.ddtree_device_check()
            walks[kind] = {"ms": t_p / (5 * n_p)}
        same = bool(torch.equal(outs["path"]["out_tokens"], outs["full"]["out_tokens"]))
        rows = int(outs["path"]["accept_len"].sum().item()) + w.B
        walks["path"]["bytes"] = rows * w.V * w.esize
        walks["full"]["bytes"] = w.B * (w.N + 1) * w.V * w.esize
        walks["same_tokens"] = same
        del outs
    except Exception as e:  # noqa: BLE001
        walks = {"unavailable": repr(e)}

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
            "kern_ms": kern_ms, "kern_method": kern_method, "x36": x36, "e2e": e2e,
            "commit": commit, "walks": walks,
            "tree_anc": tree_anc}


# ---------------------------------------------------------------------------
# the CPU oracle (reported baseline; also the `--impl reference` arm)
# ---------------------------------------------------------------------------

def oracle_step(o, w, h, attn_units):
    t0 = time.perf_counter()
    idx, _, lp32, _ = o.topk(h["draft"].reshape(w.B, w.L, w.V), w.dtype, w.K)
    t1 = time.perf_counter()
    tree = o.build_tree(lp32, idx, h["bonus"], h["prefix_len"], w.N)
    t2 = time.perf_counter()
    o.tree_attn(h["q"], h["k_cache"], h["v_cache"], h["k_tree"], h["v_tree"], h["prefix_len"],
                tree["n_nodes"], tree["anc_mask"], units=attn_units)
    t3 = time.perf_counter()
    o.accept(h["target"], w.dtype, tree, w.L, temperature=w.T, seed=wl.philox_seed(w))
    t4 = time.perf_counter()
    scale_attn = (w.B * w.Hkv) / len(attn_units)
    return (t1 - t0) + (t2 - t1) + (t3 - t2) * scale_attn + (t4 - t3)


def oracle_setup(w):
    import oracle
    h = host_inputs(w)
    draft = wl.draft_logits(w)
    idx, _, lp32, _ = oracle.topk(draft, w.dtype, w.K)
    tree = oracle.build_tree(lp32, idx, h["bonus"], h["prefix_len"], w.N)
    h["target"] = wl.target_logits(w, draft, tree["depth"])
    return oracle, h


def cpu_baseline(w, seconds, steps=None):
    o, h = oracle_setup(w)
    units = [(0, 0)]  # one (sequence, KV head) unit of tree attention per step, scaled up
    times = []
    t_start = time.perf_counter()
    while True:
        times.append(oracle_step(o, w, h, units))
        if steps is not None and len(times) >= steps:
            break
        if steps is None and (time.perf_counter() - t_start > seconds or len(times) >= 50):
            break
    per_step = float(np.mean(times))
    sample = (f"{len(times)} rounds of '{w.name}': top-K, heap and walk in full; tree attention "
              f"on 1 of {w.B * w.Hkv} (sequence, KV head) units, time scaled x{w.B * w.Hkv}")
    return {"value": w.B / per_step, "unit": "rounds/s", "cores": 1, "kind": "oracle",
            "sample": sample, "seconds_per_round": per_step}


def reference_arm(args, rank, world):
    w = wl.CONFIGS[args.workload]
    if rank != 0:
        return
    o, h = oracle_setup(w)
    units = [(0, 0)]
    for _ in range(args.warmup):
        oracle_step(o, w, h, units)
    t = [oracle_step(o, w, h, units) for _ in range(args.steps)]
    per_step = float(np.mean(t))
    value = w.B / per_step
    sample = (f"each step: one round of '{w.name}' with tree attention on 1 of "
              f"{w.B * w.Hkv} (sequence, KV head) units, time scaled x{w.B * w.Hkv}")
    line = {"impl": "reference", "metric": METRIC,
            "value": value, "unit": "rounds/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, None),
            "cpu_baseline": {"value": value, "unit": "rounds/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
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


def config_of(w, R):
    c = {"workload": w.name, "B": w.B, "L": w.L, "V": w.V, "K": w.K, "N": w.N,
         "P": list(w.P) if len(set(w.P)) > 1 else w.P[0], "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
         "temperature": w.T, "layers": 1, "walk": walk_for(w)}
    if R is not None:
        c["l2"] = f"inputs rotated over {R} copies per step (> 2x the 129 MB L2)"
    return c


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


WALK = "auto"  # step 4 of the timed round (--walk)


def walk_for(w) -> str:
    """The walk the round uses: measured on the five workloads, the path-only
    walk (a dependent chain of rows) is faster once the batch's trees hold
    128 rows or more (N = 128: 73 -> 66 us a round, ragged_serving 976 -> 736
    us), the full-tree walk (every row at once) below (8b_single: 40.1 vs
    40.5 us)."""
    if WALK != "auto":
        return WALK
    return "path" if w.B * (w.N + 1) >= 128 else "full"


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
    wk = res.get("walks") or {}
    if walk_for(w) == "path" and "path" in wk:  # the round's step 4 reads the path's rows only
        model["accept"] = {"bytes": wk["path"]["bytes"]}
    names = ["topk", "build", "tree_attn", "accept"]
    kernels = {}
    for n, ms in zip(names, res["kern_ms"]):
        k = {"ms": float(ms)}
        if "bytes" in model[n]:
            k["GBps"] = model[n]["bytes"] / (ms * 1e-3) / 1e9
            k["hbm_frac"] = k["GBps"] / peaks["hbm_gbs"]
        if "flops" in model[n]:
            k["TFLOPps"] = model[n]["flops"] / (ms * 1e-3) / 1e12
            k["tensor_frac"] = k["TFLOPps"] / peaks["bf16_tflops"]
        kernels[n] = k
    c = res.get("commit")
    if c and "ms" in c:
        kernels["commit"] = {"ms": c["ms"], "GBps": c["bytes"] / (c["ms"] * 1e-3) / 1e9,
                             "hbm_frac": c["bytes"] / (c["ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"],
                             "note": "after the round, not in its metric: the accepted "
                                     "path's K/V rows into the cache"}
    wk = res.get("walks") or {}
    for kind in ("path", "full"):
        c = wk.get(kind)
        if c and "ms" in c:
            kernels["accept_" + kind] = {
                "ms": c["ms"], "GBps": c["bytes"] / (c["ms"] * 1e-3) / 1e9,
                "hbm_frac": c["bytes"] / (c["ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "same_tokens_as_other_walk": wk.get("same_tokens"),
                "note": ("step 4 reading only the accepted path's rows (bytes = (accept_len + 1)"
                         " x V x elem per sequence)" if kind == "path" else
                         "step 4 resolving every tree row (bytes = (N + 1) x V x elem per "
                         "sequence)") + "; timed alone, outside the round"}
    a = model["tree_attn"]
    t_hbm = a["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = a["flops"] / (peaks["bf16_tflops"] * 1e12)
    ams = float(res["kern_ms"][2])
    if t_tc >= t_hbm:
        roof = {"kernel": "tree_attn", "bound": "tensor", "achieved": a["flops"] / (ams * 1e-3) / 1e12,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    else:
        roof = {"kernel": "tree_attn", "bound": "hbm", "achieved": a["bytes"] / (ams * 1e-3) / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = measured_traffic("tree_attn", w.name)
    roof["peak_source"] = f"{peaks['source']} (MEASURED_PEAKS.json burst figure)"
    roof["algorithmic_bytes"] = a["bytes"]
    roof["algorithmic_flops"] = a["flops"]
    line = {"metric": METRIC,
            "value": value, "unit": "rounds/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(w, res["R"]), "roofline": roof, "kernels": kernels,
            "kernel_timing": res["kern_method"], "gpu_launches": LAUNCHES_PER_ROUND * args.steps,
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
