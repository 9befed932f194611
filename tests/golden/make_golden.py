"""Writes tests/golden/tiny_round.json: the oracle's results for the tiny
workload (1 sequence, L=4, V=1000, K=4, N=16, P=64, 2 query heads / 1 KV head,
D=64, greedy).  Expected values come from ``oracle`` alone; inputs come from
the seeded generator.  Re-run only when the oracle's arithmetic changes for a
reason the pages justify.
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from diffusion_draft_tree_gb300 import workloads as wl  # noqa: E402


def tiny_round():
    w = wl.CONFIGS["tiny"]
    d = wl.draft_logits(w)
    idx, lp64, lp32, lse = oracle.topk(d, w.dtype, w.K)
    t = oracle.build_tree(lp32, idx, wl.bonus_tokens(w), wl.prefix_lengths(w), w.N)
    x = wl.target_logits(w, d, t["depth"])
    acc = oracle.accept(x, w.dtype, t, L=w.L)
    return {
        "workload": w.name,
        "topk_idx": idx.tolist(),
        "topk_logp": [[[float(v) for v in r] for r in b] for b in lp64],
        "lse": lse.tolist(),
        "tree": {k: t[k].tolist() for k in ("parent", "depth", "rank", "token", "pos_id",
                                             "child_count", "n_nodes")},
        "score": [[float(v) for v in r] for r in t["score"]],
        "anc_mask": t["anc_mask"].tolist(),
        "accept": {k: acc[k].tolist() for k in ("target_token", "accept_len", "accepted_nodes",
                                                 "out_tokens", "next_bonus")},
    }


if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_round.json")
    with open(out, "w") as f:
        json.dump(tiny_round(), f, indent=1)
    print("wrote", out)
