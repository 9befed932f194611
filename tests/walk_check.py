"""Test-side checks for step 4 at temperature > 0 (no GPU code here).

A sampled token is the smallest v with C_v > U*Z (C the running sum of
exp((x - max)/T) in token order).  The GPU sums in fp32 in another order
than the oracle's fp64, so where U*Z falls within rounding of a bin edge
the two may pick neighbouring tokens.  `sample_in_band` accepts a GPU token
only if its own CDF bin, computed here in fp64, lies within `band`*Z of U*Z:
that is, it is the oracle's token or the token across the nearby edge (tokens
of less mass than the band in between).  `walk` replays the acceptance walk
(DDTree §4.1) on given per-node tokens, so a sequence whose sampled tokens
differ from the oracle's inside the band is still compared, against the walk
those tokens imply.
"""
import numpy as np

import oracle
from diffusion_draft_tree_gb300 import workloads as wl


def row_f64(x, dtype, b, u):
    r = x[b, u]
    if dtype == wl.BF16:
        return wl.bf16_to_f32(np.ascontiguousarray(r)).astype(np.float64)
    return r.astype(np.float64)


def sample_in_band(row64, T, seed, step, b, u, tok, band):
    """Distance (over Z) from U*Z to the CDF bin [C_{tok-1}, C_tok] of `tok`,
    and whether it is within `band`."""
    p = np.exp((row64 - row64.max()) / T)
    c = np.cumsum(p)
    z = c[-1]
    tgt = oracle.uniform(seed, step, b, u) * z
    lo = c[tok - 1] if tok > 0 else 0.0
    hi = c[tok]
    dist = 0.0 if lo <= tgt <= hi else min(abs(tgt - lo), abs(tgt - hi))
    return dist / z, dist / z <= band


def walk(parent, token, n, tt, L):
    """The acceptance walk on per-node target tokens tt: from the root, move to
    the child whose token is tt[current] while one exists (at most L moves);
    the bonus is tt[last].  Returns the four walk outputs of one sequence."""
    acc = np.full(L, -1, np.int32)
    out = np.full(L + 1, -1, np.int32)
    cur, k = 0, 0
    while k < L:
        kids = [c for c in range(1, n + 1) if parent[c] == cur and token[c] == tt[cur]]
        if not kids:
            break
        cur = kids[0]
        acc[k] = cur
        out[k] = token[cur]
        k += 1
    out[k] = tt[cur]
    return {"accept_len": k, "accepted_nodes": acc, "out_tokens": out, "next_bonus": tt[cur]}
