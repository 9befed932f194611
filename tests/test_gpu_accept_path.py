"""GPU parity of the path-only acceptance walk (ddtree_accept_path) against the
oracle's walk.  Criteria: accepted length, accepted nodes, emitted tokens and
the bonus bit-exact; target_token equal to the oracle's on the root and the
accepted nodes and -1 on every other node.  At temperature > 0 a node's sample
may differ only where the oracle's U*Z lies within 1e-5*Z of a CDF boundary,
and the GPU's token must then be the one across that boundary (counted).  The
walk is compared for every sequence: against the oracle's where the path's
tokens agree, else against the walk the GPU's own path tokens imply (every
node it visits must carry a token, and none off its path)."""
import numpy as np
import pytest
import torch

import oracle
from diffusion_draft_tree_gb300 import ops
from diffusion_draft_tree_gb300 import workloads as wl
from tests import walk_check
from tests.gpu_util import dev_logits, host, tree_to_dev

pytestmark = pytest.mark.gpu
MARGIN = 1e-5
OUT_KEYS = ("accept_len", "accepted_nodes", "out_tokens", "next_bonus")


def _check(x, dtype, tree, L, T, seed, step, dev, unaligned=False):
    ref = oracle.accept(x, dtype, tree, L, temperature=T, seed=seed, step=step)
    dt = tree_to_dev(tree, dev)
    xd = dev_logits(x, dtype, dev)
    if unaligned:
        buf = torch.empty(xd.numel() + 1, dtype=xd.dtype, device=dev)
        buf[1:] = xd.reshape(-1)
        xd = buf[1:].view(xd.shape)
    got = ops.accept_path(xd, dt, L, temperature=T, seed=seed, step=step)
    ops.ddtree_device_check()
    tt = host(got["target_token"])
    outs = {k: host(got[k]) for k in OUT_KEYS}
    near = 0
    for b in range(x.shape[0]):
        n = int(tree["n_nodes"][b])
        # the GPU's own walk: the nodes it visited carry its tokens
        a = int(outs["accept_len"][b])
        path = [0] + [int(u) for u in outs["accepted_nodes"][b, :a]]
        assert all(0 <= u <= n for u in path), f"path of sequence {b} leaves the tree"
        off = np.ones(tt.shape[1], bool)
        off[path] = False
        assert np.all(tt[b, off] == -1), f"target token written off the path in sequence {b}"
        diff = [u for u in path if tt[b, u] != ref["target_token"][b, u]]
        for u in diff:
            assert T > 0, f"greedy target token differs in sequence {b} at node {u}"
            assert ref["margin"][b, u] < MARGIN, f"sample differs off-boundary ({b}, {u})"
            d, ok = walk_check.sample_in_band(walk_check.row_f64(x, dtype, b, u), T, seed, step,
                                              b, u, int(tt[b, u]), MARGIN)
            assert ok, f"GPU token of ({b}, {u}) is not across the nearby CDF edge ({d:.3g})"
        near += len(diff)
        if not diff:
            for k in OUT_KEYS:
                np.testing.assert_array_equal(outs[k][b], ref[k][b], err_msg=f"{k} of seq {b}")
        else:
            want = walk_check.walk(tree["parent"][b], tree["token"][b], n, tt[b], L)
            for k in OUT_KEYS:
                np.testing.assert_array_equal(outs[k][b], want[k], err_msg=f"{k} of seq {b}")
    return ref, near


def _tree(w):
    draft = wl.draft_logits(w)
    idx, _, lp32, _ = oracle.topk(draft, w.dtype, w.K)
    t = oracle.build_tree(lp32, idx, wl.bonus_tokens(w), wl.prefix_lengths(w), w.N)
    return draft, t


@pytest.mark.parametrize("name", ["tiny", "8b_single", "budget_sweep_n256", "long_context_70b",
                                  "ragged_serving"])
def test_accept_path_workloads(cuda_device, name):
    w = wl.CONFIGS[name]
    draft, t = _tree(w)
    x = wl.target_logits(w, draft, t["depth"])
    _, near = _check(x, w.dtype, t, w.L, w.T, wl.philox_seed(w), 0, cuda_device)
    if w.T > 0:
        print(f"{name}: {near} sampled path tokens differ, all inside the {MARGIN:g}*Z band")


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_accept_path_matches_full_tree_walk(cuda_device, T):
    """Both GPU walks on one input: identical accepted paths and tokens, and the
    path-only target tokens agree with the full-tree ones on the path."""
    w = wl.CONFIGS["8b_single"].with_(B=8, P=(2048,) * 8, T=T)
    draft, t = _tree(w)
    xh = wl.target_logits(w, draft, t["depth"])
    x = dev_logits(xh, w.dtype, cuda_device)
    dt = tree_to_dev(t, cuda_device)
    full = ops.accept(x, dt, w.L, temperature=T, seed=11, step=3)
    path = ops.accept_path(x, dt, w.L, temperature=T, seed=11, step=3)
    ops.ddtree_device_check()
    # the two walks may split only at a node whose oracle U*Z lies in the band
    ref = oracle.accept(xh, w.dtype, t, w.L, temperature=T, seed=11, step=3)
    tf_all, tp_all = host(full["target_token"]), host(path["target_token"])
    firm = np.ones(w.B, bool)
    for b in range(w.B):
        a = int(host(full["accept_len"])[b])
        for u in [0] + [int(v) for v in host(full["accepted_nodes"])[b, :a]]:
            if tp_all[b, u] != tf_all[b, u]:
                assert T > 0 and ref["margin"][b, u] < MARGIN, f"walks split in sequence {b}"
                firm[b] = False
                break
    print(f"T={T}: {w.B - firm.sum()} of {w.B} sequences split inside the band")
    for k in OUT_KEYS:
        np.testing.assert_array_equal(host(path[k])[firm], host(full[k])[firm], err_msg=k)
    tf, tp = host(full["target_token"])[firm], host(path["target_token"])[firm]
    on = tp >= 0
    np.testing.assert_array_equal(tp[on], tf[on])
    assert np.all(on.sum(1) == host(full["accept_len"])[firm] + 1)


def test_accept_path_planted_agreement_walks_rank0_chain(cuda_device):
    """Noise-free target on the 8B-class workload, greedy: the walk accepts the
    whole all-rank-0 chain of the tree, one row per level."""
    w = wl.CONFIGS["8b_single"].with_(noise_std=0.0)
    draft, t = _tree(w)
    x = wl.target_logits(w, draft, t["depth"])
    ref, _ = _check(x, w.dtype, t, w.L, 0.0, 0, 0, cuda_device)
    chain_depth, cur = 0, 0
    while True:
        kids = [c for c in range(1, t["n_nodes"][0] + 1)
                if t["parent"][0, c] == cur and t["rank"][0, c] == 0]
        if not kids:
            break
        cur, chain_depth = kids[0], chain_depth + 1
    assert chain_depth > 1 and ref["accept_len"][0] == chain_depth


@pytest.mark.parametrize("V,dtype,T,unaligned", [
    (1000, wl.FP32, 0.0, False), (1001, wl.BF16, 0.0, True), (8193, wl.BF16, 1.0, False),
    (16384, wl.BF16, 0.7, False), (16385, wl.FP32, 2.0, True), (151936, wl.BF16, 1.0, False),
    (5, wl.FP32, 1.0, False)])
def test_accept_path_edge_cases(cuda_device, V, dtype, T, unaligned):
    rng = np.random.default_rng(V + int(T * 10) + 1)
    B, L, K, N = 3, 5, 3, 30
    lp = -np.sort(rng.exponential(1.0, size=(B, L, K)).astype(np.float32), axis=2)
    lp = -np.sort(-lp, axis=2)
    tok = np.stack([[rng.permutation(V)[:K] if V >= K else np.arange(K) % V
                     for _ in range(L)] for _ in range(B)]).astype(np.int32)
    t = oracle.build_tree(lp, tok, rng.integers(0, V, size=B).astype(np.int32),
                          np.zeros(B, np.int32), N)
    x = (rng.standard_normal((B, N + 1, V)) * 2).astype(np.float32)
    for b in range(B):
        for c in range(1, t["n_nodes"][b] + 1):
            if rng.random() < 0.7:
                x[b, t["parent"][b, c], t["token"][b, c]] += 12
    x[0, 0, :] = 0.0  # a flat row: greedy picks token 0
    raw = wl.bf16_bits(x) if dtype == wl.BF16 else x
    _check(raw, dtype, t, L, T, 1234, 7, cuda_device, unaligned)


def test_accept_path_reads_only_the_path(cuda_device):
    """Every row off the accepted path holds NaN: the walk never reads it."""
    w = wl.CONFIGS["8b_single"].with_(B=2)
    draft, t = _tree(w)
    x = wl.target_logits(w, draft, t["depth"])
    ref = oracle.accept(x, w.dtype, t, w.L, temperature=0.0)
    poisoned = x.copy()
    nan_bits = np.uint16(0x7fc0) if w.dtype == wl.BF16 else np.float32(np.nan)
    for b in range(w.B):
        keep = {0} | {int(u) for u in ref["accepted_nodes"][b, :ref["accept_len"][b]]}
        for u in range(w.N + 1):
            if u not in keep:
                poisoned[b, u] = nan_bits
    dt = tree_to_dev(t, cuda_device)
    got = ops.accept_path(dev_logits(poisoned, w.dtype, cuda_device), dt, w.L)
    ops.ddtree_device_check()
    for k in OUT_KEYS:
        np.testing.assert_array_equal(host(got[k]), ref[k], err_msg=k)


def test_accept_path_bad_n_nodes_is_reported(cuda_device):
    w = wl.CONFIGS["tiny"]
    draft, t = _tree(w)
    x = wl.target_logits(w, draft, t["depth"])
    dt = tree_to_dev(t, cuda_device)
    dt["n_nodes"][:] = w.N + 5
    ops.accept_path(dev_logits(x, w.dtype, cuda_device), dt, w.L)
    with pytest.raises(ops.DDTreeError) as e:
        ops.ddtree_device_check()
    assert e.value.detail == 0x04000002


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_accept_budget_1024(cuda_device, T):
    """The largest budget (1025 rows, ancestor masks of 33 words): both walks
    against the oracle."""
    from tests.test_gpu_accept import _check as check_full
    rng = np.random.default_rng(1024 + int(T))
    B, L, K, N, V = 2, 16, 32, 1024, 3000
    lp = -np.sort(rng.exponential(0.5, size=(B, L, K)).astype(np.float32), axis=2)
    lp = -np.sort(-lp, axis=2)
    tok = np.stack([[rng.permutation(V)[:K] for _ in range(L)] for _ in range(B)]).astype(np.int32)
    t = oracle.build_tree(lp, tok, rng.integers(0, V, size=B).astype(np.int32),
                          np.zeros(B, np.int32), N)
    assert np.all(t["n_nodes"] == N)
    x = (rng.standard_normal((B, N + 1, V)) * 2).astype(np.float32)
    for b in range(B):
        for c in range(1, N + 1):
            if t["rank"][b, c] == 0:
                x[b, t["parent"][b, c], t["token"][b, c]] += 12
    ref, _ = _check(x, wl.FP32, t, L, T, 77, 5, cuda_device)
    check_full(x, wl.FP32, t, L, T, 77, 5, cuda_device)
    if T == 0.0:
        assert ref["accept_len"].min() >= 2  # the planted rank-0 chain is walked


@pytest.mark.parametrize("B,V,dtype,T", [
    (2, 151936, wl.FP32, 1.0),   # 19 chunks over a cluster of 10: two chunks on most CTAs
    (320, 40000, wl.FP32, 0.0),  # more sequences than CTA slots: one CTA each, 5 chunks in turn
    (320, 40000, wl.BF16, 1.0)])
def test_accept_path_cluster_shapes(cuda_device, B, V, dtype, T):
    rng = np.random.default_rng(B * 7 + V + int(T))
    L, K, N = 4, 3, 6
    lp = -np.sort(rng.exponential(1.0, size=(B, L, K)).astype(np.float32), axis=2)
    lp = -np.sort(-lp, axis=2)
    tok = np.stack([[rng.permutation(V)[:K] for _ in range(L)] for _ in range(B)]).astype(np.int32)
    t = oracle.build_tree(lp, tok, rng.integers(0, V, size=B).astype(np.int32),
                          np.zeros(B, np.int32), N)
    x = (rng.standard_normal((B, N + 1, V)) * 2).astype(np.float32)
    for b in range(B):
        for c in range(1, t["n_nodes"][b] + 1):
            if rng.random() < 0.6:
                x[b, t["parent"][b, c], t["token"][b, c]] += 12
    raw = wl.bf16_bits(x) if dtype == wl.BF16 else x
    _check(raw, dtype, t, L, T, 99, 1, cuda_device)
