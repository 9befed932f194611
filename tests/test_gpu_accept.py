"""GPU parity of step 4 (target decoding rule + acceptance walk) against the
oracle.  Criteria: target tokens, accepted length, accepted nodes and emitted
tokens bit-exact.  At temperature > 0 a node's sampled token may differ only
where the oracle's U*Z lies within 1e-5*Z of a CDF boundary, and then the GPU's
token must be the one across that boundary (its own CDF bin within 1e-5*Z of
U*Z); such nodes are counted.  Every sequence's walk is compared: bit-exact
with the oracle's where no token differs, else bit-exact with the walk that
the GPU's own per-node tokens imply."""
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
    got = ops.accept(xd, dt, L, temperature=T, seed=seed, step=step)
    ops.ddtree_device_check()
    tt = host(got["target_token"])
    outs = {k: host(got[k]) for k in OUT_KEYS}
    near = 0
    for b in range(x.shape[0]):
        n = tree["n_nodes"][b]
        diff = np.nonzero(tt[b, :n + 1] != ref["target_token"][b, :n + 1])[0]
        for u in diff:
            assert T > 0, f"greedy target token differs in sequence {b} at node {u}"
            assert ref["margin"][b, u] < MARGIN, f"sample differs off-boundary ({b}, {u})"
            d, ok = walk_check.sample_in_band(walk_check.row_f64(x, dtype, b, u), T, seed, step,
                                              b, u, int(tt[b, u]), MARGIN)
            assert ok, f"GPU token of ({b}, {u}) is not across the nearby CDF edge ({d:.3g})"
        near += len(diff)
        assert np.all(tt[b, n + 1:] == -1)
        want = ref if len(diff) == 0 else walk_check.walk(tree["parent"][b], tree["token"][b],
                                                          n, tt[b], L)
        for k in OUT_KEYS:
            exp = want[k][b] if want is ref else want[k]
            np.testing.assert_array_equal(outs[k][b], exp, err_msg=f"{k} of sequence {b}")
    return ref, near


def _tree(w):
    draft = wl.draft_logits(w)
    idx, _, lp32, _ = oracle.topk(draft, w.dtype, w.K)
    t = oracle.build_tree(lp32, idx, wl.bonus_tokens(w), wl.prefix_lengths(w), w.N)
    return draft, t


@pytest.mark.parametrize("name", ["tiny", "8b_single", "budget_sweep_n256", "long_context_70b",
                                  "ragged_serving"])
def test_accept_workloads(cuda_device, name):
    w = wl.CONFIGS[name]
    draft, t = _tree(w)
    x = wl.target_logits(w, draft, t["depth"])
    ref, near = _check(x, w.dtype, t, w.L, w.T, wl.philox_seed(w), 0, cuda_device)
    if w.T > 0:
        band = int(sum((ref["margin"][b, :t["n_nodes"][b] + 1] < MARGIN).sum()
                       for b in range(w.B)))
        print(f"{name}: {near} sampled tokens differ, all inside the {MARGIN:g}*Z band "
              f"({band} oracle nodes lie in it)")


def test_accept_planted_agreement_walks_rank0_chain(cuda_device):
    """Target row = draft row depth(u) with no noise, greedy: every drafted top-1
    token is accepted, to full depth L (the all-rank-0 chain is in the tree)."""
    w = wl.CONFIGS["8b_single"].with_(noise_std=0.0)
    draft, t = _tree(w)
    x = wl.target_logits(w, draft, t["depth"])
    ref, _ = _check(x, w.dtype, t, w.L, 0.0, 0, 0, cuda_device)
    chain_depth = 0
    cur = 0
    while True:
        kids = [c for c in range(1, t["n_nodes"][0] + 1)
                if t["parent"][0, c] == cur and t["rank"][0, c] == 0]
        if not kids:
            break
        cur, chain_depth = kids[0], chain_depth + 1
    assert ref["accept_len"][0] == chain_depth


@pytest.mark.parametrize("V,dtype,T,unaligned", [
    (1000, wl.FP32, 0.0, False), (1001, wl.BF16, 0.0, True), (8193, wl.BF16, 1.0, False),
    (16384, wl.BF16, 0.7, False), (16385, wl.FP32, 2.0, True), (151936, wl.BF16, 1.0, False),
    (5, wl.FP32, 1.0, False)])
def test_accept_edge_cases(cuda_device, V, dtype, T, unaligned):
    rng = np.random.default_rng(V + int(T * 10))
    B, L, K, N = 3, 5, 3, 30
    lp = -np.sort(rng.exponential(1.0, size=(B, L, K)).astype(np.float32), axis=2)
    lp = -np.sort(-lp, axis=2)
    tok = np.stack([[rng.permutation(V)[:K] if V >= K else np.arange(K) % V
                     for _ in range(L)] for _ in range(B)]).astype(np.int32)
    t = oracle.build_tree(lp, tok, rng.integers(0, V, size=B).astype(np.int32),
                          np.zeros(B, np.int32), N)
    x = (rng.standard_normal((B, N + 1, V)) * 2).astype(np.float32)
    # make the target agree with the tree often: boost each node's first child token
    for b in range(B):
        for c in range(1, t["n_nodes"][b] + 1):
            if rng.random() < 0.7:
                x[b, t["parent"][b, c], t["token"][b, c]] += 12
    x[0, 0, :] = 0.0  # a flat row: greedy picks token 0
    raw = wl.bf16_bits(x) if dtype == wl.BF16 else x
    _check(raw, dtype, t, L, T, 1234, 7, cuda_device, unaligned)


def test_accept_padding_rows_are_not_read(cuda_device):
    """A tree smaller than the budget: rows past n_nodes hold NaN and are skipped."""
    rng = np.random.default_rng(2)
    B, L, K, N, V = 2, 2, 2, 20, 3000
    lp = -np.sort(rng.exponential(1.0, size=(B, L, K)).astype(np.float32), axis=2)
    lp = -np.sort(-lp, axis=2)
    tok = rng.integers(0, V, size=(B, L, K)).astype(np.int32)
    t = oracle.build_tree(lp, tok, np.zeros(B, np.int32), np.zeros(B, np.int32), N)
    assert t["n_nodes"][0] == 6
    x = rng.standard_normal((B, N + 1, V)).astype(np.float32)
    x[:, 7:] = np.nan
    _check(x, wl.FP32, t, L, 0.0, 0, 0, cuda_device)
    _check(x, wl.FP32, t, L, 1.0, 5, 1, cuda_device)


def test_accept_bad_n_nodes_is_reported(cuda_device):
    w = wl.CONFIGS["tiny"]
    draft, t = _tree(w)
    x = wl.target_logits(w, draft, t["depth"])
    dt = tree_to_dev(t, cuda_device)
    dt["n_nodes"][:] = w.N + 5
    ops.accept(dev_logits(x, w.dtype, cuda_device), dt, w.L)
    with pytest.raises(ops.DDTreeError) as e:
        ops.ddtree_device_check()
    assert e.value.detail == 0x04000002
