"""GPU parity of step 3 (tree attention, tcgen05) against the fp64 oracle.
Criterion: bf16 outputs within 1e-2 max absolute error on unit-variance
inputs; logsumexp within 5e-3.  Cache rows past each prefix and tree rows past
each tree are NaN, so any leak of unread memory into a result fails."""
import numpy as np
import pytest
import torch

import oracle
from diffusion_draft_tree_gb300 import ops
from diffusion_draft_tree_gb300 import workloads as wl
from tests.gpu_util import dev_bf16, dev_i32, host, tree_to_dev

pytestmark = pytest.mark.gpu
TOL = 1e-2
LSE_TOL = 5e-3


def _tree_for(w):
    idx, _, lp32, _ = oracle.topk(wl.draft_logits(w), w.dtype, w.K)
    return oracle.build_tree(lp32, idx, wl.bonus_tokens(w), wl.prefix_lengths(w), w.N)


def _run(q, kc, vc, kt, vt, plen, tree, dev):
    dt = tree_to_dev(tree, dev)
    out, lse = ops.tree_attn(dev_bf16(q, dev), dev_bf16(kc, dev), dev_bf16(vc, dev),
                             dev_bf16(kt, dev), dev_bf16(vt, dev), dev_i32(plen, dev),
                             dt["n_nodes"], dt["anc_mask"])
    ops.ddtree_device_check()
    return host(out), host(lse)


def _compare(out, lse, ref, ref_lse, Hkv, units=None, rows=None, tree=None):
    B, R, Hq, D = out.shape
    Gs = Hq // Hkv
    sel = np.zeros((B, R, Hq), bool)
    lo, hi = rows if rows else (0, R)
    if units is None:
        sel[:, lo:hi] = True
    else:
        for b, g in units:
            sel[b, lo:hi, g * Gs:(g + 1) * Gs] = True
    assert np.isfinite(out[sel]).all()
    err = np.abs(out[sel] - ref[sel]).max()
    assert err <= TOL, f"max abs err {err}"
    live = sel & np.isfinite(ref_lse)
    assert np.abs(lse[live] - ref_lse[live]).max() <= LSE_TOL
    if tree is not None:  # padding rows: zero output, -inf lse
        for b in range(B):
            n = tree["n_nodes"][b]
            assert np.all(out[b, n + 1:] == 0) and np.all(np.isneginf(lse[b, n + 1:]))
    return err


def test_attn_tiny(cuda_device):
    w = wl.CONFIGS["tiny"]
    t = _tree_for(w)
    args = (wl.queries(w), wl.kv_cache(w, 0), wl.kv_cache(w, 1), wl.kv_tree(w, 0),
            wl.kv_tree(w, 1), wl.prefix_lengths(w))
    out, lse = _run(*args, t, cuda_device)
    ref, ref_lse = oracle.tree_attn(*args[:6], t["n_nodes"], t["anc_mask"])
    _compare(out, lse, ref, ref_lse, w.Hkv, tree=t)


def test_attn_8b_single_full(cuda_device):
    w = wl.CONFIGS["8b_single"]
    t = _tree_for(w)
    args = (wl.queries(w), wl.kv_cache(w, 0), wl.kv_cache(w, 1), wl.kv_tree(w, 0),
            wl.kv_tree(w, 1), wl.prefix_lengths(w))
    out, lse = _run(*args, t, cuda_device)
    ref, ref_lse = oracle.tree_attn(*args[:6], t["n_nodes"], t["anc_mask"])
    _compare(out, lse, ref, ref_lse, w.Hkv)


@pytest.mark.parametrize("name,units,rows", [
    ("budget_sweep_n512", [(0, 3)], None),
    ("budget_sweep_n32", [(0, 0), (0, 7)], None),
    ("ragged_serving", "longest_and_shortest", None),
    ("long_context_70b", [(1, 5)], (0, 6)),
    ("long_context_70b", [(3, 0)], (250, 257)),
])
def test_attn_workloads_sampled(cuda_device, name, units, rows):
    """Full-size launch; the oracle recomputes a seeded sample of (sequence, KV
    head) units and node rows one by one."""
    w = wl.CONFIGS[name]
    if units == "longest_and_shortest":
        units = [(int(np.argmax(w.P)), 2), (int(np.argmin(w.P)), 6)]
    t = _tree_for(w)
    args = (wl.queries(w), wl.kv_cache(w, 0), wl.kv_cache(w, 1), wl.kv_tree(w, 0),
            wl.kv_tree(w, 1), wl.prefix_lengths(w))
    out, lse = _run(*args, t, cuda_device)
    ref, ref_lse = oracle.tree_attn(*args[:6], t["n_nodes"], t["anc_mask"], units=units,
                                    rows=rows)
    _compare(out, lse, ref, ref_lse, w.Hkv, units=units, rows=rows)


def _random_case(seed, B, N, Hq, Hkv, D, P, cap, L=4, K=3):
    rng = np.random.default_rng(seed)
    q = wl.bf16_bits(rng.standard_normal((B, N + 1, Hq, D)).astype(np.float32))
    kc = np.full((B, Hkv, cap, D), wl.BF16_NAN, np.uint16)
    vc = np.full((B, Hkv, cap, D), wl.BF16_NAN, np.uint16)
    for b in range(B):
        kc[b, :, :P[b]] = wl.bf16_bits(rng.standard_normal((Hkv, P[b], D)).astype(np.float32))
        vc[b, :, :P[b]] = wl.bf16_bits(rng.standard_normal((Hkv, P[b], D)).astype(np.float32))
    kt = wl.bf16_bits(rng.standard_normal((B, N + 1, Hkv, D)).astype(np.float32))
    vt = wl.bf16_bits(rng.standard_normal((B, N + 1, Hkv, D)).astype(np.float32))
    lp = -np.sort(rng.exponential(1.0, size=(B, L, K)).astype(np.float32), axis=2)
    lp = -np.sort(-lp, axis=2)
    tok = rng.integers(0, 1000, size=(B, L, K)).astype(np.int32)
    t = oracle.build_tree(lp, tok, np.zeros(B, np.int32), np.asarray(P, np.int32), N)
    for b in range(B):  # rows of nodes past the tree are never read: poison them
        n = t["n_nodes"][b]
        kt[b, n + 1:] = wl.BF16_NAN
        vt[b, n + 1:] = wl.BF16_NAN
    return q, kc, vc, kt, vt, np.asarray(P, np.int32), t


@pytest.mark.parametrize("B,N,Hq,Hkv,D,P,cap,L,K", [
    (1, 0, 8, 2, 128, (65,), 80, 4, 3),          # root only
    (1, 5, 4, 4, 128, (0,), 16, 4, 3),           # empty prefix
    (1, 40, 16, 2, 128, (1,), 1, 4, 3),
    (2, 40, 8, 1, 64, (63, 64), 70, 4, 3),       # G = 8, D = 64
    (2, 127, 8, 8, 128, (65, 127), 300, 5, 3),   # G = 1
    (3, 128, 32, 8, 128, (128, 129, 300), 300, 6, 4),
    (1, 200, 32, 2, 128, (1000,), 1000, 6, 4),  # G = 16
    (2, 60, 4, 2, 64, (257, 3), 260, 3, 3),      # K^L = 39 < N: padding rows
    (1, 511, 8, 1, 128, (2000,), 2048, 16, 16),  # G = 8, N + 1 = 512
    (1, 1024, 4, 2, 128, (129,), 129, 16, 16),   # largest budget
    (3, 30, 8, 2, 64, (0, 2000, 700), 2048, 4, 3),  # 8-CTA clusters, some CTAs idle
])
def test_attn_edge_cases(cuda_device, B, N, Hq, Hkv, D, P, cap, L, K):
    q, kc, vc, kt, vt, plen, t = _random_case(B * 7 + N + D + cap, B, N, Hq, Hkv, D, P, cap, L, K)
    out, lse = _run(q, kc, vc, kt, vt, plen, t, cuda_device)
    ref, ref_lse = oracle.tree_attn(q, kc, vc, kt, vt, plen, t["n_nodes"], t["anc_mask"])
    _compare(out, lse, ref, ref_lse, Hkv, tree=t)


def test_attn_bad_prefix_len_is_reported_not_read(cuda_device):
    q, kc, vc, kt, vt, plen, t = _random_case(3, 1, 8, 4, 1, 128, (40,), 40)
    plen = np.array([41], np.int32)  # longer than the cache
    dt = tree_to_dev(t, cuda_device)
    ops.tree_attn(dev_bf16(q, cuda_device), dev_bf16(kc, cuda_device), dev_bf16(vc, cuda_device),
                  dev_bf16(kt, cuda_device), dev_bf16(vt, cuda_device),
                  dev_i32(plen, cuda_device), dt["n_nodes"], dt["anc_mask"])
    with pytest.raises(ops.DDTreeError) as e:
        ops.ddtree_device_check()
    assert e.value.detail == 0x03000001
    ops.ddtree_device_check()  # cleared
