"""GPU parity of the KV commit (after the walk, the root and the accepted
nodes join the prefix) against the oracle: caches and prefix lengths are
compared bit for bit; a path that does not fit is reported and left alone."""
import numpy as np
import pytest
import torch

import oracle
from diffusion_draft_tree_gb300 import ops
from diffusion_draft_tree_gb300 import workloads as wl
from tests.gpu_util import dev_bf16, dev_i32

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _case(seed, B, N, Hkv, D, L, cap, alens=None):
    rng = np.random.default_rng(seed)
    kc = wl.bf16_bits(rng.standard_normal((B, Hkv, cap, D)).astype(np.float32))
    vc = wl.bf16_bits(rng.standard_normal((B, Hkv, cap, D)).astype(np.float32))
    kt = wl.bf16_bits(rng.standard_normal((B, N + 1, Hkv, D)).astype(np.float32))
    vt = wl.bf16_bits(rng.standard_normal((B, N + 1, Hkv, D)).astype(np.float32))
    if alens is None:
        alens = rng.integers(0, L + 1, size=B)
    alen = np.asarray(alens, np.int32)
    acc = np.full((B, L), -1, np.int32)
    for b in range(B):
        acc[b, :alen[b]] = rng.choice(np.arange(1, N + 1), size=alen[b], replace=False)
    P = np.array([rng.integers(0, cap - alen[b]) for b in range(B)], np.int32)
    return kc, vc, kt, vt, alen, acc, P


def _run(kc, vc, kt, vt, alen, acc, P, dev):
    dkc, dvc = dev_bf16(kc, dev), dev_bf16(vc, dev)
    dplen = dev_i32(P, dev)
    ops.ddtree_commit(dkc, dvc, dev_bf16(kt, dev), dev_bf16(vt, dev), dev_i32(alen, dev),
                      dev_i32(acc, dev), dplen)
    return dkc, dvc, dplen


@pytest.mark.parametrize("B,N,Hkv,D,L,cap", [
    (1, 16, 1, 64, 4, 80),       # tiny shape
    (3, 64, 8, 128, 16, 2100),   # 8B-class heads
    (16, 128, 8, 128, 16, 200),  # a ragged batch
    (2, 1024, 2, 64, 16, 40),    # largest budget, nearly full caches
])
def test_commit_matches_oracle(cuda_device, B, N, Hkv, D, L, cap):
    kc, vc, kt, vt, alen, acc, P = _case(B * 31 + N, B, N, Hkv, D, L, cap)
    dkc, dvc, dplen = _run(kc, vc, kt, vt, alen, acc, P, cuda_device)
    ops.ddtree_device_check()
    rk, rv, rp = oracle.commit(kc, vc, kt, vt, alen, acc, P)
    np.testing.assert_array_equal(dplen.cpu().numpy(), rp)
    np.testing.assert_array_equal(_bits(dkc), rk)
    np.testing.assert_array_equal(_bits(dvc), rv)


def test_commit_extremes(cuda_device):
    """Root only (accept_len 0) and a full block (accept_len L), side by side;
    a path that ends exactly at the cache capacity."""
    B, N, Hkv, D, L, cap = 3, 40, 4, 128, 16, 64
    kc, vc, kt, vt, alen, acc, P = _case(7, B, N, Hkv, D, L, cap, alens=[0, L, L])
    P[2] = cap - L - 1
    dkc, dvc, dplen = _run(kc, vc, kt, vt, alen, acc, P, cuda_device)
    ops.ddtree_device_check()
    rk, rv, rp = oracle.commit(kc, vc, kt, vt, alen, acc, P)
    np.testing.assert_array_equal(dplen.cpu().numpy(), rp)
    np.testing.assert_array_equal(_bits(dkc), rk)
    np.testing.assert_array_equal(_bits(dvc), rv)


def test_commit_overflow_is_reported_and_skipped(cuda_device):
    B, N, Hkv, D, L, cap = 2, 20, 2, 64, 8, 30
    kc, vc, kt, vt, alen, acc, P = _case(9, B, N, Hkv, D, L, cap, alens=[5, 3])
    P[0] = cap - 5  # 5 accepted + the root do not fit
    dkc, dvc, dplen = _run(kc, vc, kt, vt, alen, acc, P, cuda_device)
    with pytest.raises(ops.DDTreeError) as e:
        ops.ddtree_device_check()
    assert e.value.detail == 0x05000001
    got = dplen.cpu().numpy()
    assert got[0] == P[0] and got[1] == P[1] + alen[1] + 1
    np.testing.assert_array_equal(_bits(dkc)[0], kc[0])
    _, _, rp = oracle.commit(kc[1:], vc[1:], kt[1:], vt[1:], alen[1:], acc[1:], P[1:])
    assert got[1] == rp[0]


def test_round_then_commit_8b_single(cuda_device):
    """The accept outputs of a full GPU round drive the commit; the result
    equals the oracle's commit of the same path."""
    w = wl.CONFIGS["8b_single"]
    dev = cuda_device
    draft = dev_bf16(wl.draft_logits(w).reshape(w.B * w.L, w.V), dev)
    idx, lp, _ = ops.topk(draft, w.K)
    tree = ops.build(lp.view(w.B, w.L, w.K), idx.view(w.B, w.L, w.K),
                     dev_i32(wl.bonus_tokens(w), dev), dev_i32(wl.prefix_lengths(w), dev), w.N)
    depth = tree["depth"].cpu().numpy()
    target = dev_bf16(wl.target_logits(w, wl.draft_logits(w), depth), dev)
    acc = ops.accept(target, tree, w.L, w.T, wl.philox_seed(w), 0)
    kc, vc = wl.kv_cache(w, 0), wl.kv_cache(w, 1)
    kt, vt = wl.kv_tree(w, 0), wl.kv_tree(w, 1)
    P = wl.prefix_lengths(w)
    cap = kc.shape[2]
    grow = w.L + 1
    kc2 = np.concatenate([kc, np.zeros(kc.shape[:2] + (grow, kc.shape[3]), np.uint16)], axis=2)
    vc2 = np.concatenate([vc, np.zeros(vc.shape[:2] + (grow, vc.shape[3]), np.uint16)], axis=2)
    dkc, dvc = dev_bf16(kc2, dev), dev_bf16(vc2, dev)
    dplen = dev_i32(P, dev)
    ops.ddtree_commit(dkc, dvc, dev_bf16(kt, dev), dev_bf16(vt, dev), acc["accept_len"],
                      acc["accepted_nodes"], dplen)
    ops.ddtree_device_check()
    alen = acc["accept_len"].cpu().numpy()
    nodes = acc["accepted_nodes"].cpu().numpy()
    rk, rv, rp = oracle.commit(kc2, vc2, kt, vt, alen, nodes, P)
    assert cap + grow == kc2.shape[2]
    np.testing.assert_array_equal(dplen.cpu().numpy(), rp)
    np.testing.assert_array_equal(_bits(dkc), rk)
    np.testing.assert_array_equal(_bits(dvc), rv)
