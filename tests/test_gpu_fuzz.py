"""A seeded sweep of random small shapes through the whole round, each call
through the C ABI against the oracle: top-K (indices bit-exact, log-probs
within 1e-5), the build fed the oracle's fp32 table (bit-exact), tree
attention (1e-2 max abs error, lse 5e-3), and both walks (greedy bit-exact; at
T > 0 a token may differ only inside the oracle's 1e-5 band).  Shapes cover
V not a multiple of the vector width, K from 1 to 32, budgets from 0 to 300,
L from 1 to 16, empty and ragged prefixes, bf16 and fp32 rows, G from 1 to 8
and D in {64, 128}.  (A hypothesis-driven version would need a package that
the GPU machines do not carry; the seeds are fixed so a failure reproduces.)"""
import numpy as np
import pytest
import torch

import oracle
from diffusion_draft_tree_gb300 import ops
from diffusion_draft_tree_gb300 import workloads as wl
from tests.gpu_util import dev_bf16, dev_f32, dev_i32, dev_logits, host, tree_to_dev
from tests.test_gpu_accept import _check as check_full_walk
from tests.test_gpu_accept_path import _check as check_path_walk
from tests.test_gpu_attn import _compare

pytestmark = pytest.mark.gpu


def _shape(seed):
    rng = np.random.default_rng(seed)
    dtype = wl.BF16 if rng.random() < 0.6 else wl.FP32
    V = int(rng.integers(40, 24000))
    K = int(min(V, rng.choice([1, 2, 3, 8, 16, 32])))
    L = int(rng.choice([1, 2, 5, 16]))
    N = int(rng.choice([0, 1, K, 17, 64, 65, 130, 300]))
    B = int(rng.integers(1, 4))
    G = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([1, 2]))
    D = int(rng.choice([64, 128]))
    cap = int(rng.integers(1, 400))
    P = [int(rng.integers(0, cap + 1)) for _ in range(B)]
    T = float(rng.choice([0.0, 0.0, 0.7, 1.5]))
    return rng, dict(dtype=dtype, V=V, K=K, L=L, N=N, B=B, Hq=G * Hkv, Hkv=Hkv, D=D, cap=cap,
                     P=P, T=T)


@pytest.mark.parametrize("seed", list(range(24)))
def test_random_round(cuda_device, seed):
    rng, s = _shape(1000 + seed)
    B, L, V, K, N, dtype = s["B"], s["L"], s["V"], s["K"], s["N"], s["dtype"]
    dev = cuda_device

    # step 1: top-K of random draft rows
    x = (rng.standard_normal((B, L, V)) * 3).astype(np.float32)
    raw = wl.bf16_bits(x) if dtype == wl.BF16 else x
    o_idx, o_lp64, o_lp32, o_lse = oracle.topk(raw, dtype, K)
    idx, lp, lse = ops.topk(dev_logits(raw.reshape(B * L, V), dtype, dev), K)
    ops.ddtree_device_check()
    np.testing.assert_array_equal(host(idx).reshape(B, L, K), o_idx)
    assert np.abs(host(lp).reshape(B, L, K) - o_lp64).max() <= 1e-5
    assert np.abs(host(lse).reshape(B, L) - o_lse).max() <= 1e-5

    # step 2: the tree from the oracle's fp32 table
    bonus = rng.integers(0, V, size=B).astype(np.int32)
    plen = np.asarray(s["P"], np.int32)
    t = oracle.build_tree(o_lp32, o_idx, bonus, plen, N)
    got = ops.build(dev_f32(o_lp32, dev), dev_i32(o_idx, dev), dev_i32(bonus, dev),
                    dev_i32(plen, dev), N)
    ops.ddtree_device_check()
    for k in ("parent", "depth", "rank", "token", "pos_id", "child_count", "n_nodes"):
        np.testing.assert_array_equal(host(got[k]), t[k], err_msg=k)
    np.testing.assert_array_equal(host(got["score"]).view(np.uint32), t["score"].view(np.uint32))
    np.testing.assert_array_equal(host(got["anc_mask"]).view(np.uint32), t["anc_mask"])

    # step 3: tree attention on random Q/K/V (rows that must not be read are NaN)
    Hq, Hkv, D, cap = s["Hq"], s["Hkv"], s["D"], s["cap"]
    q = wl.bf16_bits(rng.standard_normal((B, N + 1, Hq, D)).astype(np.float32))
    kc = np.full((B, Hkv, cap, D), wl.BF16_NAN, np.uint16)
    vc = np.full((B, Hkv, cap, D), wl.BF16_NAN, np.uint16)
    for b in range(B):
        kc[b, :, :plen[b]] = wl.bf16_bits(rng.standard_normal((Hkv, plen[b], D)).astype(np.float32))
        vc[b, :, :plen[b]] = wl.bf16_bits(rng.standard_normal((Hkv, plen[b], D)).astype(np.float32))
    kt = wl.bf16_bits(rng.standard_normal((B, N + 1, Hkv, D)).astype(np.float32))
    vt = wl.bf16_bits(rng.standard_normal((B, N + 1, Hkv, D)).astype(np.float32))
    for b in range(B):
        kt[b, t["n_nodes"][b] + 1:] = wl.BF16_NAN
        vt[b, t["n_nodes"][b] + 1:] = wl.BF16_NAN
    dt = tree_to_dev(t, dev)
    out, alse = ops.tree_attn(dev_bf16(q, dev), dev_bf16(kc, dev), dev_bf16(vc, dev),
                              dev_bf16(kt, dev), dev_bf16(vt, dev), dev_i32(plen, dev),
                              dt["n_nodes"], dt["anc_mask"])
    ops.ddtree_device_check()
    ref, ref_lse = oracle.tree_attn(q, kc, vc, kt, vt, plen, t["n_nodes"], t["anc_mask"])
    _compare(host(out), host(alse), ref, ref_lse, Hkv, tree=t)

    # step 4: both walks over random target rows that often agree with the tree
    y = (rng.standard_normal((B, N + 1, V)) * 2).astype(np.float32)
    for b in range(B):
        for c in range(1, t["n_nodes"][b] + 1):
            if rng.random() < 0.5:
                y[b, t["parent"][b, c], t["token"][b, c]] += 10
    yraw = wl.bf16_bits(y) if dtype == wl.BF16 else y
    check_full_walk(yraw, dtype, t, L, s["T"], seed, 3, dev)
    check_path_walk(yraw, dtype, t, L, s["T"], seed, 3, dev)
