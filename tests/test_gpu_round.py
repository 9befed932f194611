"""One whole DDTree round on the GPU (top-K -> heap -> tree attention -> walk),
each step fed by the previous GPU step, against the oracle's own chain.

The GPU's fp32 log-probs agree with the oracle's to ~1e-6, so prefixes whose
scores differ by less than that may be popped in the other order: node ids
are compared through their token paths, and the accepted tokens exactly."""
import numpy as np
import pytest

import oracle
from diffusion_draft_tree_gb300 import ops
from diffusion_draft_tree_gb300 import workloads as wl
from tests.gpu_util import dev_bf16, dev_i32, dev_logits, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "8b_single", "8b_single_chain"])
def test_round_chain_matches_oracle_chain(cuda_device, name):
    """8b_single_chain is the vanilla DFlash chain (K = 1, N = L): one token per
    draft position, accepted while it matches the target's token."""
    w = (wl.CONFIGS["8b_single"].with_(K=1, N=16) if name == "8b_single_chain"
         else wl.CONFIGS[name])
    dev = cuda_device
    draft, bonus, plen = wl.draft_logits(w), wl.bonus_tokens(w), wl.prefix_lengths(w)
    o_idx, _, o_lp32, _ = oracle.topk(draft, w.dtype, w.K)
    o_tree = oracle.build_tree(o_lp32, o_idx, bonus, plen, w.N)
    x = wl.target_logits(w, draft, o_tree["depth"])
    o_acc = oracle.accept(x, w.dtype, o_tree, w.L)

    idx, lp, _ = ops.topk(dev_logits(draft, w.dtype, dev), w.K)
    tree = ops.build(lp, idx, dev_i32(bonus, dev), dev_i32(plen, dev), w.N)
    g_paths = _paths(host(tree["parent"])[0], host(tree["token"])[0], host(tree["n_nodes"])[0])
    o_paths = _paths(o_tree["parent"][0], o_tree["token"][0], o_tree["n_nodes"][0])
    assert set(g_paths) == set(o_paths)
    g_score = dict(zip(g_paths, host(tree["score"])[0]))
    for p, s in zip(o_paths, o_tree["score"][0]):
        assert abs(g_score[p] - s) <= 1e-5 * max(1, len(p))
    q, kc, vc, kt, vt = (wl.queries(w), wl.kv_cache(w, 0), wl.kv_cache(w, 1), wl.kv_tree(w, 0),
                         wl.kv_tree(w, 1))
    out, _ = ops.tree_attn(dev_bf16(q, dev), dev_bf16(kc, dev), dev_bf16(vc, dev),
                           dev_bf16(kt, dev), dev_bf16(vt, dev), dev_i32(plen, dev),
                           tree["n_nodes"], tree["anc_mask"])
    ref, _ = oracle.tree_attn(q, kc, vc, kt, vt, plen, o_tree["n_nodes"], o_tree["anc_mask"],
                              units=[(0, 0)])
    G = w.Hq // w.Hkv
    assert np.abs(host(out)[0, :, :G] - ref[0, :, :G]).max() <= 1e-2
    acc = ops.accept(dev_logits(x, w.dtype, dev), tree, w.L)
    ops.ddtree_device_check()
    for k in ("accept_len", "out_tokens", "next_bonus"):
        np.testing.assert_array_equal(host(acc[k]), o_acc[k], err_msg=k)
    n_acc = o_acc["accept_len"][0]
    assert [g_paths[u] for u in host(acc["accepted_nodes"])[0, :n_acc]] == \
        [o_paths[u] for u in o_acc["accepted_nodes"][0, :n_acc]]
    if w.K == 1:
        # the chain: node d is the draft argmax at position d-1; accepted while it
        # equals the target's argmax at node d-1
        t = np.argmax(wl.bf16_to_f32(x[0]), axis=1)
        chain_tok = np.argmax(wl.bf16_to_f32(draft[0]), axis=1)
        expect = 0
        while expect < w.L and chain_tok[expect] == t[expect]:
            expect += 1
        assert host(acc["accept_len"])[0] == expect


def _paths(parent, token, n):
    """Token path (root excluded) of every node 0..n."""
    out = []
    for u in range(n + 1):
        p, a = [], u
        while a > 0:
            p.append(int(token[a]))
            a = parent[a]
        out.append(tuple(reversed(p)))
    return out
