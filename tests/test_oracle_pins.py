"""Pins for the CPU oracle: checks against facts the pages and the mathematics
fix, computed independently of the oracle's own code (library routines, brute
force, closed forms, special cases).  CPU only.

Pages: "Accelerating Speculative Decoding with Block Diffusion Draft Trees"
(paperlayer.ai summary): §3 marginals, §4.1 tree + walk, §4.2 surrogate and
Proposition 2, §4.3 / App. A the best-first heap.
"""
import functools
import itertools

import numpy as np
import pytest
import torch

import oracle
from diffusion_draft_tree_gb300 import workloads as wl


# --------------------------------------------------------------------------
# step 1: log-softmax + top-K
# --------------------------------------------------------------------------

def _rows_with_ties(rng, rows, V, dtype):
    x = rng.standard_normal((rows, V)).astype(np.float32) * 3
    # plant exact ties among the largest values and a -0.0 / +0.0 pair
    x[:, 5] = x[:, 7] = x.max(axis=1) + 1
    x[:, 9] = x[:, 5]
    x[:, 11], x[:, 12] = -0.0, 0.0
    if dtype == wl.BF16:
        return wl.bf16_bits(x), wl.bf16_to_f32(wl.bf16_bits(x)).astype(np.float64)
    return x, x.astype(np.float64)


@pytest.mark.parametrize("dtype", [wl.FP32, wl.BF16])
@pytest.mark.parametrize("V,K", [(37, 1), (1000, 4), (4099, 16), (64, 64)])
def test_topk_against_sort_and_logsumexp(dtype, V, K):
    rng = np.random.default_rng(V * 7 + K)
    raw, x = _rows_with_ties(rng, 5, V, dtype)
    idx, lp64, lp32, lse = oracle.topk(raw, dtype, K)
    for r in range(x.shape[0]):
        order = np.lexsort((np.arange(V), -x[r]))  # value desc, index asc (stable library sort)
        np.testing.assert_array_equal(idx[r], order[:K])
        ref_lse = torch.logsumexp(torch.from_numpy(x[r]), dim=0).item()
        assert abs(lse[r] - ref_lse) <= 1e-12 * max(1.0, abs(ref_lse))
        np.testing.assert_allclose(lp64[r], x[r][order[:K]] - ref_lse, rtol=0, atol=1e-12)
        np.testing.assert_array_equal(lp32[r], lp64[r].astype(np.float32))
        assert np.all(lp64[r] <= 0) and np.all(np.diff(lp64[r]) <= 0)
        # the whole row's probabilities, from the oracle's lse, sum to one
        assert abs(np.exp(x[r] - lse[r]).sum() - 1.0) < 1e-12
        tv, _ = torch.topk(torch.from_numpy(x[r]), K)
        np.testing.assert_array_equal(tv.numpy(), x[r][idx[r]])


def test_topk_signed_zero_ties_by_index():
    x = np.array([[-0.0, 0.0, -1.0, -0.0]], np.float32)
    idx, _, _, _ = oracle.topk(x, wl.FP32, 4)
    np.testing.assert_array_equal(idx[0], [0, 1, 3, 2])


# --------------------------------------------------------------------------
# step 2: best-first heap (Algorithm 1) vs brute force and Proposition 2
# --------------------------------------------------------------------------

def _enumerate_prefixes(lp32, L, K):
    """All prefixes of the K-restricted set with their fp32 path sums (path order)."""
    score = {(): np.float32(0)}
    frontier = [()]
    for d in range(L):
        nxt = []
        for p in frontier:
            for r in range(K):
                c = p + (r,)
                score[c] = np.float32(score[p] + lp32[d, r])
                nxt.append(c)
        frontier = nxt
    return score


def _brute_force_tree(lp32, tok, N):
    """Sort every prefix by the heap's priority order; keep the first N."""
    L, K = lp32.shape
    score = _enumerate_prefixes(lp32, L, K)

    @functools.lru_cache(maxsize=None)
    def cmp(a, b):
        if a == b:
            return 0
        if score[a] != score[b]:
            return -1 if score[a] > score[b] else 1
        if len(a) != len(b):
            return -1 if len(a) < len(b) else 1
        if a[:-1] != b[:-1]:
            return cmp(a[:-1], b[:-1])
        return -1 if a[-1] < b[-1] else 1

    prefixes = sorted((p for p in score if p), key=functools.cmp_to_key(cmp))[:N]
    node_of = {(): 0}
    rows = [(-1, 0, -1, None, 0.0)]
    for i, p in enumerate(prefixes, start=1):
        node_of[p] = i
        rows.append((node_of[p[:-1]], len(p), p[-1], int(tok[len(p) - 1, p[-1]]), score[p]))
    return rows


def _tables(rng, L, K, ties=False):
    if ties:  # coarse values: many exact equalities between path sums
        lp = -rng.integers(1, 4, size=(L, K)).astype(np.float32) / 4
        lp = -np.sort(-lp, axis=1)
    else:
        lp = -np.sort(rng.exponential(1.0, size=(L, K)).astype(np.float32), axis=1)
        lp = -np.sort(-lp, axis=1)
    tok = np.stack([rng.permutation(1000)[:K] for _ in range(L)]).astype(np.int32)
    return lp, tok


@pytest.mark.parametrize("K,L,N,ties", [(2, 3, 5, False), (3, 3, 12, False), (2, 5, 20, True),
                                        (4, 4, 16, False), (3, 4, 40, True), (2, 3, 14, False),
                                        (2, 3, 30, False), (1, 6, 4, False), (5, 2, 30, True)])
def test_heap_equals_brute_force_order(K, L, N, ties):
    rng = np.random.default_rng(K * 100 + L * 10 + N)
    lp, tok = _tables(rng, L, K, ties)
    t = oracle.build_tree(lp[None], tok[None], np.array([7]), np.array([50]), N)
    ref = _brute_force_tree(lp, tok, N)
    n = t["n_nodes"][0]
    assert n == len(ref) - 1 == min(N, sum(K ** d for d in range(1, L + 1)))
    for u, (par, dep, rk, tk, sc) in enumerate(ref):
        assert t["parent"][0, u] == par and t["depth"][0, u] == dep
        if u:
            assert t["rank"][0, u] == rk and t["token"][0, u] == tk
            assert t["score"][0, u] == sc
    # padding rows
    assert np.all(t["parent"][0, n + 1:] == -1) and np.all(t["child_count"][0, n + 1:] == 0)
    assert np.all(t["anc_mask"][0, n + 1:] == 0)


@pytest.mark.parametrize("N", range(1, 7))
def test_heap_tree_is_optimal_among_all_valid_trees(N):
    """Proposition 2: the surrogate (sum of prefix probabilities, §4.2) of the
    heap's tree equals the maximum over every prefix-closed set of <= N nodes."""
    rng = np.random.default_rng(N)
    L, K = 3, 2
    lp, tok = _tables(rng, L, K)
    score = _enumerate_prefixes(lp, L, K)
    nodes = [p for p in score if p]
    prob = {p: float(np.exp(np.float64(score[p]))) for p in nodes}
    best = 0.0
    for mask in range(1 << len(nodes)):
        chosen = {nodes[i] for i in range(len(nodes)) if mask >> i & 1}
        if len(chosen) > N or any(p[:-1] and p[:-1] not in chosen for p in chosen):
            continue
        best = max(best, sum(prob[p] for p in chosen))
    t = oracle.build_tree(lp[None], tok[None], np.array([0]), np.array([0]), N)
    got = float(np.exp(t["score"][0, 1:t["n_nodes"][0] + 1].astype(np.float64)).sum())
    assert abs(got - best) < 1e-12


def _root_path(parent, u):
    path = []
    while u >= 0:
        path.append(u)
        u = parent[u]
    return path[::-1]


def test_heap_structure_invariants():
    w = wl.CONFIGS["tiny"]
    idx, _, lp32, _ = oracle.topk(wl.draft_logits(w), w.dtype, w.K)
    t = oracle.build_tree(lp32, idx, wl.bonus_tokens(w), wl.prefix_lengths(w), w.N)
    n = t["n_nodes"][0]
    par, dep = t["parent"][0], t["depth"][0]
    for u in range(1, n + 1):
        assert 0 <= par[u] < u                      # topological (pop) order
        assert dep[u] == dep[par[u]] + 1
        assert t["score"][0, par[u]] >= t["score"][0, u]   # App. A: ancestors are likelier
        assert t["pos_id"][0, u] == w.P[0] + dep[u]
        assert t["token"][0, u] == idx[0, dep[u] - 1, t["rank"][0, u]]
    for u in range(n + 1):
        bits = {a for a in range(n + 1) if t["anc_mask"][0, u, a // 32] >> (a % 32) & 1}
        assert bits == set(_root_path(par, u))     # ancestors are exactly the root path
        assert t["child_count"][0, u] == int(np.sum(par[1:n + 1] == u))
    assert t["token"][0, 0] == wl.bonus_tokens(w)[0] and t["pos_id"][0, 0] == w.P[0]


def test_heap_k1_is_the_argmax_chain():
    rng = np.random.default_rng(3)
    lp, tok = _tables(rng, 6, 1)
    for N in (0, 3, 6, 10):
        t = oracle.build_tree(lp[None], tok[None], np.array([1]), np.array([4]), N)
        n = min(N, 6)
        assert t["n_nodes"][0] == n
        np.testing.assert_array_equal(t["parent"][0, :n + 1], np.arange(-1, n))
        np.testing.assert_array_equal(t["token"][0, 1:n + 1], tok[:n, 0])


@pytest.mark.slow
def test_surrogate_is_expected_accepted_length_monte_carlo():
    """§4.2: E[accepted length] under the factorised draft distribution equals
    the sum of the tree's prefix probabilities.  Paths are drawn token by token
    from the full softmax of every position (not only the top-K)."""
    w = wl.CONFIGS["tiny"]
    x = wl.draft_logits(w)[0].astype(np.float64)           # [L][V]
    idx, _, lp32, _ = oracle.topk(x.astype(np.float32)[None], wl.FP32, w.K)
    t = oracle.build_tree(lp32, idx, np.array([0]), np.array([0]), w.N)
    n = t["n_nodes"][0]
    p = np.exp(x - x.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    rng = np.random.default_rng(11)
    S = 400_000
    ys = np.stack([np.searchsorted(np.cumsum(p[d]), rng.random(S), side="right")
                   for d in range(w.L)], axis=1)
    child = {}
    for u in range(1, n + 1):
        child[(t["parent"][0, u], t["token"][0, u])] = u
    acc = np.zeros(S)
    for s in range(S):
        cur = 0
        for d in range(w.L):
            cur = child.get((cur, ys[s, d]), -1)
            if cur < 0:
                break
            acc[s] += 1
    expect = float(np.exp(t["score"][0, 1:n + 1].astype(np.float64)).sum())
    sigma = acc.std() / np.sqrt(S)
    assert abs(acc.mean() - expect) < 4 * sigma + 1e-6


# --------------------------------------------------------------------------
# step 3: tree attention vs torch scaled_dot_product_attention (fp64)
# --------------------------------------------------------------------------

def _attn_inputs(rng, B, N, Hq, Hkv, D, P, cap):
    q = wl.bf16_bits(rng.standard_normal((B, N + 1, Hq, D)).astype(np.float32))
    kc = np.full((B, Hkv, cap, D), wl.BF16_NAN, np.uint16)
    vc = np.full((B, Hkv, cap, D), wl.BF16_NAN, np.uint16)
    for b in range(B):
        kc[b, :, :P[b]] = wl.bf16_bits(rng.standard_normal((Hkv, P[b], D)).astype(np.float32))
        vc[b, :, :P[b]] = wl.bf16_bits(rng.standard_normal((Hkv, P[b], D)).astype(np.float32))
    kt = wl.bf16_bits(rng.standard_normal((B, N + 1, Hkv, D)).astype(np.float32))
    vt = wl.bf16_bits(rng.standard_normal((B, N + 1, Hkv, D)).astype(np.float32))
    return q, kc, vc, kt, vt


def _f64(bits):
    return torch.from_numpy(wl.bf16_to_f32(bits).astype(np.float64))


def _random_tree(rng, B, N, L, K):
    lp = -np.sort(rng.exponential(1.0, size=(B, L, K)).astype(np.float32), axis=2)
    lp = -np.sort(-lp, axis=2)
    tok = rng.integers(0, 100, size=(B, L, K)).astype(np.int32)
    return oracle.build_tree(lp, tok, np.zeros(B, np.int32), np.zeros(B, np.int32), N)


@pytest.mark.parametrize("B,N,Hq,Hkv,D,P", [(1, 16, 2, 1, 64, (64,)), (2, 20, 8, 2, 32, (5, 0)),
                                            (1, 7, 4, 4, 16, (33,))])
def test_tree_attention_is_sdpa_over_each_root_path(B, N, Hq, Hkv, D, P):
    """§4.1: a tree token attends to the prefix and to its own root path, and to
    nothing else; so each row equals plain attention over [prefix; root path]."""
    rng = np.random.default_rng(N + D)
    cap = max(P) + 3
    q, kc, vc, kt, vt = _attn_inputs(rng, B, N, Hq, Hkv, D, P, cap)
    t = _random_tree(rng, B, N, L=4, K=3)
    out, lse = oracle.tree_attn(q, kc, vc, kt, vt, np.array(P), t["n_nodes"], t["anc_mask"])
    G = Hq // Hkv
    for b in range(B):
        for u in range(t["n_nodes"][b] + 1):
            path = _root_path(t["parent"][b], u)
            for h in range(Hq):
                g = h // G
                k = torch.cat([_f64(kc[b, g, :P[b]]), _f64(kt[b, path, g])])
                v = torch.cat([_f64(vc[b, g, :P[b]]), _f64(vt[b, path, g])])
                ref = torch.nn.functional.scaled_dot_product_attention(
                    _f64(q[b, u, h])[None, None], k[None], v[None])[0, 0]
                np.testing.assert_allclose(out[b, u, h], ref.numpy(), rtol=0, atol=1e-12)
                s = (_f64(q[b, u, h]) @ k.T) / np.sqrt(D)
                assert abs(lse[b, u, h] - torch.logsumexp(s, 0).item()) < 1e-12
        assert np.all(out[b, t["n_nodes"][b] + 1:] == 0)


def test_tree_attention_chain_is_causal_attention():
    """A chain tree (K = 1) is ordinary causal attention over [prefix; chain]."""
    rng = np.random.default_rng(5)
    B, N, Hq, Hkv, D, P = 1, 9, 4, 2, 32, (20,)
    q, kc, vc, kt, vt = _attn_inputs(rng, B, N, Hq, Hkv, D, P, 24)
    t = _random_tree(rng, B, N, L=12, K=1)
    out, _ = oracle.tree_attn(q, kc, vc, kt, vt, np.array(P), t["n_nodes"], t["anc_mask"])
    G = Hq // Hkv
    for h in range(Hq):
        k = torch.cat([_f64(kc[0, h // G, :P[0]]), _f64(kt[0, :, h // G])])
        v = torch.cat([_f64(vc[0, h // G, :P[0]]), _f64(vt[0, :, h // G])])
        S = P[0] + N + 1
        mask = torch.ones(N + 1, S, dtype=torch.bool).tril(diagonal=P[0])
        ref = torch.nn.functional.scaled_dot_product_attention(
            _f64(q[0, :, h])[None], k[None], v[None], attn_mask=mask[None])[0]
        np.testing.assert_allclose(out[0, :, h], ref.numpy(), rtol=0, atol=1e-12)


def test_tree_attention_root_only_is_decode_attention():
    rng = np.random.default_rng(6)
    q, kc, vc, kt, vt = _attn_inputs(rng, 1, 0, 2, 1, 16, (11,), 11)
    t = _random_tree(rng, 1, 0, L=3, K=2)
    out, _ = oracle.tree_attn(q, kc, vc, kt, vt, np.array([11]), t["n_nodes"], t["anc_mask"])
    for h in range(2):
        k = torch.cat([_f64(kc[0, 0]), _f64(kt[0, :1, 0])])
        v = torch.cat([_f64(vc[0, 0]), _f64(vt[0, :1, 0])])
        ref = torch.nn.functional.scaled_dot_product_attention(_f64(q[0, 0, h])[None, None],
                                                               k[None], v[None])[0, 0]
        np.testing.assert_allclose(out[0, 0, h], ref.numpy(), rtol=0, atol=1e-12)


def test_sibling_mask_rows_differ_only_in_own_bit():
    rng = np.random.default_rng(8)
    t = _random_tree(rng, 1, 40, L=4, K=4)
    par, am = t["parent"][0], t["anc_mask"][0]
    n = t["n_nodes"][0]
    for a in range(1, n + 1):
        for c in range(a + 1, n + 1):
            if par[a] == par[c]:
                diff = am[a] ^ am[c]
                bits = {i for i in range((n + 32) // 32 * 32) if diff[i // 32] >> (i % 32) & 1}
                assert bits == {a, c}


# --------------------------------------------------------------------------
# step 4: decoding rule and acceptance walk
# --------------------------------------------------------------------------

@pytest.mark.parametrize("ctr,key", [([0, 0, 0, 0], [0, 0]), ([3, 9, 0, 0], [0xDD7EE, 0]),
                                     ([2**64 - 1] * 4, [2**64 - 1] * 2),
                                     ([0x243F6A8885A308D3, 0x13198A2E03707344, 0xA4093822299F31D0,
                                       0x082EFA98EC4E6C89], [0x452821E638D01377,
                                                             0xBE5466CF34E90C6C])])
def test_philox_matches_numpy(ctr, key):
    """numpy.random.Philox is Philox4x64-10; it advances its counter by one
    before producing its first block."""
    prev = (sum(c << (64 * i) for i, c in enumerate(ctr)) - 1) % (1 << 256)
    prev_words = [(prev >> (64 * i)) & (2**64 - 1) for i in range(4)]
    bg = np.random.Philox(counter=np.array(prev_words, np.uint64), key=np.array(key, np.uint64))
    np.testing.assert_array_equal(oracle.philox4x64_10(ctr, key), bg.random_raw(4))


def test_uniform_is_top_24_bits():
    x0 = int(oracle.philox4x64_10([2, 5, 0, 0], [77, 3])[0])
    assert oracle.uniform(77, 3, 2, 5) == (x0 >> 40) / 2**24


def _chain(tok_chain, bonus=0):
    n = len(tok_chain)
    R = n + 1
    tree = {"parent": np.arange(-1, n, dtype=np.int32)[None],
            "token": np.array([bonus] + list(tok_chain), np.int32)[None],
            "n_nodes": np.array([n], np.int32)}
    assert tree["parent"].shape == (1, R)
    return tree


def test_greedy_rule_is_argmax_first_index():
    rng = np.random.default_rng(1)
    x = rng.integers(-3, 3, size=(1, 9, 50)).astype(np.float32)   # many ties
    tree = _chain(list(range(1, 9)))
    out = oracle.accept(x, wl.FP32, tree, L=8)
    np.testing.assert_array_equal(out["target_token"][0], np.argmax(x[0], axis=1))


def test_chain_walk_is_vanilla_dflash_acceptance():
    """A single drafted trajectory (§4.1 with K = 1) is vanilla DFlash: accept
    drafted tokens while they equal the target's token at the previous position,
    then emit the target's token at the first mismatch."""
    rng = np.random.default_rng(2)
    L, V = 8, 30
    for trial in range(50):
        draft = rng.integers(0, 4, size=L)
        x = rng.standard_normal((1, L + 1, V)).astype(np.float32)
        tgt = np.argmax(x[0], axis=1)
        k = 0
        while k < L and draft[k] == tgt[k]:
            k += 1
        expect = list(draft[:k]) + [tgt[k]]
        out = oracle.accept(x, wl.FP32, _chain(draft), L=L)
        assert out["accept_len"][0] == k
        np.testing.assert_array_equal(out["out_tokens"][0, :k + 1], expect)
        assert np.all(out["out_tokens"][0, k + 1:] == -1)
        np.testing.assert_array_equal(out["accepted_nodes"][0, :k], np.arange(1, k + 1))
        assert out["next_bonus"][0] == tgt[k]


def test_planted_agreement_follows_rank0_chain():
    """Target row at node u = draft row depth(u), no noise, greedy: every drafted
    top-1 token is accepted, so the walk descends the all-rank-0 chain."""
    w = wl.CONFIGS["tiny"]
    d = wl.draft_logits(w)
    idx, _, lp32, _ = oracle.topk(d, w.dtype, w.K)
    t = oracle.build_tree(lp32, idx, wl.bonus_tokens(w), wl.prefix_lengths(w), w.N)
    rows = np.minimum(np.maximum(t["depth"][0], 0), w.L - 1)
    x = np.ascontiguousarray(d[0][rows][None])
    out = oracle.accept(x, w.dtype, t, L=w.L)
    chain, cur = [], 0
    while True:
        kids = [c for c in range(1, t["n_nodes"][0] + 1)
                if t["parent"][0, c] == cur and t["rank"][0, c] == 0]
        if not kids:
            break
        cur = kids[0]
        chain.append(cur)
    assert out["accept_len"][0] == len(chain)
    np.testing.assert_array_equal(out["accepted_nodes"][0, :len(chain)], chain)


def test_sampling_rule_is_inverse_cdf():
    rng = np.random.default_rng(4)
    V = 40
    x = (rng.standard_normal((1, 6, V)) * 2).astype(np.float32)
    tree = _chain([1, 2, 3, 4, 5])
    for T, step in [(1.0, 0), (0.7, 3), (1.5, 9)]:
        out = oracle.accept(x, wl.FP32, tree, L=5, temperature=T, seed=123, step=step)
        for u in range(6):
            p = np.exp((x[0, u].astype(np.float64) - x[0, u].max()) / T)
            c = np.cumsum(p)
            tgt = oracle.uniform(123, step, 0, u) * c[-1]
            assert out["target_token"][0, u] == np.searchsorted(c, tgt, side="right")
            assert out["margin"][0, u] > 0


def _margin_by_numpy(x64, T, seed, step, b, u):
    """The distance from U*Z to the nearest edge of the sampled token's CDF bin,
    over Z, written from the definition with numpy (fp64 sequential cumsum,
    searchsorted): bin t = [C_{t-1}, C_t) with C_{-1} = 0."""
    p = np.exp((x64 - x64.max()) / T)
    c = np.cumsum(p)
    z = c[-1]
    tgt = oracle.uniform(seed, step, b, u) * z
    t = int(np.searchsorted(c, tgt, side="right"))
    lo = c[t - 1] if t > 0 else 0.0
    return t, min(tgt - lo, c[t] - tgt) / z


@pytest.mark.parametrize("V,T,flat", [(40, 1.0, False), (1000, 1.0, False), (1000, 0.5, True),
                                      (151936, 1.0, False)])
def test_sampling_margin_is_distance_to_nearest_cdf_edge(V, T, flat):
    """The oracle's per-node margin (the band the T > 0 GPU parity check admits)
    equals min(U*Z - C_{t-1}, C_t - U*Z) / Z for every node, recomputed from the
    definition; the flat rows put many tokens of similar mass next to U*Z."""
    rng = np.random.default_rng(V + int(10 * T))
    R = 6 if V > 10000 else 31
    x = (rng.standard_normal((2, R, V)) * (0.05 if flat else 2.5)).astype(np.float32)
    par = np.array([[-1] + [max(0, (u - 1) // 2) for u in range(1, R)]] * 2, np.int32)
    tree = {"parent": par, "token": rng.integers(0, V, size=(2, R)).astype(np.int32),
            "n_nodes": np.array([R - 1, R - 3], np.int32)}
    for seed, step in [(11, 0), (0xDD7EE, 5)]:
        out = oracle.accept(x, wl.FP32, tree, L=4, temperature=T, seed=seed, step=step)
        for b in range(2):
            n = tree["n_nodes"][b]
            for u in range(n + 1):
                t, mg = _margin_by_numpy(x[b, u].astype(np.float64), T, seed, step, b, u)
                assert out["target_token"][b, u] == t
                assert abs(out["margin"][b, u] - mg) <= 1e-12, (b, u)
            assert np.all(np.isinf(out["margin"][b, n + 1:]))
    # greedy: no band at all
    out = oracle.accept(x, wl.FP32, tree, L=4, temperature=0.0)
    assert np.all(np.isinf(out["margin"]))


@pytest.mark.slow
def test_sampling_frequencies_match_softmax():
    from scipy.stats import chisquare
    rng = np.random.default_rng(9)
    V = 12
    x = (rng.standard_normal((1, 1, V)) * 1.5).astype(np.float32)
    tree = {"parent": np.array([[-1]], np.int32), "token": np.array([[0]], np.int32),
            "n_nodes": np.array([0], np.int32)}
    draws = [oracle.accept(x, wl.FP32, tree, L=1, temperature=1.0, seed=5, step=s)
             ["target_token"][0, 0] for s in range(20000)]
    p = np.exp(x[0, 0].astype(np.float64) - x[0, 0].max())
    p /= p.sum()
    obs = np.bincount(draws, minlength=V)
    assert chisquare(obs, p * len(draws)).pvalue > 1e-4


# --------------------------------------------------------------------------
# after the walk: committing the accepted path to the KV cache
# --------------------------------------------------------------------------

def _commit_case(seed, B=3, N=20, Hkv=2, D=16, L=5, K=3, cap=40):
    rng = np.random.default_rng(seed)
    P = rng.integers(0, cap - L - 1, size=B).astype(np.int32)
    q, kc, vc, kt, vt = _attn_inputs(rng, B, N, 2 * Hkv, Hkv, D, list(P), cap)
    t = _random_tree(rng, B, N, L=L, K=K)
    # an accepted path per sequence: follow a random child from the root
    acc = np.full((B, L), -1, np.int32)
    alen = np.zeros(B, np.int32)
    for b in range(B):
        cur, depth = 0, 0
        while depth < L:
            kids = [c for c in range(1, t["n_nodes"][b] + 1) if t["parent"][b, c] == cur]
            if not kids or rng.random() < 0.2:
                break
            cur = int(rng.choice(kids))
            acc[b, depth] = cur
            depth += 1
        alen[b] = depth
    return q, kc, vc, kt, vt, P, t, acc, alen


def test_commit_is_a_gather_of_the_root_path():
    """§4.1: the bonus token (the root) and the accepted tokens join the
    prefix, in path order, at positions P..P+a; nothing else changes."""
    for seed in range(4):
        q, kc, vc, kt, vt, P, t, acc, alen = _commit_case(seed)
        k2, v2, p2 = oracle.commit(kc, vc, kt, vt, alen, acc, P)
        np.testing.assert_array_equal(p2, P + alen + 1)
        for b in range(len(P)):
            rows = np.concatenate([[0], acc[b, :alen[b]]])
            seg = slice(P[b], P[b] + alen[b] + 1)
            # numpy's gather of the tree rows, transposed to [Hkv][a+1][D]
            np.testing.assert_array_equal(k2[b, :, seg], np.take(kt[b], rows, axis=0).transpose(1, 0, 2))
            np.testing.assert_array_equal(v2[b, :, seg], np.take(vt[b], rows, axis=0).transpose(1, 0, 2))
            keep = np.ones(kc.shape[2], bool)
            keep[seg] = False
            np.testing.assert_array_equal(k2[b][:, keep].view(np.uint16), kc[b][:, keep])
            np.testing.assert_array_equal(v2[b][:, keep].view(np.uint16), vc[b][:, keep])


def test_commit_then_decode_equals_tree_attention_of_the_last_accepted_node():
    """The committed rows are exactly the last accepted node's root path, so its
    tree-attention row (prefix + ancestors) equals plain attention of the same
    query over the extended cache (torch SDPA, fp64)."""
    q, kc, vc, kt, vt, P, t, acc, alen = _commit_case(11)
    out, _ = oracle.tree_attn(q, kc, vc, kt, vt, P, t["n_nodes"], t["anc_mask"])
    k2, v2, p2 = oracle.commit(kc, vc, kt, vt, alen, acc, P)
    Hq, Hkv = q.shape[2], kc.shape[1]
    G = Hq // Hkv
    for b in range(len(P)):
        u = 0 if alen[b] == 0 else int(acc[b, alen[b] - 1])
        for h in range(Hq):
            k = _f64(k2[b, h // G, :p2[b]])
            v = _f64(v2[b, h // G, :p2[b]])
            ref = torch.nn.functional.scaled_dot_product_attention(
                _f64(q[b, u, h])[None, None], k[None], v[None])[0, 0]
            np.testing.assert_allclose(out[b, u, h], ref.numpy(), rtol=0, atol=1e-12)


def test_commit_rejects_bad_paths():
    q, kc, vc, kt, vt, P, t, acc, alen = _commit_case(3)
    with pytest.raises(ValueError):
        oracle.commit(kc, vc, kt, vt, np.full_like(alen, 6), acc, P)  # longer than L
    bad = acc.copy()
    bad[0, 0] = 21  # past the tree
    with pytest.raises(ValueError):
        oracle.commit(kc, vc, kt, vt, np.maximum(alen, 1), bad, P)
    with pytest.raises(ValueError):
        oracle.commit(kc, vc, kt, vt, alen, acc, np.full_like(P, kc.shape[2] - alen.min()))
