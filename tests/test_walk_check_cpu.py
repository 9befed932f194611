"""CPU checks of the test-side step-4 helpers (tests/walk_check.py) that the
GPU parity tests use at temperature > 0: the replayed walk reproduces the
oracle's walk from the oracle's own tokens, and the band check accepts the
oracle's token and the tokens across a nearby CDF edge only."""
import numpy as np

import oracle
from diffusion_draft_tree_gb300 import workloads as wl
from tests import walk_check


def _tree(w):
    draft = wl.draft_logits(w)
    idx, _, lp32, _ = oracle.topk(draft, w.dtype, w.K)
    return draft, oracle.build_tree(lp32, idx, wl.bonus_tokens(w), wl.prefix_lengths(w), w.N)


def test_replayed_walk_equals_oracle_walk():
    for T in (0.0, 1.0):
        w = wl.CONFIGS["tiny"].with_(B=3, P=(64, 10, 0), T=T)
        draft, t = _tree(w)
        x = wl.target_logits(w, draft, t["depth"])
        ref = oracle.accept(x, w.dtype, t, w.L, temperature=T, seed=3, step=1)
        for b in range(w.B):
            got = walk_check.walk(t["parent"][b], t["token"][b], t["n_nodes"][b],
                                  ref["target_token"][b], w.L)
            for k in ("accept_len", "accepted_nodes", "out_tokens", "next_bonus"):
                np.testing.assert_array_equal(got[k], ref[k][b], err_msg=k)


def test_band_accepts_only_the_edge_neighbours():
    rng = np.random.default_rng(5)
    V, T = 50, 1.0
    x = rng.standard_normal((1, 1, V)).astype(np.float32)
    row = walk_check.row_f64(x, wl.FP32, 0, 0)
    ref = oracle.accept(x, wl.FP32, {"parent": np.array([[-1]], np.int32),
                                     "token": np.array([[0]], np.int32),
                                     "n_nodes": np.array([0], np.int32)}, L=1, temperature=T,
                        seed=8, step=2)
    t = int(ref["target_token"][0, 0])
    d, ok = walk_check.sample_in_band(row, T, 8, 2, 0, 0, t, 1e-5)
    assert ok and d == 0.0
    # a token two bins away is never within a band smaller than the bin between
    for other in (t - 2, t + 2):
        if 0 <= other < V:
            _, ok = walk_check.sample_in_band(row, T, 8, 2, 0, 0, other, 1e-5)
            assert not ok
    # the distances to the two neighbours' bins are the distances to the two
    # edges of t's bin; the nearer one is the oracle's margin
    assert 0 < t < V - 1
    d_up, _ = walk_check.sample_in_band(row, T, 8, 2, 0, 0, t + 1, 1.0)
    d_dn, _ = walk_check.sample_in_band(row, T, 8, 2, 0, 0, t - 1, 1.0)
    assert abs(min(d_up, d_dn) - ref["margin"][0, 0]) <= 1e-12
