"""GPU parity of step 2 (best-first heap tree build) against the oracle.
Criterion: every output array bit-exact when both sides are fed the oracle's
own fp32 log-prob table."""
import numpy as np
import pytest

import oracle
from diffusion_draft_tree_gb300 import ops
from diffusion_draft_tree_gb300 import workloads as wl
from tests.gpu_util import dev_f32, dev_i32, host

pytestmark = pytest.mark.gpu
KEYS = ("parent", "depth", "rank", "token", "pos_id", "child_count", "n_nodes")


def _check(lp32, tok, bonus, plen, N, dev, heap):
    ref = oracle.build_tree(lp32, tok, bonus, plen, N)
    got = ops.build(dev_f32(lp32, dev), dev_i32(tok, dev), dev_i32(bonus, dev),
                    dev_i32(plen, dev), N, heap=heap)
    for k in KEYS:
        np.testing.assert_array_equal(host(got[k]), ref[k], err_msg=k)
    np.testing.assert_array_equal(host(got["score"]).view(np.uint32),
                                  ref["score"].view(np.uint32))
    np.testing.assert_array_equal(host(got["anc_mask"]).view(np.uint32), ref["anc_mask"])
    ops.ddtree_device_check()
    return ref


@pytest.mark.parametrize("name", ["tiny", "8b_single", "budget_sweep_n32", "budget_sweep_n128",
                                  "budget_sweep_n256", "budget_sweep_n512", "ragged_serving",
                                  "long_context_70b"])
@pytest.mark.parametrize("heap", [False, True], ids=["level", "heap"])
def test_build_workloads(cuda_device, name, heap):
    w = wl.CONFIGS[name]
    idx, _, lp32, _ = oracle.topk(wl.draft_logits(w), w.dtype, w.K)
    ref = _check(lp32, idx, wl.bonus_tokens(w), wl.prefix_lengths(w), w.N, cuda_device, heap)
    assert np.all(ref["n_nodes"] == w.N)


def _table(rng, B, L, K, ties):
    if ties:
        lp = -rng.integers(1, 5, size=(B, L, K)).astype(np.float32) / 4
    else:
        lp = -rng.exponential(1.5, size=(B, L, K)).astype(np.float32)
    lp = -np.sort(-lp, axis=2)
    tok = rng.integers(0, 150000, size=(B, L, K)).astype(np.int32)
    return lp, tok


@pytest.mark.parametrize("B,L,K,N,ties", [
    (1, 16, 32, 1024, False), (2, 16, 32, 1024, True), (3, 4, 4, 16, True), (1, 16, 1, 20, False),
    (2, 3, 2, 40, False),      # fewer prefixes (14) than the budget
    (1, 5, 3, 0, False),       # root only
    (4, 1, 7, 7, True),        # one position
    (1, 16, 16, 543, True), (1, 16, 16, 544, True), (1, 9, 5, 95, False), (1, 9, 5, 96, False),
    (5, 16, 8, 63, True), (5, 16, 8, 64, False),
    # 128-thread build with more children than its register cache holds (level 3
    # recomputes the keys every pass) and an N-th-key select with a tie group
    (2, 16, 32, 64, False), (2, 16, 32, 64, True), (1, 8, 32, 60, False)])
@pytest.mark.parametrize("heap", [False, True], ids=["level", "heap"])
def test_build_edge_cases(cuda_device, B, L, K, N, ties, heap):
    rng = np.random.default_rng(B * 1000 + L * 100 + K * 10 + N)
    lp, tok = _table(rng, B, L, K, ties)
    bonus = rng.integers(0, 1000, size=B).astype(np.int32)
    plen = rng.integers(0, 5000, size=B).astype(np.int32)
    _check(lp, tok, bonus, plen, N, cuda_device, heap)
