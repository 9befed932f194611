"""GPU parity of step 1 (log-softmax + top-K) against the oracle.
Criteria: indices bit-exact; log-probs and logsumexp within 1e-5 absolute of
the oracle's fp64 values.  Rows are streamed in 4 KB segments by warps that
each take an equal run of them, so a row is cut into one or many pieces and a
warp's run may cross many rows; the edge shapes run once as they are (six
rows: a row spans many warps) and once with their rows repeated 64 times
(longer runs, crossing row ends)."""
import numpy as np
import pytest
import torch

import oracle
from diffusion_draft_tree_gb300 import ops
from diffusion_draft_tree_gb300 import workloads as wl
from tests.gpu_util import dev_logits, host

pytestmark = pytest.mark.gpu
TOL = 1e-5


def _check(raw, dtype, K, dev, unaligned=False):
    rows, V = raw.shape
    o_idx, o_lp64, _, o_lse = oracle.topk(raw, dtype, K)
    x = dev_logits(raw, dtype, dev)
    if unaligned:  # same values, row starts shifted off the 16-byte grid
        buf = torch.empty(rows * V + 1, dtype=x.dtype, device=dev)
        buf[1:] = x.reshape(-1)
        x = buf[1:].view(rows, V)
        assert x.data_ptr() % 16 != 0
    idx, lp, lse = ops.topk(x, K)
    np.testing.assert_array_equal(host(idx), o_idx)
    assert np.abs(host(lp) - o_lp64).max() <= TOL
    assert np.abs(host(lse) - o_lse).max() <= TOL
    ops.ddtree_device_check()


@pytest.mark.parametrize("name", ["tiny", "8b_single", "budget_sweep_n64", "long_context_70b",
                                  "ragged_serving"])
def test_topk_workloads(cuda_device, name):
    w = wl.CONFIGS[name]
    raw = wl.draft_logits(w).reshape(w.B * w.L, w.V)
    _check(raw, w.dtype, w.K, cuda_device)


@pytest.mark.parametrize("V,K,dtype,unaligned", [
    (1001, 3, wl.BF16, False), (1001, 3, wl.BF16, True), (8191, 16, wl.BF16, False),
    (16384, 32, wl.BF16, False), (16385, 1, wl.BF16, True), (40000, 8, wl.FP32, False),
    (40001, 8, wl.FP32, True), (50, 32, wl.BF16, False), (7, 1, wl.FP32, False),
    (151936, 2, wl.BF16, False), (300000, 16, wl.BF16, False)])
@pytest.mark.parametrize("reps", [1, 64])
def test_topk_edge_shapes_and_ties(cuda_device, V, K, dtype, unaligned, reps):
    if reps > 1 and V > 100000:
        pytest.skip("the long-row workloads above already stream many rows per warp")
    rng = np.random.default_rng(V + K)
    x = (rng.standard_normal((6, V)) * 3).astype(np.float32)
    x[1, :] = 0.0                                     # a constant row: ties everywhere
    top = x[2].max() + 1
    x[2, [3, V // 2, V - 1]] = top                    # equal maxima far apart
    x[3, ::2] = np.float32(-0.0)                      # signed zeros tie by index
    x[3, 1::2] = np.float32(0.0)
    x[4, :] = np.round(x[4] * 2) / 2                  # heavy quantisation: many ties
    x = np.tile(x, (reps, 1))
    raw = wl.bf16_bits(x) if dtype == wl.BF16 else x
    _check(raw, dtype, K, cuda_device, unaligned)


def test_topk_spike_is_top1(cuda_device):
    w = wl.CONFIGS["8b_single"]
    raw = wl.draft_logits(w).reshape(w.L, w.V)
    idx, _, _ = ops.topk(dev_logits(raw, w.dtype, cuda_device), w.K)
    np.testing.assert_array_equal(host(idx)[:, 0], np.argmax(wl.bf16_to_f32(raw), axis=1))


def test_topk_leaves_its_workspace_zero_and_reuses_it_across_sizes(cuda_device):
    """Every top-K call returns the workspace it used to zero (row counters,
    row bounds and piece slots), so one workspace serves calls of different
    sizes one after another; each result still matches the oracle."""
    w1, w2 = wl.CONFIGS["8b_single"], wl.CONFIGS["long_context_70b"]
    cases = [(wl.draft_logits(w2).reshape(w2.B * w2.L, w2.V), w2.dtype, 16),
             (wl.draft_logits(w1).reshape(w1.B * w1.L, w1.V), w1.dtype, w1.K),
             (wl.draft_logits(w2).reshape(w2.B * w2.L, w2.V)[:5], w2.dtype, 3)]
    need = max(ops.workspace_size(ops.OP_TOPK, B=r.shape[0], L=1, V=r.shape[1], K=K, dtype=d)
               for r, d, K in cases)
    ws = ops.alloc_workspace(need, cuda_device)
    for raw, dtype, K in cases:
        o_idx, o_lp64, _, o_lse = oracle.topk(raw, dtype, K)
        idx, lp, lse = ops.topk(dev_logits(raw, dtype, cuda_device), K, workspace=ws)
        ops.ddtree_device_check()
        np.testing.assert_array_equal(host(idx), o_idx)
        assert np.abs(host(lp) - o_lp64).max() <= TOL
        assert np.abs(host(lse) - o_lse).max() <= TOL
        assert int(torch.count_nonzero(ws)) == 0
