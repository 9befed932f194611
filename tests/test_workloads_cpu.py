"""The seeded input generators (diffusion_draft_tree_gb300/workloads.py), which
feed both the CUDA path and the oracle: bf16 rounding against torch's own
round-to-nearest-even conversion, determinism, independent streams, and the
recipe each workload states (spike, ragged prefixes, NaN poison where no
kernel may read, target rows built from the draft row at the node's depth)."""
import numpy as np
import torch

from diffusion_draft_tree_gb300 import workloads as wl


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32),
        # exact halfway points between neighbouring bf16 values (both signs,
        # even and odd lower neighbours): ties to even
        ((np.concatenate([np.arange(0x3F80, 0x4080), np.arange(0xBF80, 0xC080)])
          .astype(np.uint32) << np.uint32(16)) | np.uint32(0x8000)).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, -3.3895314e38], np.float32)])
    ours = wl.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    # widening is exact, and rounding a bf16 value gives it back
    back = wl.bf16_to_f32(ours)
    np.testing.assert_array_equal(wl.bf16_bits(back), ours)


def test_generators_are_deterministic_and_streams_independent():
    w = wl.CONFIGS["tiny"]
    np.testing.assert_array_equal(wl.draft_logits(w), wl.draft_logits(w))
    np.testing.assert_array_equal(wl.queries(w), wl.queries(w))
    k = wl.kv_cache(w, 0)
    np.testing.assert_array_equal(k[0, 0], wl.kv_cache_slice(w, 0, 0, 0))
    # K and V caches, tree K and V, queries: different streams, different draws
    assert not np.array_equal(wl.kv_cache(w, 0), wl.kv_cache(w, 1))
    assert not np.array_equal(wl.kv_tree(w, 0), wl.kv_tree(w, 1))
    assert not np.array_equal(wl.queries(w)[0, :, 0, :], wl.kv_tree(w, 0)[0, :, 0, :])


def test_draft_rows_scale_and_spike():
    w = wl.CONFIGS["8b_single"].with_(V=20000, dtype=wl.FP32)
    x = wl.draft_logits(w)
    plain = wl.draft_logits(w.with_(spike=None))
    diff = x - plain
    hit = np.abs(diff) > 1e-3
    # exactly one spiked token per (sequence, position), raised by the spike
    np.testing.assert_array_equal(hit.sum(axis=-1), np.ones((w.B, w.L)))
    np.testing.assert_allclose(diff[hit], 6.0, atol=1e-5)
    # the rest is draft_scale * N(0, 1): mean and std within five standard errors
    n = plain.size
    assert abs(plain.mean()) < 5 * 3.0 / np.sqrt(n)
    assert abs(plain.std() - 3.0) < 5 * 3.0 / np.sqrt(2 * n)


def test_ragged_prefixes_and_cache_poison():
    w = wl.CONFIGS["ragged_serving"]
    P = np.asarray(w.P)
    assert len(P) == w.B == 16 and P.min() >= 1024 and P.max() <= 32768
    assert len(set(P.tolist())) > 1  # ragged
    small = w.with_(P=(5, 0, 17), B=3, D=64, Hkv=2)
    k = wl.kv_cache(small, 0, cap=24)
    for b, p in enumerate(small.P):
        assert (k[b, :, p:] == wl.BF16_NAN).all()           # never read
        assert np.isfinite(wl.bf16_to_f32(k[b, :, :p])).all()


def test_target_rows_follow_the_draft_row_at_the_node_depth():
    w = wl.CONFIGS["tiny"]  # fp32 rows, so the sum is exact to check
    draft = wl.draft_logits(w)
    depth = np.array([[0, 1, 1, 2, 3, 4, 5] + [-1] * (w.N + 1 - 7)], np.int32)
    t = wl.target_logits(w, draft, depth)
    noise = wl.target_noise(w, 0)
    for u in range(7):
        np.testing.assert_array_equal(t[0, u], draft[0, min(depth[0, u], w.L - 1)] + noise[u])
    assert np.isnan(t[0, 7:]).all()  # padding rows are poisoned
