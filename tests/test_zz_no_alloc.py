"""ddtree_topk_noalloc: top-K for callers that may not allocate device memory
(code inside a host framework whose memory pool it does not own, or a path
where cudaMalloc's implicit synchronisation is not allowed), so cannot hand
the library a workspace.  The entry point uses a fixed scratch array built into
the library instead.

It must give the oracle's answer (indices bit-exact, log-probs and logsumexp
within the 1e-5 of fp64 that the other top-K tests use) and the same answer as
ddtree_topk, on two calls in a row -- the second with a different shape, so
stale partials left in the shared array by the first call would show -- and
leave the device error word clear after each.  This file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from diffusion_draft_tree_gb300 import ops
from diffusion_draft_tree_gb300 import workloads as wl
from tests.gpu_util import dev_logits, host

TOL = 1e-5
SCRATCH_BYTES = 1 << 20


def _noalloc():
    f = ops.lib.ddtree_topk_noalloc
    P = ctypes.c_void_p
    f.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int, P,
                  P, P, P]
    f.restype = ctypes.c_int
    return f


def _call_noalloc(x: torch.Tensor, K: int):
    rows, V = x.shape
    idx = torch.full((rows, K), -7, dtype=torch.int32, device=x.device)
    lp = torch.full((rows, K), float("nan"), dtype=torch.float32, device=x.device)
    lse = torch.full((rows,), float("nan"), dtype=torch.float32, device=x.device)
    st = _noalloc()(ctypes.c_void_p(x.data_ptr()), ops.BF16 if x.dtype == torch.bfloat16
                    else ops.FP32, rows, V, V, K, ctypes.c_void_p(idx.data_ptr()),
                    ctypes.c_void_p(lp.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, ops.STATUS.get(st, st)
    return idx, lp, lse


@pytest.mark.gpu
def test_noalloc_topk_matches_workspace_topk_twice(cuda_device):
    first = wl.CONFIGS["8b_single"]
    second = wl.CONFIGS["long_context_70b"]
    cases = [(wl.draft_logits(first).reshape(first.B * first.L, first.V), first.dtype, first.K),
             (wl.draft_logits(second).reshape(second.B * second.L, second.V), second.dtype, 16)]
    for raw, dtype, K in cases:
        o_idx, o_lp64, _, o_lse = oracle.topk(raw, dtype, K)
        x = dev_logits(raw, dtype, cuda_device)
        need = ops.workspace_size(ops.OP_TOPK, B=x.shape[0], L=1, V=x.shape[1], K=K,
                                  dtype=dtype)
        assert 0 < need <= SCRATCH_BYTES
        idx, lp, lse = _call_noalloc(x, K)
        ops.ddtree_device_check()  # raises if a kernel recorded an error
        np.testing.assert_array_equal(host(idx), o_idx)
        assert np.abs(host(lp) - o_lp64).max() <= TOL
        assert np.abs(host(lse) - o_lse).max() <= TOL
        ref_idx, ref_lp, ref_lse = ops.topk(x, K)
        ops.ddtree_device_check()
        np.testing.assert_array_equal(host(idx), host(ref_idx))
        assert np.abs(host(lp) - host(ref_lp)).max() <= TOL
        assert np.abs(host(lse) - host(ref_lse)).max() <= TOL


def test_noalloc_rejects_problems_beyond_its_scratch():
    """Sizes are checked on the host before anything is enqueued: no GPU needed."""
    f = _noalloc()
    fake = ctypes.c_void_p(0x1000)
    rows = 20000  # 20000 rows of a 151936-token bf16 vocabulary need ~1.9 MB at K = 8
    assert ops.workspace_size(ops.OP_TOPK, B=rows, L=1, V=151936, K=8,
                              dtype=ops.BF16) > SCRATCH_BYTES
    assert f(fake, ops.BF16, rows, 151936, 151936, 8, fake, fake, None, None) == 2
