"""Failure reporting without a GPU fault.  Every wait inside the library's
kernels (a bulk copy landing, the tensor core finishing, another warp's
results) is bounded in wall time; when the bound passes the kernel records a
timeout in the device error word and unwinds.  ddtree_selftest_wait runs that
same bounded wait on a barrier nothing ever signals: the host must read the
timeout, the error word must clear, and the CUDA context must still serve a
normal call afterwards.  Nothing here faults a GPU; the wait always ends."""
import numpy as np
import pytest

import oracle
from diffusion_draft_tree_gb300 import ops
from diffusion_draft_tree_gb300 import workloads as wl
from tests.gpu_util import dev_logits, host

pytestmark = pytest.mark.gpu

SELFTEST_TIMEOUT = 0x0F000004  # stage 15 (self-test), reason 4 (a bounded wait timed out)


def test_bounded_wait_reports_a_timeout_and_the_context_survives(cuda_device):
    ops.ddtree_device_check()  # nothing pending before
    ops.ddtree_selftest_wait(20000)  # 20 ms
    with pytest.raises(ops.DDTreeError) as e:
        ops.ddtree_device_check()
    assert e.value.status == 4 and e.value.detail == SELFTEST_TIMEOUT
    ops.ddtree_device_check()  # read once, then cleared

    # the context is intact: a normal call right after matches the oracle
    w = wl.CONFIGS["tiny"]
    raw = wl.draft_logits(w).reshape(w.B * w.L, w.V)
    idx, lp, lse = ops.topk(dev_logits(raw, w.dtype, cuda_device), w.K)
    o_idx, o_lp64, _, o_lse = oracle.topk(raw, w.dtype, w.K)
    np.testing.assert_array_equal(host(idx), o_idx)
    assert np.abs(host(lp) - o_lp64).max() <= 1e-5
    ops.ddtree_device_check()


def test_selftest_rejects_limits_out_of_range(cuda_device):
    for bad in (0, 1000001):
        with pytest.raises(ops.DDTreeError) as e:
            ops.ddtree_selftest_wait(bad)
        assert e.value.status == 1
    ops.ddtree_device_check()
