"""CPU-only checks of the C-ABI library: it loads without a GPU driver, exports
every entry point include/ddtree.h declares, and rejects bad arguments on the
host before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build_library()
    from diffusion_draft_tree_gb300 import ops
    return ops


def _declared():
    with open(os.path.join(ROOT, "include", "ddtree.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(ddtree_\w+)\s*\(", text, re.M)))


def test_header_declares_the_round(lib):
    names = _declared()
    for n in ("ddtree_topk", "ddtree_build", "ddtree_tree_attn", "ddtree_accept",
              "ddtree_accept_path", "ddtree_commit", "ddtree_workspace_size",
              "ddtree_device_check", "ddtree_status_str"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for n in _declared():
        assert hasattr(so, n), n


def test_status_strings(lib):
    for s in range(5):
        assert lib.lib.ddtree_status_str(s)


def test_workspace_sizes(lib):
    # 8B-class single stream: 16 rows of V=151936 bf16 split into chunks
    assert lib.workspace_size(lib.OP_TOPK, B=1, L=16, V=151936, dtype=lib.BF16) > 0
    # a tiny vocabulary fits one chunk, which still leaves one partial per row
    small = lib.workspace_size(lib.OP_TOPK, B=1, L=4, V=1000, K=4, dtype=lib.FP32)
    assert 0 < small < lib.workspace_size(lib.OP_TOPK, B=1, L=16, V=151936, dtype=lib.BF16)
    assert lib.workspace_size(lib.OP_ACCEPT, B=1, N=64, V=151936, dtype=lib.BF16) > 0
    # tree attention merges its KV splits on chip (cluster shared memory)
    assert lib.workspace_size(lib.OP_TREE_ATTN, B=1, N=64, Hq=32, Hkv=8, D=128,
                              cache_cap=2048) == 0
    assert lib.workspace_size(lib.OP_TOPK, B=0, L=1, V=10) == 0


def test_invalid_arguments_rejected_before_launch(lib):
    L = lib.lib
    P = ctypes.c_void_p
    fake = P(0x1000)
    # null logits
    assert L.ddtree_topk(None, 0, 1, 10, 10, 2, fake, fake, None, None, 0, None) == 1
    # K > V
    assert L.ddtree_topk(fake, 0, 1, 4, 4, 5, fake, fake, None, None, 0, None) == 1
    # K above the implementation limit
    assert L.ddtree_topk(fake, 0, 1, 4000, 4000, 33, fake, fake, None, None, 0, None) == 2
    # row stride shorter than a row
    assert L.ddtree_topk(fake, 0, 1, 10, 9, 2, fake, fake, None, None, 0, None) == 1
    # unsupported head dim / non power-of-two group
    args = [fake, fake, fake, 64, fake, fake, fake, fake, fake, 1, 4, 8, 2, 96, 0.1, fake, None,
            None, 0, None]
    assert L.ddtree_tree_attn(*args) == 2
    args[11], args[12], args[13] = 12, 4, 128  # G = 3
    assert L.ddtree_tree_attn(*args) == 2
    args[11], args[12] = 8, 3  # Hq % Hkv != 0
    assert L.ddtree_tree_attn(*args) == 1
    # budget above the limit
    assert L.ddtree_build(fake, fake, fake, fake, 1, 4, 4, 5000, *([fake] * 9), None) == 2
    # negative temperature
    assert L.ddtree_accept(fake, 0, 10, fake, fake, fake, 1, 4, 4, 10, -1.0, 0, 0, None, fake,
                           fake, fake, fake, fake, 1 << 20, None) == 1
    # accept without workspace
    assert L.ddtree_accept(fake, 0, 10, fake, fake, fake, 1, 4, 4, 10, 0.0, 0, 0, None, fake,
                           fake, fake, fake, None, 0, None) == 1
    # path-only accept: negative temperature, budget above the limit
    assert L.ddtree_accept_path(fake, 0, 10, fake, fake, fake, 1, 4, 4, 10, -1.0, 0, 0, None,
                                fake, fake, fake, fake, None) == 1
    assert L.ddtree_accept_path(fake, 0, 10, fake, fake, fake, 1, 4, 5000, 10, 0.0, 0, 0, None,
                                fake, fake, fake, fake, None) == 2
    # commit: null cache, a head dimension that is not a multiple of 8, unaligned K/V
    assert L.ddtree_commit(None, fake, 64, fake, fake, fake, fake, fake, 1, 4, 8, 2, 64,
                           None) == 1
    assert L.ddtree_commit(fake, fake, 64, fake, fake, fake, fake, fake, 1, 4, 8, 2, 60,
                           None) == 2
    assert L.ddtree_commit(P(0x1008), fake, 64, fake, fake, fake, fake, fake, 1, 4, 8, 2, 64,
                           None) == 1


def test_misaligned_element_arrays_rejected(lib):
    """Every int32 / uint32 / float array off its 4-byte grid is refused on the
    host (a device access through it would fault); the other arguments of each
    call are well formed, so the misaligned pointer is the only fault."""
    L = lib.lib
    P = ctypes.c_void_p
    ok, odd = P(0x10000), P(0x10002)
    ws, wsb = P(0x100000), 1 << 24
    for i in range(3):  # top-K: indices, log-probs, logsumexp
        outs = [ok, ok, ok]
        outs[i] = odd
        assert L.ddtree_topk(ok, 0, 1, 1000, 1000, 4, *outs, ws, wsb, None) == 1
    for i in range(13):  # the build's inputs and outputs
        ptrs = [ok] * 13
        ptrs[i] = odd
        assert L.ddtree_build(*ptrs[:4], 1, 4, 4, 16, *ptrs[4:], None) == 1
        assert L.ddtree_build_heap(*ptrs[:4], 1, 4, 4, 16, *ptrs[4:], None) == 1
    for i in range(4):  # tree attention: prefix lengths, tree sizes, mask, lse
        p4 = [ok] * 4
        p4[i] = odd
        assert L.ddtree_tree_attn(ok, ok, ok, 64, ok, ok, p4[0], p4[1], p4[2], 1, 16, 2, 1, 64,
                                  0.125, ok, p4[3], ws, wsb, None) == 1
    for i in range(8):  # both walks: tree arrays and outputs
        p8 = [ok] * 8
        p8[i] = odd
        common = [ok, 0, 1000, p8[0], p8[1], p8[2], 1, 4, 16, 1000, 0.0, 1, 0, *p8[3:]]
        assert L.ddtree_accept(*common, ws, wsb, None) == 1
        assert L.ddtree_accept_path(*common, None) == 1
    # the no-workspace top-K checks the same
    assert L.ddtree_topk_noalloc(ok, 0, 1, 1000, 1000, 4, odd, ok, None, None) == 1


def test_selftest_rejects_limits_out_of_range_on_the_host(lib):
    """Checked before anything is enqueued: no GPU needed."""
    L = ctypes.CDLL(lib.LIB_PATH)
    L.ddtree_selftest_wait.argtypes = [ctypes.c_uint32, ctypes.c_void_p]
    L.ddtree_selftest_wait.restype = ctypes.c_int
    assert L.ddtree_selftest_wait(0, None) == 1
    assert L.ddtree_selftest_wait(1000001, None) == 1
