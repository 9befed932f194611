"""CPU oracle for one DDTree round (TEST INFRASTRUCTURE ONLY).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it and must fail loudly when its CUDA
extension is missing instead of falling back here.

The arithmetic lives in ``ddtree_oracle.c`` (plain C, fp64); this module only
compiles it with gcc on first use and marshals numpy arrays through ctypes.
Each function cites the passage of "Accelerating Speculative Decoding with
Block Diffusion Draft Trees" (paperlayer.ai summary) that it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ddtree_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "libddtree_oracle.so")
_lock = threading.Lock()
_lib = None

BF16, FP32 = 0, 1


def _compile(src: str, so: str) -> None:
    """gcc with portable flags: the same source runs on x86 and Arm."""
    tmp = so + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, so)


def build(force: bool = False) -> str:
    """Compile the oracle (once; again when the source is newer)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        _compile(_SRC, _SO)
    return _SO


def _bind(lib):
    """Declares the C signatures on a loaded oracle library."""
    P = ctypes.c_void_p
    i32, i64, f64, u64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_uint64
    lib.ddo_topk.argtypes = [P, i32, i32, i32, i64, i32, P, P, P, P]
    lib.ddo_build.argtypes = [P, P, P, P, i32, i32, i32, i32] + [P] * 9
    lib.ddo_tree_attn_unit.argtypes = [i32, i32, i32, i32, P, P, P, i64, P, P, P, P, P, i32, i32,
                                       i32, i32, i32, f64, P, P]
    lib.ddo_tree_attn.argtypes = [P, P, P, i64, P, P, P, P, P, i32, i32, i32, i32, i32, f64, P,
                                  P]
    lib.ddo_philox4x64_10.argtypes = [P, P, P]
    lib.ddo_uniform.argtypes = [u64, u64, u64, u64]
    lib.ddo_uniform.restype = f64
    lib.ddo_accept.argtypes = [P, i32, i64, P, P, P, i32, i32, i32, i32, f64, u64, u64, P, P,
                               P, P, P, P]
    lib.ddo_commit.argtypes = [P, P, i64, P, P, P, P, P, i32, i32, i32, i32, i32]
    for f in (lib.ddo_topk, lib.ddo_build, lib.ddo_tree_attn_unit, lib.ddo_tree_attn,
              lib.ddo_accept, lib.ddo_commit):
        f.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments")


def topk(logits: np.ndarray, dtype: int, K: int):
    """Log-softmax and top-K of every row (pages §3: per-position marginals;
    §4.3: work in log-probabilities).  ``logits`` is [..., V] (uint16 bf16 bits
    or float32).  Returns (idx int32 [...,K], logp64 [...,K], logp32 [...,K],
    lse float64 [...])."""
    logits = np.ascontiguousarray(logits)
    *lead, V = logits.shape
    rows = int(np.prod(lead)) if lead else 1
    idx = np.empty((rows, K), np.int32)
    lp64 = np.empty((rows, K), np.float64)
    lp32 = np.empty((rows, K), np.float32)
    lse = np.empty((rows,), np.float64)
    _check(_load().ddo_topk(_p(logits), dtype, rows, V, V, K, _p(idx), _p(lp64), _p(lp32),
                            _p(lse)), "topk")
    shp = tuple(lead)
    return (idx.reshape(shp + (K,)), lp64.reshape(shp + (K,)), lp32.reshape(shp + (K,)),
            lse.reshape(shp))


def build_tree(logp32: np.ndarray, tok: np.ndarray, bonus: np.ndarray, prefix_len: np.ndarray,
               N: int) -> dict:
    """Best-first heap under node budget N (pages §4.2-§4.3, App. A).
    ``logp32``/``tok`` are [B][L][K].  Returns a dict of the tree arrays."""
    logp32 = np.ascontiguousarray(logp32, np.float32)
    tok = np.ascontiguousarray(tok, np.int32)
    B, L, K = logp32.shape
    R, W = N + 1, (N + 1 + 31) // 32
    out = {k: np.empty((B, R), np.int32) for k in
           ("parent", "depth", "rank", "token", "pos_id", "child_count")}
    out["score"] = np.empty((B, R), np.float32)
    out["anc_mask"] = np.empty((B, R, W), np.uint32)
    out["n_nodes"] = np.empty((B,), np.int32)
    _check(_load().ddo_build(_p(logp32), _p(tok), _p(np.ascontiguousarray(bonus, np.int32)),
                             _p(np.ascontiguousarray(prefix_len, np.int32)), B, L, K, N,
                             _p(out["parent"]), _p(out["depth"]), _p(out["rank"]),
                             _p(out["token"]), _p(out["pos_id"]), _p(out["score"]),
                             _p(out["child_count"]), _p(out["anc_mask"]), _p(out["n_nodes"])),
           "build")
    return out


def tree_attn(q, k_cache, v_cache, k_tree, v_tree, prefix_len, n_nodes, anc_mask, scale=None,
              units=None, rows=None):
    """fp64 tree attention of one layer (pages §4.1: ancestor-only mask over the
    tree, full prefix).  bf16-bit inputs: q [B][N+1][Hq][D], caches
    [B][Hkv][cap][D], tree K/V [B][N+1][Hkv][D].  ``units`` optionally limits
    the work to a list of (b, kv_head) pairs and ``rows`` to a node range
    (lo, hi); rows not computed are left NaN.
    Returns (out float64 [B][N+1][Hq][D], lse float64 [B][N+1][Hq])."""
    B, R, Hq, D = q.shape
    Hkv, cap = k_cache.shape[1], k_cache.shape[2]
    N = R - 1
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    out = np.full((B, R, Hq, D), np.nan, np.float64)
    lse = np.full((B, R, Hq), np.nan, np.float64)
    arrs = [np.ascontiguousarray(a) for a in (q, k_cache, v_cache, k_tree, v_tree)]
    pl = np.ascontiguousarray(prefix_len, np.int32)
    nn = np.ascontiguousarray(n_nodes, np.int32)
    am = np.ascontiguousarray(anc_mask, np.uint32)
    lib = _load()
    if units is None:
        units = [(b, g) for b in range(B) for g in range(Hkv)]
    lo, hi = rows if rows is not None else (0, R)
    for b, g in units:
        _check(lib.ddo_tree_attn_unit(b, g, lo, hi, _p(arrs[0]), _p(arrs[1]), _p(arrs[2]), cap,
                                      _p(arrs[3]), _p(arrs[4]), _p(pl), _p(nn), _p(am), B, N, Hq,
                                      Hkv, D, scale, _p(out), _p(lse)), "tree_attn")
    return out, lse


def tree_attn_tasks(q, k_cache, v_cache, k_tree, v_tree, prefix_len, n_nodes, anc_mask, tasks,
                    threads: int = 1, scale=None):
    """The same fp64 tree attention on a list of (b, kv_head, u_lo, u_hi) tasks
    -- node rows [u_lo, u_hi) of one (sequence, KV head) unit -- run on
    `threads` host threads at once (each call of the C routine releases the
    interpreter lock; tasks write disjoint rows of one output).  Rows not in a
    task stay NaN.  Returns (out, lse) as tree_attn does."""
    import concurrent.futures
    B, R, Hq, D = q.shape
    Hkv, cap = k_cache.shape[1], k_cache.shape[2]
    N = R - 1
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    out = np.full((B, R, Hq, D), np.nan, np.float64)
    lse = np.full((B, R, Hq), np.nan, np.float64)
    arrs = [np.ascontiguousarray(a) for a in (q, k_cache, v_cache, k_tree, v_tree)]
    pl = np.ascontiguousarray(prefix_len, np.int32)
    nn = np.ascontiguousarray(n_nodes, np.int32)
    am = np.ascontiguousarray(anc_mask, np.uint32)
    lib = _load()

    def run(t):
        b, g, lo, hi = t
        return lib.ddo_tree_attn_unit(b, g, lo, hi, _p(arrs[0]), _p(arrs[1]), _p(arrs[2]), cap,
                                      _p(arrs[3]), _p(arrs[4]), _p(pl), _p(nn), _p(am), B, N,
                                      Hq, Hkv, D, scale, _p(out), _p(lse))

    if threads <= 1:
        rcs = [run(t) for t in tasks]
    else:
        with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
            rcs = list(ex.map(run, tasks))
    for rc in rcs:
        _check(rc, "tree_attn")
    return out, lse


def philox4x64_10(counter, key) -> np.ndarray:
    """Philox4x64-10 block function (Salmon et al., SC'11)."""
    c = np.ascontiguousarray(counter, np.uint64)
    k = np.ascontiguousarray(key, np.uint64)
    o = np.empty(4, np.uint64)
    _load().ddo_philox4x64_10(_p(c), _p(k), _p(o))
    return o


def uniform(seed: int, step: int, seq: int, node: int) -> float:
    return _load().ddo_uniform(seed, step, seq, node)


def accept(logits, dtype: int, tree: dict, L: int, temperature: float = 0.0, seed: int = 0,
           step: int = 0) -> dict:
    """Target decoding rule per node, then the acceptance walk (pages §4.1).
    ``logits`` is [B][N+1][V]."""
    logits = np.ascontiguousarray(logits)
    B, R, V = logits.shape
    N = R - 1
    out = {"target_token": np.empty((B, R), np.int32), "accept_len": np.empty((B,), np.int32),
           "accepted_nodes": np.empty((B, L), np.int32),
           "out_tokens": np.empty((B, L + 1), np.int32), "next_bonus": np.empty((B,), np.int32),
           "margin": np.empty((B, R), np.float64)}
    _check(_load().ddo_accept(_p(logits), dtype, V, _p(np.ascontiguousarray(tree["parent"])),
                              _p(np.ascontiguousarray(tree["token"])),
                              _p(np.ascontiguousarray(tree["n_nodes"])), B, L, N, V,
                              float(temperature), seed, step, _p(out["target_token"]),
                              _p(out["accept_len"]), _p(out["accepted_nodes"]),
                              _p(out["out_tokens"]), _p(out["next_bonus"]), _p(out["margin"])),
           "accept")
    return out


def commit(k_cache, v_cache, k_tree, v_tree, accept_len, accepted_nodes, prefix_len):
    """Commit the accepted path -- the root (this round's bonus token) and the
    accepted nodes -- to the KV cache (pages §3, §4.1: verified tokens join the
    prefix).  Caches are [B][Hkv][cap][D] uint16 bf16 bits, tree K/V
    [B][N+1][Hkv][D]; returns (k_cache, v_cache, prefix_len) as new arrays."""
    kc = np.array(k_cache, dtype=np.uint16, order="C", copy=True)
    vc = np.array(v_cache, dtype=np.uint16, order="C", copy=True)
    kt = np.ascontiguousarray(k_tree, dtype=np.uint16)
    vt = np.ascontiguousarray(v_tree, dtype=np.uint16)
    B, Hkv, cap, D = kc.shape
    N = kt.shape[1] - 1
    L = np.asarray(accepted_nodes).shape[1]
    plen = np.array(prefix_len, dtype=np.int32, copy=True)
    _check(_load().ddo_commit(_p(kc), _p(vc), cap, _p(kt), _p(vt),
                              _p(np.ascontiguousarray(accept_len, dtype=np.int32)),
                              _p(np.ascontiguousarray(accepted_nodes, dtype=np.int32)), _p(plen),
                              B, L, N, Hkv, D), "commit")
    return kc, vc, plen
