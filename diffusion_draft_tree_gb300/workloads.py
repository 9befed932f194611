"""Seeded synthetic inputs for one DDTree round.

This module only draws random numbers and lays them out.  It holds none of
the method's arithmetic (no softmax, no top-K, no tree, no attention, no
acceptance), so that both the CUDA path and the CPU oracle can be fed the
same bytes from it without sharing any of the computation under test.

Shapes follow the DDTree setting ("Accelerating Speculative Decoding with
Block Diffusion Draft Trees", §3-§4.1): per sequence one block of L draft
positions with a vocabulary-sized logit row each, a bonus token that becomes
the tree root, a KV prefix of P tokens, and target logits for every tree node.
The pages run on real datasets and Qwen3 models; those are replaced here by
seeded normal draws with the sizes listed in ``CONFIGS``.

Every array is produced from ``numpy.random.default_rng(SeedSequence([cfg, stream, ...]))``
so that any slice can be regenerated on its own.  bf16 tensors are fp32 draws
rounded to nearest-even once and handed around as their raw uint16 bits.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

# dtype codes shared by the C ABI and the oracle's own enum (values, not code)
BF16 = 0
FP32 = 1

# stream ids of the seeded generators (one independent stream per tensor)
S_DRAFT, S_SPIKE, S_PREFIX, S_Q, S_KCACHE, S_VCACHE, S_KVTREE, S_NOISE, S_BONUS = range(9)

BF16_NAN = np.uint16(0x7FC0)  # poison written where a kernel must not read


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    cfg_id: int
    B: int            # sequences
    L: int            # draft positions per block
    V: int            # vocabulary
    K: int            # top-K kept per position
    N: int            # node budget (drafted nodes, root excluded)
    P: tuple          # prefix length per sequence
    Hq: int
    Hkv: int
    D: int
    dtype: int        # BF16 or FP32 for the logit rows
    T: float          # target temperature (0 = greedy)
    draft_scale: float
    spike: Optional[float]
    noise_std: float

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def P_cap(self) -> int:
        return max(self.P) if len(self.P) else 0

    @property
    def esize(self) -> int:
        return 2 if self.dtype == BF16 else 4

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _rng(cfg_id: int, stream: int, *sub: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([cfg_id, stream, *sub]))


def _prefix_uniform(cfg_id: int, B: int, lo: int, hi: int) -> tuple:
    rng = _rng(cfg_id, S_PREFIX)
    return tuple(int(x) for x in rng.integers(lo, hi, size=B, endpoint=True))


# The five workloads: a tiny case, the single-stream 8B-class shape, the
# node-budget sweep, ragged batched serving at temperature 1 and the
# long-context 70B-class shape.
CONFIGS = {
    "tiny": Workload("tiny", 0, B=1, L=4, V=1000, K=4, N=16, P=(64,), Hq=2, Hkv=1, D=64,
                     dtype=FP32, T=0.0, draft_scale=2.0, spike=None, noise_std=0.5),
    "8b_single": Workload("8b_single", 1, B=1, L=16, V=151936, K=8, N=64, P=(2048,), Hq=32,
                          Hkv=8, D=128, dtype=BF16, T=0.0, draft_scale=3.0, spike=6.0,
                          noise_std=1.0),
    "ragged_serving": Workload("ragged_serving", 3, B=16, L=16, V=151936, K=8, N=128,
                               P=_prefix_uniform(3, 16, 1024, 32768), Hq=32, Hkv=8, D=128,
                               dtype=BF16, T=1.0, draft_scale=3.0, spike=6.0, noise_std=1.0),
    "long_context_70b": Workload("long_context_70b", 4, B=4, L=16, V=128256, K=8, N=256,
                                 P=(131072,) * 4, Hq=64, Hkv=8, D=128, dtype=BF16, T=0.0,
                                 draft_scale=3.0, spike=6.0, noise_std=1.5),
}
for _n in (32, 64, 128, 256, 512):
    CONFIGS[f"budget_sweep_n{_n}"] = Workload(
        f"budget_sweep_n{_n}", 2, B=1, L=16, V=151936, K=16, N=_n, P=(8192,), Hq=32, Hkv=8,
        D=128, dtype=BF16, T=0.0, draft_scale=3.0, spike=6.0, noise_std=1.0)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns the uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to fp32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _encode(x32: np.ndarray, dtype: int) -> np.ndarray:
    return bf16_bits(x32) if dtype == BF16 else np.ascontiguousarray(x32, dtype=np.float32)


def draft_logits(w: Workload) -> np.ndarray:
    """[B][L][V] draft logits: draft_scale * N(0,1), plus `spike` at one seeded token per row."""
    x = _rng(w.cfg_id, S_DRAFT).standard_normal((w.B, w.L, w.V), dtype=np.float32)
    x *= np.float32(w.draft_scale)
    if w.spike is not None:
        tok = _rng(w.cfg_id, S_SPIKE).integers(0, w.V, size=(w.B, w.L))
        bi, li = np.meshgrid(np.arange(w.B), np.arange(w.L), indexing="ij")
        x[bi, li, tok] += np.float32(w.spike)
    return _encode(x, w.dtype)


def bonus_tokens(w: Workload) -> np.ndarray:
    return _rng(w.cfg_id, S_BONUS).integers(0, w.V, size=w.B).astype(np.int32)


def prefix_lengths(w: Workload) -> np.ndarray:
    return np.asarray(w.P, dtype=np.int32)


def queries(w: Workload) -> np.ndarray:
    """[B][N+1][Hq][D] bf16 bits, N(0,1)."""
    x = _rng(w.cfg_id, S_Q).standard_normal((w.B, w.N + 1, w.Hq, w.D), dtype=np.float32)
    return bf16_bits(x)


def kv_cache_slice(w: Workload, which: int, b: int, g: int, cap: Optional[int] = None) -> np.ndarray:
    """[cap][D] bf16 bits of the K (which=0) or V (which=1) cache of sequence b, KV head g.

    Rows past the sequence's prefix length are poisoned with NaN: a kernel that
    lets them into its result fails parity instead of passing by luck.
    """
    cap = w.P_cap if cap is None else cap
    P = w.P[b]
    out = np.full((cap, w.D), BF16_NAN, dtype=np.uint16)
    x = _rng(w.cfg_id, S_KCACHE if which == 0 else S_VCACHE, b, g).standard_normal(
        (P, w.D), dtype=np.float32)
    out[:P] = bf16_bits(x)
    return out


def kv_cache(w: Workload, which: int, cap: Optional[int] = None) -> np.ndarray:
    """[B][Hkv][cap][D] bf16 bits (see kv_cache_slice)."""
    cap = w.P_cap if cap is None else cap
    out = np.empty((w.B, w.Hkv, cap, w.D), dtype=np.uint16)
    for b in range(w.B):
        for g in range(w.Hkv):
            out[b, g] = kv_cache_slice(w, which, b, g, cap)
    return out


def kv_tree(w: Workload, which: int) -> np.ndarray:
    """[B][N+1][Hkv][D] bf16 bits of the tree tokens' keys (0) or values (1), N(0,1)."""
    x = _rng(w.cfg_id, S_KVTREE, which).standard_normal((w.B, w.N + 1, w.Hkv, w.D),
                                                         dtype=np.float32)
    return bf16_bits(x)


def target_noise(w: Workload, b: int) -> np.ndarray:
    """[N+1][V] fp32 noise added to the draft rows to synthesise sequence b's target logits."""
    x = _rng(w.cfg_id, S_NOISE, b).standard_normal((w.N + 1, w.V), dtype=np.float32)
    x *= np.float32(w.noise_std)
    return x


def target_logits(w: Workload, draft: np.ndarray, depth: np.ndarray) -> np.ndarray:
    """[B][N+1][V] target logits, encoded like the draft rows.

    Node u of sequence b gets draft row min(depth[u], L-1) of that sequence plus
    seeded noise: the target's next-token row at a node at depth d looks like the
    drafter's marginal for position d+1.  Rows of padding nodes (depth < 0) are
    poisoned with NaN; no kernel may read them.
    """
    draft32 = bf16_to_f32(draft) if w.dtype == BF16 else np.asarray(draft, dtype=np.float32)
    out32 = np.full((w.B, w.N + 1, w.V), np.nan, dtype=np.float32)
    for b in range(w.B):
        d = np.asarray(depth[b])
        live = d >= 0
        rows = np.minimum(d[live], w.L - 1)
        out32[b, live] = draft32[b, rows] + target_noise(w, b)[live]
    return _encode(out32, w.dtype)


def philox_seed(w: Workload) -> int:
    return 0xDD7EE + w.cfg_id
