"""Mutation check of the oracle's pins (CPU only).

Each case plants one plausible mistake in a copy of the oracle's C source (a
dropped term, a wrong index, a transposed operand, a flipped tie-break),
compiles the copy with the oracle's own compiler flags, swaps it in for the
real library and runs the pins that guard that part of the method.  At least
one of them must fail: a pin set that a plausible mistake slips through does
not pin the oracle.  The real oracle is untouched; the mutants live in a
temporary directory.
"""
import ctypes
import os

import numpy as np
import pytest

import oracle
from tests import test_oracle_pins as pins


def _mutant(tmp_path, old: str, new: str):
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"mutation site not unique: {old!r}"
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    so = os.path.join(tmp_path, "libmutant.so")
    oracle._compile(path, so)
    return oracle._bind(ctypes.CDLL(so))


def _margin_pins():
    for V, T, flat in [(40, 1.0, False), (1000, 1.0, False), (1000, 0.5, True)]:
        pins.test_sampling_margin_is_distance_to_nearest_cdf_edge(V, T, flat)


def _heap_pins():
    for args in [(2, 3, 5, False), (3, 3, 12, False), (2, 5, 20, True), (4, 4, 16, False),
                 (3, 4, 40, True)]:
        pins.test_heap_equals_brute_force_order(*args)
    pins.test_heap_structure_invariants()
    for N in (3, 5):
        pins.test_heap_tree_is_optimal_among_all_valid_trees(N)


def _attn_pins():
    pins.test_tree_attention_is_sdpa_over_each_root_path(1, 16, 2, 1, 64, (64,))
    pins.test_tree_attention_is_sdpa_over_each_root_path(2, 20, 8, 2, 32, (5, 0))
    pins.test_tree_attention_chain_is_causal_attention()
    pins.test_tree_attention_root_only_is_decode_attention()


def _topk_pins():
    from diffusion_draft_tree_gb300 import workloads as wl
    for dtype in (wl.FP32, wl.BF16):
        for V, K in [(37, 1), (1000, 4), (64, 64)]:
            pins.test_topk_against_sort_and_logsumexp(dtype, V, K)
    pins.test_topk_signed_zero_ties_by_index()


def _sampling_pins():
    pins.test_sampling_rule_is_inverse_cdf()
    _margin_pins()


def _walk_pins():
    pins.test_greedy_rule_is_argmax_first_index()
    pins.test_chain_walk_is_vanilla_dflash_acceptance()
    pins.test_planted_agreement_follows_rank0_chain()


def _philox_pins():
    for ctr, key in [([0, 0, 0, 0], [0, 0]), ([3, 9, 0, 0], [0xDD7EE, 0])]:
        pins.test_philox_matches_numpy(ctr, key)
    pins.test_uniform_is_top_24_bits()


MUTANTS = {
    # T > 0 band: the margin that admits GPU/oracle disagreements
    "margin_drops_lower_edge": ("double d0 = target - prev, d1 = c - target;",
                                "double d0 = target, d1 = c - target;", _margin_pins),
    "margin_takes_far_edge": ("(d0 < d1 ? d0 : d1) / z", "(d0 < d1 ? d1 : d0) / z",
                              _margin_pins),
    "margin_not_normalised": ("(d0 < d1 ? d0 : d1) / z", "(d0 < d1 ? d0 : d1)", _margin_pins),
    "cdf_prev_not_advanced": ("prev = c;\n", "", _sampling_pins),
    # step 1
    "lse_without_max": ("const double l = m + log(s);", "const double l = log(s);", _topk_pins),
    "topk_higher_index_wins_ties": ("if (best_i < 0 || x > best_x)",
                                    "if (best_i < 0 || x >= best_x)", _topk_pins),
    # step 2
    "child_reads_parent_depth_row": ("c.score + lp[c.depth * K + 0]",
                                     "c.score + lp[(c.depth - 1) * K + 0]", _heap_pins),
    "sibling_from_node_score": ("sc[c.parent] + lp[(c.depth - 1) * K + c.rank + 1]",
                                "c.score + lp[(c.depth - 1) * K + c.rank + 1]", _heap_pins),
    "no_parent_tie_break": ("if (a->parent != b->parent) return a->parent < b->parent;", "",
                            _heap_pins),
    "mask_without_self": ("for (int a = u; a >= 0; a = par[a])",
                          "for (int a = par[u]; a >= 0; a = par[a])", _heap_pins),
    # step 3
    "gqa_modulo_mapping": ("for (int h = g * G; h < (g + 1) * G; ++h)",
                           "for (int h = g; h < Hq; h += Hkv)", _attn_pins),
    "score_without_scale": ("s[j] = dot * scale;", "s[j] = dot;", _attn_pins),
    # step 4
    "argmax_last_index": ("if (x > m) { m = x; am = v; }", "if (x >= m) { m = x; am = v; }",
                          _walk_pins),
    "bonus_from_root": ("ot[len] = t[cur];", "ot[len] = t[0];", _walk_pins),
    "philox_words_swapped": ("out[0] = x0; out[1] = x1;", "out[0] = x1; out[1] = x0;",
                             _philox_pins),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, monkeypatch, name):
    old, new, run_pins = MUTANTS[name]
    lib = _mutant(str(tmp_path), old, new)
    monkeypatch.setattr(oracle, "_lib", lib)
    with pytest.raises((AssertionError, ValueError)):
        run_pins()


def test_unmutated_oracle_passes_the_same_pins():
    """The pin groups above pass on the real oracle (so a failure under a
    mutant is the mutant's doing)."""
    for run in (_margin_pins, _heap_pins, _attn_pins, _topk_pins, _sampling_pins, _walk_pins,
                _philox_pins):
        run()
    assert np.isfinite(oracle.uniform(1, 2, 3, 4))
