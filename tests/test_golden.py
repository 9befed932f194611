"""The oracle reproduces its committed results for the tiny workload on this
machine (x86 or Arm): a regression guard for the oracle itself.  The stored
file is written by tests/golden/make_golden.py, which calls only the oracle."""
import json
import os

import numpy as np

from tests.golden.make_golden import tiny_round

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_round_matches_golden():
    with open(os.path.join(HERE, "golden", "tiny_round.json")) as f:
        gold = json.load(f)
    now = tiny_round()
    assert now["topk_idx"] == gold["topk_idx"]
    np.testing.assert_allclose(now["topk_logp"], gold["topk_logp"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(now["lse"], gold["lse"], rtol=0, atol=1e-12)
    assert now["tree"] == gold["tree"]
    assert now["score"] == gold["score"]
    assert now["anc_mask"] == gold["anc_mask"]
    assert now["accept"] == gold["accept"]
