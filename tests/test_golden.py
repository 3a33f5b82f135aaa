"""Regression pin: the oracle and the input recipe still give the frozen PR1
values written by tests/golden/make_golden.py."""
import os

import numpy as np

import oracle
from attention_forward_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pr1_oracle.txt")


def test_pr1_oracle_unchanged():
    lines = [ln for ln in open(GOLDEN).read().splitlines() if not ln.startswith("#")]
    lse_ref = np.array(lines[0].split(), float)
    w = inputs.PR1
    q, k, v = (t.float().numpy() for t in w.make())
    o, lse = oracle.attention(q, k, v, w.scale, w.causal)
    assert np.abs(lse.reshape(-1) - lse_ref).max() < 1e-14
    for r, ln in zip((0, 1, 63, 64, 127), lines[1:]):
        assert np.abs(o[0, 0, r] - np.array(ln.split(), float)).max() < 1e-14
