"""Acceptance metrics against the worked figures printed on the pages."""

import json
import os

import numpy as np
import pytest

from mtp_speculative_decoding_draft_gb300.metrics import acceptance_metrics, mean_length_from_positions

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "acceptance_worked_examples.json")))


def _lengths_from_positions(pos, n):
    """A batch of n sequence-steps whose per-depth acceptance fractions are pos."""
    counts = [int(round(p * n)) for p in pos]          # #{a >= j}
    a_hist = []
    prev = n
    for j, c in enumerate(counts):
        a_hist.append(prev - c)                        # exactly j accepted
        prev = c
    a_hist.append(prev)                                # all k accepted
    return np.repeat(np.arange(len(pos) + 1) + 1, a_hist)


def test_skyrl_worked_example():
    g = GOLD["skyrl_depth3"]
    L = _lengths_from_positions(g["pos"], 1000)
    m = acceptance_metrics(L, g["k"])
    for j, p in enumerate(g["pos"], start=1):
        assert m["draft_acceptance_rate_pos_%d" % j] == pytest.approx(p, abs=1e-12)
    tol = g["printed_precision"]
    assert abs(m["draft_acceptance_rate"] - g["draft_acceptance_rate"]) <= tol["draft_acceptance_rate"]
    assert abs(m["draft_mean_acceptance_length"] - g["draft_mean_acceptance_length"]) <= tol["draft_mean_acceptance_length"]
    assert m["draft_num_draft_tokens"] == 3000
    assert m["draft_num_accepted_tokens"] == 886 + 770 + 663


def test_fastmtp_table_implied_lengths():
    g = GOLD["fastmtp_table"]
    assert mean_length_from_positions(g["base_pos"]) == pytest.approx(g["implied_mean_length_base"], abs=1e-9)
    assert mean_length_from_positions(g["finetuned_pos"]) == pytest.approx(g["implied_mean_length_finetuned"], abs=1e-9)


def test_bounds_and_extremes():
    k = 4
    m = acceptance_metrics([1] * 10, k)           # nothing accepted: no gain
    assert m["draft_mean_acceptance_length"] == 1.0 and m["draft_acceptance_rate"] == 0.0
    m = acceptance_metrics([k + 1] * 10, k)       # everything accepted: the k+1 ceiling
    assert m["draft_mean_acceptance_length"] == k + 1 and m["draft_acceptance_rate"] == 1.0
    with pytest.raises(ValueError):
        acceptance_metrics([0, 1], k)
    with pytest.raises(ValueError):
        acceptance_metrics([k + 2], k)


def test_mean_length_identity_random():
    rng = np.random.default_rng(3)
    for k in (1, 3, 5):
        L = rng.integers(1, k + 2, size=257)
        m = acceptance_metrics(L, k)
        pos = [m["draft_acceptance_rate_pos_%d" % j] for j in range(1, k + 1)]
        assert m["draft_mean_acceptance_length"] == pytest.approx(mean_length_from_positions(pos), abs=1e-12)
        assert m["draft_acceptance_rate"] == pytest.approx(np.mean(pos), abs=1e-12)
