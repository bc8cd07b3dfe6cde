"""Analytic helpers pinned to the numbers the pages print."""
import json
import os

import pytest

from oracle import analytic

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_e_table_matches_printed_values():
    tab = _load("e_table.json")
    for a, row in tab["rows"].items():
        for g, printed in zip(tab["gammas"], row):
            assert round(analytic.expected_tokens(float(a), g), 2) == pytest.approx(printed, abs=1e-9), (a, g)


def test_speedup_table_matches_printed_values():
    tab = _load("speedup_table_c005.json")
    for a, row in tab["rows"].items():
        for g, printed in zip(tab["gammas"], row):
            got = analytic.speedup(float(a), g, tab["c"])
            assert round(got, 2) == pytest.approx(printed, abs=1e-9), (a, g, got)


def test_worked_numbers():
    w = _load("worked_numbers.json")
    e = w["e_and_speedup_p2"]
    assert round(analytic.expected_tokens(e["alpha"], e["gamma"]), 1) == e["E_one_decimal"]
    assert round(analytic.speedup(e["alpha"], e["gamma"], e["c"]), 1) == e["speedup_one_decimal"]
    for case in w["p4_numbers"]["cases"]:
        assert round(analytic.expected_tokens(case["alpha"], case["k"]), case["decimals"]) == case["E"]
    cc = w["p4_numbers"]["cost_case"]
    assert cc["k"] * cc["c"] + 1 == pytest.approx(cc["denominator"])
    assert cc["E"] / cc["denominator"] == pytest.approx(cc["speedup"])
    d = w["p1_decay"]
    assert round(d["alpha"] ** d["run"], 2) == d["run_probability_two_decimals"]
    assert analytic.expected_tokens_upper_bound(d["alpha"]) == pytest.approx(d["upper_bound"])
    r = w["round_example"]
    assert r["accepted"] + 1 == r["emitted"]


def test_expected_tokens_limits():
    # a = 0: every first draft rejected, exactly one token; a -> 1: all gamma+1 tokens
    assert analytic.expected_tokens(0.0, 7) == 1.0
    assert analytic.expected_tokens(1.0, 7) == 8.0
    assert analytic.expected_tokens(0.999999, 7) == pytest.approx(8.0, rel=1e-5)
    # growing gamma approaches the ceiling 1/(1-a)
    assert analytic.expected_tokens(0.8, 200) == pytest.approx(analytic.expected_tokens_upper_bound(0.8))


def test_acceptance_rate_and_pmf():
    p = [0.1, 0.6, 0.3]
    q = [0.4, 0.3, 0.3]
    # sum_x min(p, q) = 0.1 + 0.3 + 0.3
    assert analytic.acceptance_rate(p, q) == pytest.approx(0.7)
    pmf = analytic.accepted_count_pmf([0.8] * 4)
    assert pmf.sum() == pytest.approx(1.0)
    mean_tokens = sum((k + 1) * pmf[k] for k in range(5))
    assert mean_tokens == pytest.approx(analytic.expected_tokens(0.8, 4))
