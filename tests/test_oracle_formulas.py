"""Pins of oracle.formulas against the numbers the pages print (tests/golden/formulas.json)."""
import json
import os

import numpy as np
import pytest

from oracle import formulas as F

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "formulas.json")))


def half_unit(v):
    s = repr(float(v))
    dec = len(s.split(".")[1]) if "." in s else 0
    return 0.5 * 10.0 ** (-dec) + 1e-12


def test_expected_tokens_printed_values():
    g = GOLD["expected_tokens"]
    for gamma, val in g["cases"]:
        assert abs(F.expected_tokens(g["alpha"], gamma) - val) <= half_unit(val)
    # ceiling 1/(1-alpha) as gamma grows
    assert abs(F.expected_tokens(g["alpha"], 400) - g["ceiling"]) < 1e-9
    gamma, one_in = g["one_in"]
    assert round(1.0 / g["alpha"] ** gamma) == one_in


def test_expected_tokens_equals_geometric_sum_and_bruteforce():
    # the series form printed on the vLLM page and a brute-force expectation
    for a in (0.1, 0.5, 0.75, 0.95):
        for gamma in range(0, 12):
            series = sum(a ** i for i in range(gamma + 1))
            assert abs(F.expected_tokens(a, gamma) - series) < 1e-12
            # enumerate the first-rejection index: P(n = i) = a^i (1 - a), n = gamma w.p. a^gamma
            e = sum((i + 1) * a ** i * (1 - a) for i in range(gamma)) + (gamma + 1) * a ** gamma
            assert abs(F.expected_tokens(a, gamma) - e) < 1e-12
    assert F.expected_tokens(1.0, 7) == 8.0


def test_theorem_3_11():
    g = GOLD["theorem_3_11"]
    v = F.arithmetic_increase(g["alpha"], g["gamma"], g["c_hat"])
    assert abs(v - g["value"]) <= half_unit(g["value"])
    # gamma = 0 means no speculation: no extra arithmetic
    assert abs(F.arithmetic_increase(0.3, 0, 0.0) - 1.0) < 1e-12


def test_speedup_table():
    g = GOLD["speedup_table_c010"]
    for a, row in g["rows"].items():
        for k, val in zip(g["k"], row):
            assert abs(F.speedup_model(float(a), k, g["c"]) - val) <= half_unit(val) + 1e-9, (a, k)


def test_break_even_table():
    g = GOLD["break_even"]
    for c, row in g["rows"].items():
        for k, val in zip(g["k"], row):
            assert abs(F.break_even_alpha(k, float(c)) - val) <= 0.005 + 1e-3, (c, k)
    for k, val in zip(g["k"], g["script_c010_3dp"]):
        assert abs(F.break_even_alpha(k, 0.10) - val) <= 0.0005 + 1e-6
    # a free drafter (c = 0) can't lose
    assert F.break_even_alpha(4, 0.0) == 0.0
    # at the break-even alpha the model gives speedup 1
    a = F.break_even_alpha(4, 0.2)
    assert abs(F.speedup_model(a, 4, 0.2) - 1.0) < 1e-9


def test_best_k():
    ks = GOLD["speedup_table_c010"]["k"]
    for a, kbest, val in GOLD["best_k_c010"]["rows"]:
        s = [F.speedup_model(a, k, 0.10) for k in ks]
        assert ks[int(np.argmax(s))] == kbest
        assert abs(max(s) - val) <= half_unit(val)


def test_verify_division():
    g = GOLD["verify_division"]
    t_dec = 1000.0 / g["decode_tok_s"]
    tok_s = 1000.0 * F.verify_cost_rate(g["p"], g["t_verify_ms"], g["t_draft_ms"])
    assert abs(tok_s - g["tok_s"]) <= g["tok_s_tol"]
    be = F.verify_break_even_ms(g["p"], t_dec, g["t_draft_ms"])
    assert abs(be - g["break_even_ms"]) <= 0.05
    assert abs(be / t_dec - g["break_even_ratio"]) <= 0.005
    # the page's corollary: if verify = 2 decode passes, speedup < (1 + p) / 2 <= 1
    for p in (0.0, 0.5, 1.0):
        assert F.verify_speedup(p, t_dec, 2 * t_dec, g["t_draft_ms"]) < (1 + p) / 2 <= 1.0


def test_verify_division_july():
    g = GOLD["verify_division_july"]
    for key in ("wrong", "right"):
        t = g[key]["t_token_ms"]
        tok_s = 1000.0 * F.verify_cost_rate(g["p"], 2 * t, g["t_draft_ms"])
        assert abs(tok_s - g[key]["tok_s"]) <= 0.05
        assert abs(round(tok_s, 1) / g["baseline_tok_s"] - g[key]["ratio"]) <= 1e-3
    t = g["right"]["t_token_ms"]
    assert abs(F.verify_speedup(1.0, t, 2 * t, g["t_draft_ms"]) - g["p1_ceiling"]) <= 0.0005


def test_vllm_metric_definitions():
    g = GOLD["vllm_log"]
    rounds = g["drafted"] // g["gamma"]
    # Rebuild a set of rounds whose per-position survival matches the printed vector
    # exactly (to the count), then check every printed metric follows from the definitions.
    surv = [round(x * rounds) for x in g["per_position"]]
    n_acc = np.zeros(rounds, dtype=np.int64)
    for i, s in enumerate(surv):
        n_acc[:s] = i + 1
    gam = np.full(rounds, g["gamma"])
    m = F.spec_metrics(n_acc, gam)
    # each printed entry is rounded to 3 decimals: +-0.0005 * rounds per position
    assert abs(m["accepted"] - g["accepted"]) <= 0.0005 * rounds * g["gamma"]
    assert abs(m["mean_acceptance_length"] - g["mean_acceptance_length"]) <= 0.005
    assert abs(100 * m["acceptance_rate"] - g["acceptance_rate_percent"]) <= 0.05
    for got, want in zip(m["per_position"], g["per_position"]):
        assert abs(got - want) <= 0.0005
    # the printed totals themselves: 1 + accepted / rounds = 2.61, accepted / drafted = 40.3 %
    assert abs(1 + g["accepted"] / rounds - g["mean_acceptance_length"]) <= 0.005
    assert abs(100 * g["accepted"] / g["drafted"] - g["acceptance_rate_percent"]) <= 0.05


def test_acceptance_probability_is_one_minus_tv():
    rng = np.random.default_rng(3)
    for _ in range(20):
        p = rng.dirichlet(np.ones(9))
        q = rng.dirichlet(np.ones(9))
        tv = 0.5 * np.abs(p - q).sum()
        assert abs(F.acceptance_probability(p, q) - (1 - tv)) < 1e-12
    p = np.array([0.5, 0.5, 0.0])
    assert F.acceptance_probability(p, p) == pytest.approx(1.0)
    assert F.acceptance_probability(np.array([1.0, 0.0]), np.array([0.0, 1.0])) == 0.0
