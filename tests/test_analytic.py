"""Pins of the cost-model closed forms against the numbers the e-book page prints
("Giai ma dau co: doan truoc roi kiem mot luot": "Expected tokens per round",
"Reading the default numbers", "Guessing further is better? No", "When the peak
moves", the round table and "Round table, and why it draws no lots")."""
import numpy as np
import pytest

from oracle import analytic as A


def _num(s):
    return None if s == "-" else float(s)


def test_printed_cost_model_values(golden):
    for key, alpha, gamma, cd, cv, value in golden("cost_model.txt"):
        alpha, cd, cv, value = _num(alpha), _num(cd), _num(cv), float(value)
        g = None if gamma == "-" else int(gamma)
        if key == "expected_tokens":
            assert A.expected_tokens(alpha, g) == pytest.approx(value, abs=5e-4)
        elif key == "round_cost":
            assert A.round_cost(g, cd, cv) == pytest.approx(value, abs=5e-3)
        elif key == "speedup":
            assert A.speedup(alpha, g, cd, cv) == pytest.approx(value, abs=5e-3)
        elif key == "target_passes_per_token":
            assert 1.0 / A.speedup(alpha, g, cd, cv) == pytest.approx(value, abs=5e-4)
        elif key == "fraction_of_ceiling_pct":
            # "of the 5 tokens a round can give": E / (gamma + 1)
            assert 100 * A.expected_tokens(alpha, g) / (g + 1) == pytest.approx(value, abs=0.05)
        elif key == "best_gamma":
            assert A.best_gamma(alpha, cd, cv)[0] == int(value)
        elif key == "best_speedup":
            assert A.best_gamma(alpha, cd, cv)[1] == pytest.approx(value, abs=5e-3)
        elif key == "ceiling":
            assert A.expected_tokens(alpha, 2000) == pytest.approx(value, abs=1e-9)
        else:
            raise AssertionError(key)


@pytest.mark.parametrize("alpha", [0.0, 0.1, 0.37, 0.8, 0.95, 0.999])
@pytest.mark.parametrize("gamma", [0, 1, 4, 7, 32])
def test_geometric_closed_form(alpha, gamma):
    # the page states E both as the sum and as (1 - alpha^(gamma+1)) / (1 - alpha)
    closed = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert A.expected_tokens(alpha, gamma) == pytest.approx(closed, rel=1e-12)


def test_special_cases():
    # the three rows of the page's table of landmarks
    for g in range(0, 33):
        assert A.expected_tokens(1.0, g) == g + 1
        assert A.expected_tokens(0.0, g) == 1
    for a in (0.0, 0.3, 0.8, 1.0):
        assert A.expected_tokens(a, 0) == 1


def test_expected_tokens_monte_carlo():
    # independent positions, each accepted with probability alpha: the accepted
    # prefix length + 1, averaged, converges to E
    rng = np.random.default_rng(5)
    alpha, gamma, n = 0.8, 4, 400000
    acc = rng.random((n, gamma)) < alpha
    prefix = np.where(acc.all(1), gamma, np.argmin(acc, axis=1))
    tokens = prefix + 1
    e = A.expected_tokens(alpha, gamma)
    sd = tokens.std() / np.sqrt(n)
    assert abs(tokens.mean() - e) < 4 * sd


def test_round_table(golden):
    rows = golden("round_table.txt")
    # Table rows are rounds of accepted counts 4, 2, 0, 3, 1, 4 at gamma 4.
    flags = "".join("1" * int(r[2]) + ("0" if int(r[3]) else "") for r in rows)
    sim = A.simulate_acceptance_string(flags, 4)
    assert len(sim) == len(rows)
    for s, r in zip(sim, rows):
        n, prop, acc, rej, tok, cum, dp, tp, cost = r
        assert s["proposed"] == int(prop) and s["accepted"] == int(acc)
        assert (s["rejected_at"] or 0) == int(rej)
        assert s["tokens"] == int(tok) and s["cum_tokens"] == int(cum)
        assert s["draft_passes"] == int(dp) and s["target_passes"] == int(tp)
        assert s["cum_cost"] == pytest.approx(float(cost), abs=5e-3)


def test_acceptance_string(golden):
    g = {r[0]: r[1:] for r in golden("acceptance_string.txt")}
    flags, gamma = g["string"][0], int(g["gamma"][0])
    sim = A.simulate_acceptance_string(flags, gamma)
    assert [s["accepted"] for s in sim] == [int(x) for x in g["accepted_per_round"]]
    tokens = sim[-1]["cum_tokens"]
    assert tokens == int(g["tokens"][0])
    assert len(sim) == int(g["target_passes"][0])
    assert tokens / len(sim) == pytest.approx(float(g["tokens_per_round"][0]), abs=5e-4)
    assert sim[-1]["cum_cost"] == pytest.approx(float(g["cost"][0]), abs=5e-3)
    assert tokens / sim[-1]["cum_cost"] == pytest.approx(float(g["speedup"][0]), abs=5e-3)
    assert flags.count("1") == int(g["accepted_flags"][0]) and len(flags) == int(g["flags"][0])
    assert 100 * flags.count("1") / len(flags) == pytest.approx(float(g["rate_pct"][0]), abs=0.05)
    # every round yields k + 1 >= 1 tokens
    assert all(s["tokens"] == s["accepted"] + 1 >= 1 for s in sim)


def test_toy_distribution(golden):
    rows = golden("toy_distribution.txt")
    p = np.array([float(r[1]) for r in rows])
    q = np.array([float(r[2]) for r in rows])
    out, acc, resid = A.sampling_output_distribution(p, q)
    assert np.minimum(p, q).sum() == pytest.approx(0.90, abs=1e-12)
    assert acc == pytest.approx(0.90, abs=1e-12)
    assert resid == pytest.approx(0.10, abs=1e-12)
    for r, o in zip(rows, out):
        assert float(r[3]) == pytest.approx(min(float(r[1]), float(r[2])), abs=1e-12)
        assert float(r[4]) == pytest.approx(max(0.0, float(r[1]) - float(r[2])), abs=1e-12)
        assert float(r[6]) == pytest.approx(o, abs=1e-12)
    np.testing.assert_allclose(out, p, atol=1e-12)


def _dirichlet_set():
    rng = np.random.default_rng(729)
    pts = [np.eye(3)[i] for i in range(3)] + [np.full(3, 1 / 3), np.array([0.5, 0.5, 0.0])]
    while len(pts) < 27:
        pts.append(rng.dirichlet(np.ones(3)))
    return pts


def test_729_pairs_output_equals_p():
    # 27 x 27 = 729 distribution pairs; output column = p row by row, and the
    # acceptance probability = sum min(p, q) = 1 - total variation distance
    pts = _dirichlet_set()
    n = 0
    for p in pts:
        for q in pts:
            out, acc, resid = A.sampling_output_distribution(p, q)
            np.testing.assert_allclose(out, p, atol=1e-12)
            tv = 0.5 * np.abs(p - q).sum()
            assert acc == pytest.approx(1 - tv, abs=1e-12)
            assert resid == pytest.approx(1 - acc, abs=1e-12)
            n += 1
    assert n == 729
