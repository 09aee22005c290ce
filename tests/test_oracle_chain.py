"""Pins of the oracle's speculative-sampling acceptance (e-book page "Giai ma dau
co: doan truoc roi kiem mot luot", "Faster without changing the result" and "Why
a round always yields exactly k + 1 tokens")."""
import numpy as np
import pytest
import scipy.stats

import workloads as W
from oracle import oracle as O


def test_splitmix64_published_vectors(golden):
    rows = golden("splitmix64_vectors.txt")
    i = 0
    while i < len(rows):
        assert rows[i][0] == "seed"
        seed = int(rows[i][1])
        i += 1
        n = 1
        while i < len(rows) and rows[i][0] != "seed":
            assert O.splitmix64(seed, n) == int(rows[i][0])
            n += 1
            i += 1


def _toy(golden):
    rows = golden("toy_distribution.txt")
    p = np.array([float(r[1]) for r in rows], np.float32)
    q = np.array([float(r[2]) for r in rows], np.float32)
    return p, q


def _tile(p, q, B, gamma, seed):
    V = len(p)
    P = np.broadcast_to(p, (B, gamma + 1, V)).copy()
    Q = np.broadcast_to(q, (B, gamma, V)).copy()
    # drafts x ~ q, one per sequence and position
    rng = np.random.default_rng(seed)
    q64 = q.astype(np.float64)
    D = rng.choice(V, size=(B, gamma), p=q64 / q64.sum()).astype(np.int32)
    return P, Q, D


def test_monte_carlo_output_is_p_on_the_toy_pair(golden):
    # One draft position: the emitted first token must follow p exactly and the
    # acceptance rate must be sum min(p, q) = 0.90 (the page's 90.0%).
    p, q = _toy(golden)
    B = 200000
    P, Q, D = _tile(p, q, B, 1, seed=21)
    r = O.verify_chain(P, Q, D, seed=77, round_=0)
    first = r["out_tok"][:, 0]
    counts = np.bincount(first, minlength=4)
    p64 = p.astype(np.float64)
    chi = scipy.stats.chisquare(counts, B * p64 / p64.sum())
    assert chi.pvalue > 1e-4
    rate = r["n_acc"].mean()
    sd = np.sqrt(0.9 * 0.1 / B)
    assert abs(rate - 0.9) < 4 * sd
    # k + 1 tokens: exactly n_acc + 1 entries are set
    assert ((r["out_tok"] >= 0).sum(1) == r["n_acc"] + 1).all()


def test_monte_carlo_random_pairs_and_positions():
    rng = np.random.default_rng(22)
    V, B, gamma = 6, 120000, 3
    for trial in range(3):
        p = rng.dirichlet(np.ones(V)).astype(np.float32)
        q = rng.dirichlet(np.ones(V) * 0.7).astype(np.float32)
        P, Q, D = _tile(p, q, B, gamma, seed=30 + trial)
        r = O.verify_chain(P, Q, D, seed=1000 + trial, round_=trial)
        # every emitted token, at any position, is drawn from p
        alpha = np.minimum(p, q).astype(np.float64).sum()
        for pos in range(gamma + 1):
            sel = r["n_acc"] >= pos
            toks = r["out_tok"][sel, pos]
            counts = np.bincount(toks, minlength=V)
            assert scipy.stats.chisquare(counts, counts.sum() * p.astype(np.float64) / p.sum()).pvalue > 1e-4
        # P(n_acc >= i) = alpha^i for identical positions
        for i in range(1, gamma + 1):
            frac = (r["n_acc"] >= i).mean()
            e = alpha ** i
            assert abs(frac - e) < 4 * np.sqrt(e * (1 - e) / B) + 1e-12


def test_gamma_zero_yields_one_token_from_p():
    p = np.array([0.1, 0.6, 0.3], np.float32)
    B = 50000
    P = np.broadcast_to(p, (B, 1, 3)).copy()
    r = O.verify_chain(P, None, None, seed=5, round_=3)
    assert (r["n_acc"] == 0).all() and (r["out_tok"][:, 0] >= 0).all()
    counts = np.bincount(r["out_tok"][:, 0], minlength=3)
    p64 = p.astype(np.float64)
    assert scipy.stats.chisquare(counts, B * p64 / p64.sum()).pvalue > 1e-4


def test_identical_distributions_accept_everything_plus_bonus():
    x = W.chain_inputs(seed=6, B=16, gamma=5, V=40, sigma=0.0)
    P = x["p"].copy()
    P[:, :5] = x["q"]  # p = q on the draft positions
    r = O.verify_chain(P, x["q"], x["draft"], seed=9, round_=0)
    assert (r["n_acc"] == 5).all()
    assert np.array_equal(r["out_tok"][:, :5], x["draft"])
    assert (r["out_tok"][:, 5] >= 0).all()


def test_rejection_token_never_where_p_le_q():
    # the residual draw only lands where p > q
    x = W.chain_inputs(seed=7, B=256, gamma=4, V=30, sigma=1.0)
    r = O.verify_chain(x["p"], x["q"], x["draft"], seed=11, round_=1)
    for b in range(256):
        k = r["n_acc"][b]
        if k < 4:
            tok = r["out_tok"][b, k]
            assert x["p"][b, k, tok] > x["q"][b, k, tok]


def test_draws_are_reproducible_and_round_dependent():
    x = W.chain_inputs(seed=8, B=32, gamma=3, V=50, sigma=0.5)
    a = O.verify_chain(x["p"], x["q"], x["draft"], seed=1, round_=0)
    b = O.verify_chain(x["p"], x["q"], x["draft"], seed=1, round_=0)
    c = O.verify_chain(x["p"], x["q"], x["draft"], seed=1, round_=1)
    assert np.array_equal(a["out_tok"], b["out_tok"])
    assert not np.array_equal(a["out_tok"], c["out_tok"])
