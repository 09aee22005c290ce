"""Closed forms of the speculative-decoding cost model -- TEST INFRASTRUCTURE ONLY.

Source: the speculative-decoding e-book page "Giai ma dau co: doan truoc roi kiem
mot luot", sections "Expected tokens per round", "Reading the default numbers",
"Guessing further is better? No", "When the peak moves", "Faster without
changing the result" and the round table ("Round table, and why it draws no
lots").  Pure Python, float64, written from the definitions.
"""
from __future__ import annotations

import numpy as np


def expected_tokens(alpha: float, gamma: int) -> float:
    """E = sum_{i=0..gamma} alpha^i: the accepted prefix reaches length >= i with
    probability alpha^i when positions are independent ("Expected tokens per
    round").  Written as the sum itself, so alpha = 1 gives gamma + 1 with no
    0/0."""
    return float(sum(alpha ** i for i in range(gamma + 1)))


def round_cost(gamma: int, c_draft: float, c_verify: float) -> float:
    """Cost of one round in target-pass units: gamma draft passes + one check."""
    return gamma * c_draft + c_verify


def speedup(alpha: float, gamma: int, c_draft: float, c_verify: float = 1.0) -> float:
    return expected_tokens(alpha, gamma) / round_cost(gamma, c_draft, c_verify)


def best_gamma(alpha: float, c_draft: float, c_verify: float = 1.0, gamma_max: int = 32):
    """The gamma in [0, gamma_max] with the largest speedup (smallest gamma on ties)."""
    best, val = 0, -1.0
    for g in range(gamma_max + 1):
        s = speedup(alpha, g, c_draft, c_verify)
        if s > val:
            best, val = g, s
    return best, val


def simulate_acceptance_string(flags: str, gamma: int, c_draft: float = 0.10,
                               c_verify: float = 1.00):
    """Deterministic rounds from an acceptance string (1 = accepted, 0 = rejected).

    Each round reads flags until a 0 or until gamma flags have been read.  A round
    yields its accepted drafts plus one token: the correction token after a
    rejection, or the bonus token when all gamma were accepted.
    """
    rounds = []
    pos = 0
    tot_tok = 0
    while pos < len(flags):
        acc = 0
        rej_at = None
        while acc < gamma and pos < len(flags):
            f = flags[pos]
            pos += 1
            if f == "1":
                acc += 1
            else:
                rej_at = acc + 1
                break
        tokens = acc + 1
        tot_tok += tokens
        n = len(rounds) + 1
        rounds.append(dict(proposed=gamma, accepted=acc, rejected_at=rej_at, tokens=tokens,
                           cum_tokens=tot_tok, draft_passes=gamma * n, target_passes=n,
                           cum_cost=n * round_cost(gamma, c_draft, c_verify)))
    return rounds


def sampling_output_distribution(p, q):
    """Exact distribution of the token that the speculative-sampling rule emits.

    Enumerates the rule's branches ("Faster without changing the result"): a
    draft y is drawn with probability q(y) and kept with probability
    min(1, p(y)/q(y)); otherwise a token is drawn from max(0, p - q) normalised.
    Returns (output distribution, acceptance probability, rejection mass of the
    residual)."""
    p = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    out = np.zeros_like(p)
    p_reject = 0.0
    resid = np.maximum(0.0, p - q)
    rs = resid.sum()
    for y in range(len(q)):
        if q[y] <= 0:
            continue
        a = min(1.0, p[y] / q[y])
        out[y] += q[y] * a
        p_reject += q[y] * (1.0 - a)
    if p_reject > 0:
        out += p_reject * resid / rs
    return out, 1.0 - p_reject, rs
