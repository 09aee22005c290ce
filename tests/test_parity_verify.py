"""GPU parity of medusa_verify_accept_tree against the oracle (Medusa Heads
glossary page, "Tree attention and acceptance"; e-book page "Giai ma dau co",
"Why a round always yields exactly k + 1 tokens")."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import oracle as O
from util import (TYPICAL_BAND, check_typical, race_draw, to_dev, to_np, tree_race_band,
                  typical_outcomes)

pytestmark = pytest.mark.gpu


def _tree(kind):
    if kind == "c1":
        return O.tree_layout(O.product_tree_paths((2, 3)), 2)
    if kind == "sparse64":
        return O.tree_layout(O.sparse_tree_paths(64, 5, 8, 0.6, 0.5), 5)
    if kind == "dense":
        return O.tree_layout(O.product_tree_paths((4, 4, 4, 4)), 4)
    if kind == "root":  # no candidates: the step yields the root's next token only
        return O.tree_layout(O.sparse_tree_paths(1, 4, 4, 0.6, 0.5), 4)
    raise KeyError(kind)


def _cands(t, B, V, seed, K=5, k=8):
    lists = W.random_topk_lists(seed, B, K, k, V)
    return O.build_tree(lists, W.root_tokens(seed, B, V), t["depth"], t["rank"])


def _gpu(M, logits, cand, t, mode="greedy", T=1.0, eps=0.09, delta=0.3):
    r = M.verify_accept_tree(to_dev(logits), to_dev(cand), to_dev(t["parent"]), to_dev(t["depth"]),
                             t["max_depth"], mode, T, eps, delta)
    torch.cuda.synchronize()
    return {k: to_np(v) for k, v in r.items()}


KEYS = ("accept_len", "best_node", "path_nodes", "next_tok")


@pytest.mark.parametrize("kind,B,V,K,k", [("c1", 1, 1000, 3, 3), ("sparse64", 1, 32000, 5, 8),
                                          ("sparse64", 8, 32000, 5, 8), ("dense", 2, 5003, 4, 4),
                                          ("root", 3, 1000, 3, 3)])
def test_greedy_planted_exact(medusa, kind, B, V, K, k):
    t = _tree(kind)
    for seed in range(3):
        cand = _cands(t, B, V, seed=50 + seed, K=K, k=k)
        logits = W.planted_logits(50 + seed, cand, t["parent"], V, 0.8)
        got = _gpu(medusa, logits, cand, t)
        ref = O.verify_tree(logits, cand, t["parent"], t["depth"], t["max_depth"])
        for key in KEYS:
            assert np.array_equal(got[key], ref[key]), key


def test_greedy_ties_take_lowest_token(medusa):
    t = _tree("c1")
    B, V = 6, 300
    cand = _cands(t, B, V, seed=60, K=3, k=3)
    rng = np.random.default_rng(60)
    logits = rng.integers(0, 3, size=(B, t["N"], V)).astype(np.float32)  # many equal maxima
    for b in range(B):  # make some candidates the lowest-index argmax
        for j in range(1, t["N"]):
            if rng.random() < 0.6:
                row = logits[b, t["parent"][j]]
                row[:] = np.minimum(row, 2)
                row[cand[b, j]] = 3
                row[: cand[b, j]] = np.minimum(row[: cand[b, j]], 2)
    got = _gpu(medusa, logits, cand, t)
    ref = O.verify_tree(logits, cand, t["parent"], t["depth"], t["max_depth"])
    for key in KEYS:
        assert np.array_equal(got[key], ref[key]), key


@pytest.mark.parametrize("kind,B,T", [("dense", 4, 1.0), ("sparse64", 4, 1.0), ("sparse64", 2, 0.7),
                                      ("dense", 4, 0.7)])
def test_typical_full_size(medusa, kind, B, T):
    # every decision is compared; a node within the measured float32 band of its
    # threshold may go either way (both resolutions are allowed, nothing else)
    t = _tree(kind)
    V = 32000
    cand = _cands(t, B, V, seed=70, K=5 if kind == "sparse64" else 4, k=8 if kind == "sparse64" else 4)
    logits = W.normal_logits(70, B, t["N"], V, 3.0)
    got = _gpu(medusa, logits, cand, t, "typical", T)
    ref = O.verify_tree(logits, cand, t["parent"], t["depth"], t["max_depth"], "typical", T)
    assert check_typical(got, ref, t["parent"], t["depth"]) <= 2


def _solve_logit(x_row, c, target, branch, T):
    """A logit l for token c such that, with row[c] = l, the row's float64
    decision quantity equals `target`: x_c - E_P[x] (threshold tied to the
    entropy: P_c e^H = e^(x_c - E_P[x])) or x_c - m - ln S = ln P_c (the eps
    branch), with x = row / T.  The sums over the other tokens are taken once;
    bisection on l (both quantities increase with it).  Returns l and f(l)."""
    rest = np.delete(x_row, c)
    Mr = rest.max()
    er = np.exp(rest - Mr)
    Sr, Ar = er.sum(), (er * rest).sum()

    def f(l):
        xc = l / T
        m = max(Mr, xc)
        a, e = np.exp(Mr - m), np.exp(xc - m)
        S = Sr * a + e
        if branch == "delta":
            return xc - (Ar * a + xc * e) / S
        return xc - m - np.log(S)
    lo, hi = -80.0, 80.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if f(mid) < target:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi), f


@pytest.mark.parametrize("branch,T", [("delta", 1.0), ("delta", 0.7), ("eps", 1.0), ("eps", 0.7)])
def test_typical_decision_error_is_within_band(medusa, branch, T):
    # Measures, through the C ABI, how far the GPU's float32 typical-acceptance
    # decision P(cand) > tau sits from the float64 one, on rows of the dense
    # workload's shape (vocab 32000, logits ~ N(0, 3)).  Each sequence is a root
    # and one candidate; the candidate's logit is set so that the oracle's
    # P(cand) e^H (branch "delta": tau = delta e^-H) or P(cand) (branch "eps":
    # tau = eps) equals t0 up to float32 rounding of the logit.  Sweeping delta
    # (or eps) in relative steps of 1e-6 around t0 finds, per sequence, where the
    # GPU's decision flips; its distance to the oracle's exact value is the
    # decision error.  The parity band TYPICAL_BAND must be at least twice the
    # largest error measured here.
    B, V, step, K = 512, 32000, 1e-6, 200
    t = O.tree_layout(np.array([[0]], np.int32), 1)
    assert t["N"] == 2 and list(t["parent"]) == [-1, 0]
    logits = W.normal_logits(77, B, 2, V, 3.0)
    rng = np.random.default_rng(77)
    t0 = 0.3 if branch == "delta" else 0.09
    target = np.log(t0)
    cand = np.zeros((B, 2), np.int32)
    g_exact = np.zeros(B)
    for b in range(B):
        row = logits[b, 0].astype(np.float64)
        c = int(rng.integers(0, V))
        while c == int(np.argmax(row)):
            c = int(rng.integers(0, V))
        l, f = _solve_logit(row / T, c, target, branch, T)
        logits[b, 0, c] = np.float32(l)
        g_exact[b] = np.exp(f(float(logits[b, 0, c])))  # P e^H or P of the float32 row
        cand[b, 1] = c
    dl, dc, dp, dd = to_dev(logits), to_dev(cand), to_dev(t["parent"]), to_dev(t["depth"])
    M = medusa
    out = dict(accept_len=torch.empty(B, dtype=torch.int32, device="cuda"),
               best_node=torch.empty(B, dtype=torch.int32, device="cuda"),
               path_nodes=torch.empty((B, 2), dtype=torch.int32, device="cuda"),
               next_tok=torch.empty(B, dtype=torch.int32, device="cuda"))
    ws = torch.empty(M.verify_accept_workspace(B, 2, V), dtype=torch.uint8, device="cuda")
    ks = np.arange(-K, K + 1)
    thr = t0 * (1.0 + ks * step)
    passed = np.zeros((len(ks), B), bool)
    for i, th in enumerate(thr):
        eps, delta = (float("inf"), float(th)) if branch == "delta" else (float(th), float("inf"))
        M.verify_accept_tree(dl, dc, dp, dd, 1, "typical", T, eps, delta, out=out, ws=ws)
        passed[i] = to_np(out["accept_len"]) == 1
    torch.cuda.synchronize()
    errs = []
    for b in range(B):
        col = passed[:, b]
        assert col[0] and not col[-1], f"sequence {b}: decision flips outside +-{K * step:g}"
        last = int(np.nonzero(col)[0].max())  # passes at thr[last], fails above it
        assert not col[last + 1:].any(), f"sequence {b}: decision not monotone in the threshold"
        lo, hi = thr[last] / g_exact[b] - 1.0, thr[last + 1] / g_exact[b] - 1.0
        errs.append(max(abs(lo), abs(hi)))
    worst = max(errs)
    print(f"\ntypical decision error ({branch}, T={T}): max {worst:.2e}, mean {np.mean(errs):.2e}")
    assert worst <= TYPICAL_BAND / 2, worst


def test_typical_accepts_where_candidates_are_likely(medusa):
    # plant each candidate as a dominant token of its parent's row (+30): typical
    # acceptance with eps 0.5 takes the planted chain, exactly as the oracle does
    t = _tree("sparse64")
    B, V = 4, 32000
    cand = _cands(t, B, V, seed=71)
    logits = W.planted_logits(71, cand, t["parent"], V, 0.8)
    for b in range(B):
        for u in range(t["N"]):
            logits[b, u, int(np.argmax(logits[b, u]))] += 30.0
    got = _gpu(medusa, logits, cand, t, "typical", 1.0, 0.5, 1.0)
    ref = O.verify_tree(logits, cand, t["parent"], t["depth"], t["max_depth"], "typical", 1.0, 0.5, 1.0)
    for key in KEYS:
        assert np.array_equal(got[key], ref[key]), key
    assert (got["accept_len"] > 0).any()


def test_typical_special_cases(medusa):
    t = _tree("sparse64")
    B, V = 3, 4000
    cand = _cands(t, B, V, seed=72)
    logits = W.normal_logits(72, B, t["N"], V, 3.0)
    got = _gpu(medusa, logits, cand, t, "typical", 1.0, 0.0, 0.3)   # tau = 0: all accepted
    assert (got["accept_len"] == t["depth"].max()).all()
    ref = O.verify_tree(logits, cand, t["parent"], t["depth"], t["max_depth"], "typical", 1.0, 0.0, 0.3)
    for key in KEYS:
        assert np.array_equal(got[key], ref[key]), key
    got = _gpu(medusa, logits, cand, t, "typical", 1.0, float("inf"), float("inf"))
    assert (got["accept_len"] == 0).all() and (got["best_node"] == 0).all()
    # k + 1 tokens: accept_len + 1 >= 1 always; path root..best
    assert (got["path_nodes"][:, 0] == 0).all()


@pytest.mark.parametrize("kind,B,V,T", [("c1", 2, 1000, 1.0), ("sparse64", 4, 32000, 1.0),
                                        ("sparse64", 3, 4099, 0.7), ("dense", 2, 5003, 1.0)])
def test_typical_sampled_next_token_matches_oracle(medusa, kind, B, V, T):
    # the accepted branch as typical acceptance (every decision compared, the
    # measured band allowing either resolution of a near-threshold node); the
    # next token is the exponential-race draw from the GPU's best row, equal to
    # the oracle's except where the two best race keys are within the float32
    # bound of the keys (tree_race_band, derived per row)
    t = _tree(kind)
    K, k = (3, 3) if kind == "c1" else ((4, 4) if kind == "dense" else (5, 8))
    cand = _cands(t, B, V, seed=95, K=K, k=k)
    logits = W.normal_logits(95, B, t["N"], V, 3.0)
    typ = O.verify_tree(logits, cand, t["parent"], t["depth"], t["max_depth"], "typical", T)
    ties = 0
    for rnd in range(3):
        r = medusa.verify_accept_tree_sample(to_dev(logits), to_dev(cand), to_dev(t["parent"]),
                                             to_dev(t["depth"]), t["max_depth"], 31, rnd, T)
        torch.cuda.synchronize()
        got = {kk: to_np(v) for kk, v in r.items()}
        ref = O.verify_tree_sample(logits, cand, t["parent"], t["depth"], t["max_depth"], 31, rnd, T)
        check_typical(got, typ, t["parent"], t["depth"], next_tok=False)
        for b in range(B):
            best = int(got["best_node"][b])
            row = logits[b, best]
            if best == ref["best_node"][b]:
                want, gap = int(ref["next_tok"][b]), ref["race_gap"][b]
            else:  # an ambiguous decision moved the best node: draw from the GPU's row
                x = row.astype(np.float64) / T
                want, gap = race_draw(np.exp(x - x.max()), O.row_key(31, 4, b, rnd, 0))
            if got["next_tok"][b] != want:
                assert gap <= tree_race_band(row, T), (b, got["next_tok"][b], want, gap)
                ties += 1
    assert ties <= 1
