"""Pins of the oracle's tree acceptance (Medusa Heads glossary page, "Tree
attention and acceptance"; e-book page "Giai ma dau co", "Why a round always
yields exactly k + 1 tokens" and "Expected tokens per round")."""
import numpy as np
import pytest
import scipy.special
import scipy.stats

import workloads as W
from oracle import analytic as A
from oracle import oracle as O


def _tree(kind):
    if kind == "c1":
        return O.tree_layout(O.product_tree_paths((2, 3)), 2)
    if kind == "sparse64":
        return O.tree_layout(O.sparse_tree_paths(64, 5, 8, 0.6, 0.5), 5)
    if kind == "small":
        return O.tree_layout(O.product_tree_paths((3, 2, 2)), 3)
    raise KeyError(kind)


def _cands(t, B, V, seed, K=None, k=8):
    K = K or t["max_depth"]
    lists = W.random_topk_lists(seed, B, K, k, V)
    return O.build_tree(lists, W.root_tokens(seed, B, V), t["depth"], t["rank"])


def test_greedy_matches_brute_force_over_paths():
    # Walk every root-to-leaf path; its accepted prefix is where a candidate
    # first differs from the argmax of its parent's row.  The best node is the
    # deepest accepted one (lowest index on ties).
    t = _tree("small")
    B, V = 40, 12
    rng = np.random.default_rng(10)
    cand = _cands(t, B, V, seed=10, K=3, k=3)
    logits = rng.integers(0, 4, size=(B, t["N"], V)).astype(np.float32)  # ties in argmax
    r = O.verify_tree(logits, cand, t["parent"], t["depth"], t["max_depth"])
    for b in range(B):
        amax = [int(np.flatnonzero(logits[b, u] == logits[b, u].max())[0]) for u in range(t["N"])]
        best_depth, best = 0, 0
        accepted = {0}
        for row in t["retrieve"]:
            nodes = [x for x in row if x >= 0]
            for a, c in zip(nodes, nodes[1:]):
                if cand[b, c] != amax[a]:
                    break
                accepted.add(c)
        for n in sorted(accepted):
            if t["depth"][n] > best_depth:
                best_depth, best = t["depth"][n], n
        assert r["accept_len"][b] == best_depth
        assert r["best_node"][b] == best
        assert r["next_tok"][b] == amax[best]
        path = [x for x in r["path_nodes"][b] if x >= 0]
        assert path[0] == 0 and path[-1] == best and len(path) == best_depth + 1
        assert set(np.flatnonzero(r["accepted"][b]).tolist()) == accepted
        # k + 1 tokens: accept_len accepted candidates plus next_tok, never fewer than 1
        assert r["accept_len"][b] + 1 >= 1


@pytest.mark.parametrize("kind,chain_depth,expect", [("c1", 2, 2.44), ("sparse64", 4, 3.3616)])
def test_planted_alpha_gives_geometric_expected_tokens(kind, chain_depth, expect):
    # Planting makes each rank-0 child the argmax with probability alpha, so the
    # accepted path is the rank-0 chain cut geometrically and the mean tokens per
    # step is sum_{i<=depth} alpha^i: 3.362 at depth 4, alpha 0.8, the page's
    # default E ("Reading the default numbers").
    t = _tree(kind)
    assert A.expected_tokens(0.8, chain_depth) == pytest.approx(expect, abs=1e-4)
    V, B = 64, 64
    toks = []
    for seed in range(12):
        cand = _cands(t, B, V, seed=100 + seed)
        logits = W.planted_logits(100 + seed, cand, t["parent"], V, 0.8)
        r = O.verify_tree(logits, cand, t["parent"], t["depth"], t["max_depth"])
        toks.append(r["accept_len"] + 1)
        # the accepted path is the rank-0 chain
        for b in range(B):
            for n in r["path_nodes"][b]:
                if n > 0:
                    assert t["rank"][n] == 0
    toks = np.concatenate(toks)
    sd = toks.std() / np.sqrt(len(toks))
    assert abs(toks.mean() - expect) < 4 * sd


def test_typical_threshold_matches_library_entropy():
    t = _tree("small")
    B, V = 6, 50
    rng = np.random.default_rng(11)
    cand = _cands(t, B, V, seed=11, K=3, k=3)
    logits = (rng.standard_normal((B, t["N"], V)) * 3).astype(np.float32)
    T, eps, delta = 0.7, 0.09, 0.3
    r = O.verify_tree(logits, cand, t["parent"], t["depth"], t["max_depth"], "typical", T, eps, delta)
    for b in range(B):
        for u in range(t["N"]):
            P = scipy.special.softmax(logits[b, u].astype(np.float64) / T)
            H = scipy.stats.entropy(P)
            assert r["tau"][b, u] == pytest.approx(min(eps, delta * np.exp(-H)), rel=1e-12)
        for j in range(1, t["N"]):
            P = scipy.special.softmax(logits[b, t["parent"][j]].astype(np.float64) / T)
            assert r["pcand"][b, j] == pytest.approx(P[cand[b, j]], rel=1e-12)


def test_typical_special_cases():
    t = _tree("sparse64")
    B, V = 4, 300
    cand = _cands(t, B, V, seed=12)
    logits = W.normal_logits(12, B, t["N"], V, 3.0)
    # eps = 0 -> tau = 0 -> every candidate passes -> the deepest node is taken
    r = O.verify_tree(logits, cand, t["parent"], t["depth"], t["max_depth"], "typical", 1.0, 0.0, 0.3)
    assert (r["accept_len"] == t["depth"].max()).all()
    assert (r["accepted"] == 1).all()
    # eps = delta = inf -> tau = inf -> nothing passes
    r = O.verify_tree(logits, cand, t["parent"], t["depth"], t["max_depth"], "typical", 1.0,
                      np.inf, np.inf)
    assert (r["accept_len"] == 0).all() and (r["best_node"] == 0).all()


def test_typical_with_huge_threshold_scale_equals_greedy_on_planted_rows():
    # A planted row has one dominant token (logit max + 30): P ~ 1 there, so a
    # threshold of eps = 0.5 accepts exactly the planted argmax, like greedy.
    t = _tree("small")
    B, V = 16, 40
    cand = _cands(t, B, V, seed=13, K=3, k=3)
    logits = W.planted_logits(13, cand, t["parent"], V, 0.7)
    for b in range(B):
        for u in range(t["N"]):
            a = int(np.argmax(logits[b, u]))
            logits[b, u, a] += 30.0
    g = O.verify_tree(logits, cand, t["parent"], t["depth"], t["max_depth"])
    ty = O.verify_tree(logits, cand, t["parent"], t["depth"], t["max_depth"], "typical", 1.0, 0.5, 1.0)
    for k in ("accept_len", "best_node", "path_nodes", "next_tok"):
        assert np.array_equal(g[k], ty[k])


# ---------------------------------------------------------------------------
# typical acceptance with a sampled next token (Medusa Heads glossary page,
# "Tree attention and acceptance": in sampling, Medusa uses typical acceptance)
# ---------------------------------------------------------------------------
def test_sampled_next_token_follows_the_softmax_of_the_best_row():
    # root-only tree: the best node is the root, so the token after it is a
    # draw from softmax(row0 / T); many rounds of the counter-based generator
    # must reproduce that distribution (chi-square), for two temperatures
    t = O.tree_layout(np.zeros((0, 1), np.int32), 1)
    V = 7
    x = np.array([[[1.5, -0.3, 0.2, 2.0, -1.0, 0.7, 0.0]]], np.float32)
    cand = np.zeros((1, t["N"]), np.int32)
    R = 12000
    for T in (1.0, 0.6):
        draws = np.array([O.verify_tree_sample(x, cand, t["parent"], t["depth"], t["max_depth"], 9, r, T)
                          ["next_tok"][0] for r in range(R)])
        expect = scipy.special.softmax(x[0, 0].astype(np.float64) / T) * R
        counts = np.bincount(draws, minlength=V)
        assert scipy.stats.chisquare(counts, expect).pvalue > 1e-3


def test_sampled_next_token_keeps_the_typical_branch_and_cools_to_argmax():
    t = _tree("sparse64")
    B, V = 3, 500
    cand = _cands(t, B, V, seed=90, K=5)
    logits = W.normal_logits(90, B, t["N"], V, 3.0)
    typ = O.verify_tree(logits, cand, t["parent"], t["depth"], t["max_depth"], "typical", 1.0)
    smp = O.verify_tree_sample(logits, cand, t["parent"], t["depth"], t["max_depth"], 5, 0, 1.0)
    for key in ("accept_len", "best_node", "path_nodes"):
        assert np.array_equal(smp[key], typ[key])
    # a vanishing temperature leaves one positive weight: the row's argmax
    cold = O.verify_tree_sample(logits, cand, t["parent"], t["depth"], t["max_depth"], 5, 0, 1e-4)
    best_rows = logits[np.arange(B), cold["best_node"]]
    assert np.array_equal(cold["next_tok"], best_rows.argmax(-1))
    # the same (seed, round) draws the same token; other rounds draw others
    again = O.verify_tree_sample(logits, cand, t["parent"], t["depth"], t["max_depth"], 5, 0, 1.0)
    assert np.array_equal(again["next_tok"], smp["next_tok"])
    many = {int(O.verify_tree_sample(logits, cand, t["parent"], t["depth"], t["max_depth"], 5, r, 1.0)
                ["next_tok"][0]) for r in range(40)}
    assert len(many) > 1
