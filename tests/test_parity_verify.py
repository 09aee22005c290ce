"""GPU parity of medusa_verify_accept_tree against the oracle (Medusa Heads
glossary page, "Tree attention and acceptance"; e-book page "Giai ma dau co",
"Why a round always yields exactly k + 1 tokens")."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import oracle as O
from util import to_dev, to_np

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


def _typical_compare(got, ref, parent, band=1e-4):
    """Exact equality, except for sequences where some node's P(candidate) lies
    within a relative band of its parent's threshold (float32 and float64 may
    decide either way there); returns the number of such sequences."""
    amb = 0
    for b in range(len(ref["accept_len"])):
        tau = ref["tau"][b, parent[1:]]
        if (np.abs(ref["pcand"][b, 1:] - tau) <= band * tau).any():
            amb += 1
            continue
        for key in KEYS:
            assert np.array_equal(got[key][b], ref[key][b]), (key, b)
    return amb


@pytest.mark.parametrize("kind,B,T", [("dense", 4, 1.0), ("sparse64", 4, 1.0), ("sparse64", 2, 0.7)])
def test_typical_full_size(medusa, kind, B, T):
    t = _tree(kind)
    V = 32000
    cand = _cands(t, B, V, seed=70, K=5 if kind == "sparse64" else 4, k=8 if kind == "sparse64" else 4)
    logits = W.normal_logits(70, B, t["N"], V, 3.0)
    got = _gpu(medusa, logits, cand, t, "typical", T)
    ref = O.verify_tree(logits, cand, t["parent"], t["depth"], t["max_depth"], "typical", T)
    assert _typical_compare(got, ref, t["parent"]) <= 1


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
    # accept outputs as typical acceptance; the next token is the oracle's own
    # exponential-race draw from the best node's softmax, except where the
    # oracle's two best race keys are within 1e-5 relative (counted)
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
        amb = 0
        for b in range(B):
            tau = typ["tau"][b, t["parent"][1:]]
            if (np.abs(typ["pcand"][b, 1:] - tau) <= 1e-4 * tau).any():
                amb += 1
                continue
            for key in ("accept_len", "best_node", "path_nodes"):
                assert np.array_equal(got[key][b], ref[key][b]), (key, b)
            if got["next_tok"][b] != ref["next_tok"][b]:
                assert ref["race_gap"][b] < 1e-5, (b, got["next_tok"][b], ref["next_tok"][b])
                ties += 1
        assert amb <= 1
    assert ties <= 1
