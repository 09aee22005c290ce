"""Pins of the oracle's candidate tree (Medusa Heads glossary page, "Tree
attention and acceptance")."""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import workloads as W
from oracle import oracle as O


def _check_invariants(t):
    N, W_ = t["N"], t["W"]
    parent, depth, mask = t["parent"], t["depth"], t["mask"]
    assert parent[0] == -1 and depth[0] == 0
    for i in range(1, N):
        assert 0 <= parent[i] < i
        assert depth[i] == depth[parent[i]] + 1
    for i in range(N):
        anc = set()
        a = i
        while a >= 0:
            anc.add(a)
            a = parent[a]
        bits = {m for m in range(N) if (int(mask[i, m // 64]) >> (m % 64)) & 1}
        assert bits == anc
        assert len(bits) == depth[i] + 1
    for row in t["retrieve"]:
        nodes = [x for x in row if x >= 0]
        assert nodes[0] == 0
        for a, b in zip(nodes, nodes[1:]):
            assert parent[b] == a
        leaf = nodes[-1]
        assert leaf not in set(parent.tolist())


def test_top2_x_top3_gives_six_candidates_sharing_prefixes():
    # "top-2 of head 1 x top-3 of head 2 -> six candidates that share prefixes"
    t = O.tree_layout(O.product_tree_paths((2, 3)), 2)
    assert t["n_paths"] == 6 and t["N"] == 9
    assert t["parent"].tolist() == [-1, 0, 0, 1, 1, 1, 2, 2, 2]
    # head 2 proposes the same tokens under every head-1 branch: same rank lists
    assert t["rank"][3:6].tolist() == t["rank"][6:9].tolist() == [0, 1, 2]
    _check_invariants(t)


def test_dense_tree_256_paths():
    # top-4 of each of 4 heads, Cartesian product: 4^4 = 256 root-to-leaf paths
    t = O.tree_layout(O.product_tree_paths((4, 4, 4, 4)), 4)
    assert t["n_paths"] == 256
    assert t["N"] == 1 + 4 + 16 + 64 + 256 and t["W"] == 6
    _check_invariants(t)


def _exact_sparse(n_nodes, max_depth, max_rank, hp, rp):
    items = []
    for d in range(1, max_depth + 1):
        for tup in itertools.product(range(max_rank), repeat=d):
            prior = Fraction(1)
            for k, r in enumerate(tup, start=1):
                prior *= hp ** k * rp ** r
            items.append((-prior, d, tup))
    items.sort()
    return sorted([it[2] for it in items[: n_nodes - 1]], key=lambda t: (len(t), t))


def test_sparse_64_tree_matches_exact_rational_priors():
    # 63 most accurate combinations + root, with rank r of head k accepted with
    # 0.6^k * 0.5^r; ranked with exact rational arithmetic (Fraction), so ties
    # are exact and broken by depth then lexicographic order.
    paths = O.sparse_tree_paths(64, 5, 8, 0.6, 0.5)
    got = [tuple(int(x) for x in r if x >= 0) for r in paths]
    assert got == _exact_sparse(64, 5, 8, Fraction(3, 5), Fraction(1, 2))
    t = O.tree_layout(paths, 5)
    assert t["N"] == 64
    assert np.bincount(t["depth"]).tolist() == [1, 8, 28, 22, 5]
    assert t["n_paths"] == 42
    assert (0, 1, 3) in got and (0, 2, 2) not in got  # the exact tie at the cut
    _check_invariants(t)


def test_sparse_tree_small_cases_exact():
    for n, d, r in [(2, 3, 3), (10, 3, 4), (30, 4, 3)]:
        got = [tuple(int(x) for x in row if x >= 0) for row in O.sparse_tree_paths(n, d, r, 0.6, 0.5)]
        assert got == _exact_sparse(n, d, r, Fraction(3, 5), Fraction(1, 2))


def _brute_layout(tuples):
    nodes = {()}
    for t in tuples:
        for L in range(1, len(t) + 1):
            nodes.add(tuple(t[:L]))
    order = sorted(nodes, key=lambda t: (len(t), t))
    index = {t: i for i, t in enumerate(order)}
    parent = [-1] + [index[t[:-1]] for t in order[1:]]
    return order, parent


def test_layout_matches_brute_force_on_random_tuple_sets():
    rng = np.random.default_rng(3)
    for trial in range(40):
        maxd = int(rng.integers(1, 5))
        P = int(rng.integers(1, 12))
        tuples = []
        for _ in range(P):
            d = int(rng.integers(1, maxd + 1))
            tuples.append(tuple(int(x) for x in rng.integers(0, 4, size=d)))
        arr = np.full((P, maxd), -1, np.int32)
        for i, t in enumerate(tuples):
            arr[i, : len(t)] = t
        t = O.tree_layout(arr, maxd)
        order, parent = _brute_layout(tuples)
        assert t["N"] == len(order)
        assert t["parent"].tolist() == parent
        assert t["depth"].tolist() == [len(x) for x in order]
        assert t["rank"].tolist() == [x[-1] if x else -1 for x in order]
        _check_invariants(t)


def test_build_tree_tokens_follow_rank_tuples():
    # every root-to-leaf path carries (root token, head1[r1], head2[r2], ...)
    B, K, k, V = 3, 4, 4, 500
    tuples = O.product_tree_paths((3, 2, 2))
    t = O.tree_layout(tuples, 3)
    lists = W.random_topk_lists(seed=4, B=B, K=K, topk=k, V=V)
    root = W.root_tokens(seed=4, B=B, V=V)
    cand = O.build_tree(lists, root, t["depth"], t["rank"])
    for b in range(B):
        for row, tup in zip(sorted(t["retrieve"].tolist(), key=lambda r: r), sorted(tuples.tolist())):
            nodes = [x for x in row if x >= 0]
            assert cand[b, nodes[0]] == root[b]
            for d, node in enumerate(nodes[1:], start=1):
                assert cand[b, node] == lists[b, d - 1, tup[d - 1]]
        # siblings hold distinct tokens
        for u in range(t["N"]):
            kids = [j for j in range(t["N"]) if t["parent"][j] == u]
            assert len({int(cand[b, j]) for j in kids}) == len(kids)


def test_layout_rejects_bad_padding():
    with pytest.raises(ValueError):
        O.tree_layout(np.array([[0, -1, 1]], np.int32), 3)
