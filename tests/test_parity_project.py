"""GPU parity of medusa_verify_project_tree, the verification projection fused
with tree acceptance (Medusa Heads glossary page, "Tree attention and
acceptance": the base model scores every candidate of the tree in one pass; its
next-token logits at node u are lm_head . hidden_u).

The oracle side is the oracle's lm_head logits (float64 from the same bf16
inputs, rounded to float32 as verifier logits) followed by the oracle's tree
acceptance.  Candidates are planted through the tokens: with probability 0.8
the lowest-index child of each node carries the argmax of the node's oracle
logits row, so acceptance paths of every length occur."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import oracle as O
from util import TYPICAL_BAND, check_typical, to_dev, to_np

pytestmark = pytest.mark.gpu

KEYS = ("accept_len", "best_node", "path_nodes", "next_tok")


def _tree(kind):
    if kind == "c1":
        return O.tree_layout(O.product_tree_paths((2, 3)), 2)
    if kind == "sparse64":
        return O.tree_layout(O.sparse_tree_paths(64, 5, 8, 0.6, 0.5), 5)
    if kind == "dense":
        return O.tree_layout(O.product_tree_paths((4, 4, 4, 4)), 4)
    raise KeyError(kind)


def _inputs(t, B, H, V, seed, K, k):
    hid = W.hidden_tree(seed, B, t["N"], H, "bf16")
    lm = W.normal(seed, "LMHEAD", (V, H), 0.02, "bf16")
    lists = W.random_topk_lists(seed, B, K, k, V)
    cand = O.build_tree(lists, W.root_tokens(seed, B, V), t["depth"], t["rank"])
    return hid, lm, cand


def _oracle_logits(hid, lm):
    B, N, H = hid.shape
    return O.lm_head_logits_matmul(hid.reshape(B * N, H), lm, "bf16").reshape(B, N, -1)


def _plant(cand, parent, logits64, seed, alpha=0.8):
    """Lowest-index child of each node takes the argmax of the node's row with
    probability alpha (test-side planting; the rows themselves are not changed)."""
    cand = cand.copy()
    g = np.random.default_rng(seed)
    B, N = cand.shape
    children = [[] for _ in range(N)]
    for j in range(1, N):
        children[parent[j]].append(j)
    for b in range(B):
        for u in range(N):
            if children[u] and g.random() < alpha:
                cand[b, min(children[u])] = int(np.argmax(logits64[b, u]))
    return cand


def _near_tie_rows(logits64, band=1e-5):
    """Rows whose two largest float64 logits are within band * max(1, |top|)."""
    top2 = -np.sort(-logits64, axis=-1)[..., :2]
    return np.abs(top2[..., 0] - top2[..., 1]) <= band * np.maximum(1.0, np.abs(top2[..., 0]))


def _gpu(M, hid, lm, cand, t, mode="greedy", T=1.0, eps=0.09, delta=0.3):
    r = M.verify_project_tree(to_dev(hid), to_dev(lm), to_dev(cand), to_dev(t["parent"]),
                              to_dev(t["depth"]), t["max_depth"], mode, T, eps, delta)
    torch.cuda.synchronize()
    return {k: to_np(v) for k, v in r.items()}


def _compare_greedy(got, ref, near):
    """Exact equality, except on sequences with an oracle near-tie row (counted)."""
    amb = 0
    for b in range(len(ref["accept_len"])):
        if near[b].any():
            amb += 1
            continue
        for key in KEYS:
            assert np.array_equal(got[key][b], ref[key][b]), (key, b, got[key][b], ref[key][b])
    return amb


def _typical_band(lg, T):
    """Band of the typical decisions on the fused projection: the acceptance
    kernels' own measured band (TYPICAL_BAND) plus the float32 logits' own
    error, which moves x_c - E_P[x] by at most twice the largest logit error
    over T; that error is taken as the near-tie band of the greedy comparisons,
    1e-5 * max(1, |logit|)."""
    return TYPICAL_BAND + 2e-5 * max(1.0, float(np.abs(lg).max())) / T


# (tree, B, H, V): one row block and one vocab tile up to 11 row blocks; ragged
# last hidden slice (H % 64), ragged last vocab tile (V % 256), ragged last row
# block ((B*N) % 128)
SHAPES = [("c1", 2, 256, 1000), ("sparse64", 3, 200, 3001), ("dense", 4, 512, 2000)]


@pytest.mark.parametrize("kind,B,H,V", SHAPES)
def test_greedy_matches_oracle(medusa, kind, B, H, V):
    t = _tree(kind)
    K, k = (3, 3) if kind == "c1" else ((4, 4) if kind == "dense" else (5, 8))
    hid, lm, cand0 = _inputs(t, B, H, V, 80, K, k)
    lg = _oracle_logits(hid, lm)
    cand = _plant(cand0, t["parent"], lg, 80)
    got = _gpu(medusa, hid, lm, cand, t)
    ref = O.verify_tree(lg.astype(np.float32), cand, t["parent"], t["depth"], t["max_depth"])
    assert _compare_greedy(got, ref, _near_tie_rows(lg)) == 0
    assert (ref["accept_len"] > 0).any()


@pytest.mark.parametrize("kind,B,H,V", SHAPES)
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_typical_matches_oracle(medusa, kind, B, H, V, T):
    t = _tree(kind)
    K, k = (3, 3) if kind == "c1" else ((4, 4) if kind == "dense" else (5, 8))
    hid, lm, cand0 = _inputs(t, B, H, V, 81, K, k)
    lg = _oracle_logits(hid, lm)
    cand = _plant(cand0, t["parent"], lg, 81)
    got = _gpu(medusa, hid, lm, cand, t, "typical", T)
    ref = O.verify_tree(lg.astype(np.float32), cand, t["parent"], t["depth"], t["max_depth"],
                        "typical", T)
    # next_tok is the argmax of the best row: compared where no near tie exists
    near = _near_tie_rows(lg)
    check_typical(got, ref, t["parent"], t["depth"], band=_typical_band(lg, T), next_tok=False)
    for b in range(B):
        if not near[b, got["best_node"][b]]:
            assert got["next_tok"][b] == int(np.argmax(lg[b, got["best_node"][b]]))


def test_greedy_vicuna7b_full_size(medusa):
    # hidden 4096, vocab 32000, sparse 64-node tree, batch 1: all 64 rows from the oracle
    t = _tree("sparse64")
    hid, lm, cand0 = _inputs(t, 1, 4096, 32000, 82, 5, 8)
    lg = _oracle_logits(hid, lm)
    for seed in range(3):
        cand = _plant(cand0, t["parent"], lg, 82 + seed)
        got = _gpu(medusa, hid, lm, cand, t)
        ref = O.verify_tree(lg.astype(np.float32), cand, t["parent"], t["depth"], t["max_depth"])
        assert _compare_greedy(got, ref, _near_tie_rows(lg)) == 0


def test_greedy_dense_full_size_along_path(medusa):
    # batch 4 x 341 nodes, hidden 4096, vocab 32000 (1364 rows in 11 row blocks).
    # The oracle computes only the rows on the GPU's reported path: in greedy
    # mode siblings carry distinct tokens, so the accepted nodes form one chain
    # from the root, and the result is right iff each path node's token is the
    # argmax of its parent's row, next_tok is the argmax of the last row, and no
    # child of the last node carries that argmax.
    t = _tree("dense")
    B, H, V = 4, 4096, 32000
    hid, lm, cand = _inputs(t, B, H, V, 83, 4, 4)
    # plant along the rank-0 chain using the oracle rows of that chain only
    parent, depth, N = t["parent"], t["depth"], t["N"]
    children = [[] for _ in range(N)]
    for j in range(1, N):
        children[parent[j]].append(j)
    g = np.random.default_rng(83)
    for b in range(B):
        u = 0
        while children[u] and g.random() < 0.8:
            row = O.lm_head_logits(hid[b, u][None], lm, "bf16")[0]
            c = min(children[u])
            cand[b, c] = int(np.argmax(row))
            u = c
    got = _gpu(medusa, hid, lm, cand, t)
    for b in range(B):
        a, best = int(got["accept_len"][b]), int(got["best_node"][b])
        path = got["path_nodes"][b]
        assert 0 <= a <= t["max_depth"] and depth[best] == a and path[a] == best and path[0] == 0
        assert (path[a + 1:] == -1).all()
        rows = O.lm_head_logits(hid[b, path[: a + 1]], lm, "bf16")
        for i in range(1, a + 1):
            assert parent[path[i]] == path[i - 1]
            assert cand[b, path[i]] == int(np.argmax(rows[i - 1])), (b, i)
        top = int(np.argmax(rows[a]))
        assert got["next_tok"][b] == top
        assert all(cand[b, c] != top for c in children[best])
    assert (got["accept_len"] > 0).any()


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_typical_dense_full_size(medusa, T):
    # batch 4 x 341 nodes, hidden 4096, vocab 32000 (1364 rows in 11 row blocks,
    # the bench's tensor-bound shape) in typical mode, every row from the
    # oracle.  Candidates planted through the tokens: the lowest-index child of
    # each node carries a token of high probability under the node's row (one
    # of its top 3), so decisions of every kind occur.
    t = _tree("dense")
    B, H, V = 4, 4096, 32000
    hid, lm, cand0 = _inputs(t, B, H, V, 84, 4, 4)
    lg = _oracle_logits(hid, lm)
    cand = cand0.copy()
    g = np.random.default_rng(84)
    parent, N = t["parent"], t["N"]
    children = [[] for _ in range(N)]
    for j in range(1, N):
        children[parent[j]].append(j)
    for b in range(B):
        for u in range(N):
            if children[u] and g.random() < 0.8:
                cand[b, min(children[u])] = int(np.argsort(-lg[b, u])[g.integers(0, 3)])
    got = _gpu(medusa, hid, lm, cand, t, "typical", T, 0.05, 0.3)
    ref = O.verify_tree(lg.astype(np.float32), cand, t["parent"], t["depth"], t["max_depth"],
                        "typical", T, 0.05, 0.3)
    check_typical(got, ref, t["parent"], t["depth"], band=_typical_band(lg, T), next_tok=False)
    near = _near_tie_rows(lg)
    for b in range(B):
        if not near[b, got["best_node"][b]]:
            assert got["next_tok"][b] == int(np.argmax(lg[b, got["best_node"][b]]))
    assert (ref["accept_len"] > 0).any()


def test_rejects_bad_arguments(medusa):
    # the C ABI refuses float32 operands and a hidden size that is not a
    # multiple of 8, with nothing enqueued
    import ctypes as C
    L = medusa.lib()
    t = _tree("c1")
    hid = torch.zeros(1, t["N"], 256, device="cuda", dtype=torch.float32)
    lm = torch.zeros(1000, 256, device="cuda", dtype=torch.float32)
    i32 = [torch.zeros(t["N"], dtype=torch.int32, device="cuda") for _ in range(3)]
    outs = [torch.zeros(4, dtype=torch.int32, device="cuda") for _ in range(4)]
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    p = lambda x: C.c_void_p(x.data_ptr())
    args = lambda dt, H: (p(hid), p(lm), dt, p(i32[0]), p(i32[1]), p(i32[2]), 1, t["N"], H, 1000,
                          2, 0, C.c_float(1), C.c_float(0), C.c_float(0), *map(p, outs), p(ws),
                          ws.numel(), None)
    assert L.medusa_verify_project_tree(*args(0, 256)) == -2   # MEDUSA_F32: unsupported
    assert L.medusa_verify_project_tree(*args(1, 252)) == -2   # H % 8 != 0
    torch.cuda.synchronize()
