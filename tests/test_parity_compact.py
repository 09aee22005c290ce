"""GPU parity of medusa_kv_compact against the oracle (Medusa Heads glossary page,
"Tree attention and acceptance": keep the longest accepted branch)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import oracle as O
from util import to_dev, to_np

pytestmark = pytest.mark.gpu


def _paths(B, N, Dmax, parent, depth, seed):
    """Random accepted branches of the tree: (path_nodes, accept_len, best_node)."""
    rng = np.random.default_rng(seed)
    path = np.full((B, Dmax + 1), -1, np.int32)
    alen = np.zeros(B, np.int32)
    best = np.zeros(B, np.int32)
    for b in range(B):
        n = int(rng.integers(0, N))
        best[b] = n
        alen[b] = depth[n]
        while n >= 0:
            path[b, depth[n]] = n
            n = parent[n]
    return path, alen, best


@pytest.mark.parametrize("B,Hkv,D,lens,dtype,kind", [
    (1, 32, 128, [2048], "bf16", "sparse64"),
    (8, 40, 128, [1024, 4096, 1500, 2000, 3000, 4000, 1, 0], "bf16", "sparse64"),
    (2, 4, 64, [128, 3], "f32", "c1"),
    (3, 9, 128, [7, 300, 10], "bf16", "dense"),
])
def test_compact_exact(medusa, B, Hkv, D, lens, dtype, kind):
    if kind == "c1":
        t = O.tree_layout(O.product_tree_paths((2, 3)), 2)
    elif kind == "dense":
        t = O.tree_layout(O.product_tree_paths((4, 4, 4, 4)), 4)
    else:
        t = O.tree_layout(O.sparse_tree_paths(64, 5, 8, 0.6, 0.5), 5)
    N, Dmax = t["N"], t["max_depth"]
    Lmax = max(lens) + N
    x = W.attention_inputs(seed=B + Hkv, B=B, N=1, Hq=1, Hkv=Hkv, D=D, Lmax=Lmax, dtype=dtype)
    H = 256
    ht = W.hidden_tree(seed=B, B=B, N=N, H=H, dtype=dtype)
    kv_len = np.array(lens, np.int32)
    path, alen, best = _paths(B, N, Dmax, t["parent"], t["depth"], seed=B * 3)
    k = to_dev(x["k_cache"]); v = to_dev(x["v_cache"]); kl = to_dev(kv_len)
    h_next, src = medusa.kv_compact(k, v, kl, to_dev(path), to_dev(alen), to_dev(best), N, Dmax,
                                    hidden_tree=to_dev(ht))
    torch.cuda.synchronize()
    k2, v2, kl2, hn2, src2 = O.kv_compact(x["k_cache"], x["v_cache"], kv_len, path, alen, best, ht, N, Dmax)
    assert np.array_equal(to_np(k), k2) and np.array_equal(to_np(v), v2)
    assert np.array_equal(to_np(kl), kl2)
    assert np.array_equal(to_np(h_next), hn2)
    assert np.array_equal(to_np(src), src2)


def test_out_of_range_sequence_is_left_unchanged(medusa):
    t = O.tree_layout(O.product_tree_paths((2, 3)), 2)
    N, Dmax, B = t["N"], 2, 3
    x = W.attention_inputs(seed=3, B=B, N=1, Hq=1, Hkv=2, D=64, Lmax=40, dtype="bf16")
    kv_len = np.array([5, 5, 35], np.int32)  # sequence 2: 35 + 9 > 40
    path = np.array([[0, 1, 4], [0, 2, -1], [0, 1, 3]], np.int32)
    alen = np.array([2, 3, 2], np.int32)      # sequence 1: accept_len beyond its path
    best = np.array([4, 2, 3], np.int32)
    k = to_dev(x["k_cache"]); v = to_dev(x["v_cache"]); kl = to_dev(kv_len)
    _, src = medusa.kv_compact(k, v, kl, to_dev(path), to_dev(alen), to_dev(best), N, Dmax)
    torch.cuda.synchronize()
    src = to_np(src)
    assert (src[1] == -2).all() and (src[2] == -2).all()
    assert to_np(kl).tolist() == [8, 5, 35]
    k2 = to_np(k)
    assert np.array_equal(k2[1:], x["k_cache"][1:])
    assert np.array_equal(k2[0, :, 5 + 1], x["k_cache"][0, :, 5 + 1])
    assert np.array_equal(k2[0, :, 5 + 2], x["k_cache"][0, :, 5 + 4])
