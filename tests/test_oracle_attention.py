"""Pins of the oracle's tree attention (Medusa Heads glossary page, "Tree
attention and acceptance": all candidates scored in one pass, each seeing only
its ancestors)."""
import numpy as np
import pytest

import workloads as W
from oracle import oracle as O


def _ancestors(parent, i):
    out = set()
    while i >= 0:
        out.add(i)
        i = parent[i]
    return out


def _numpy_masked_attention(q, k, v, kv_len, parent, scale, group):
    # Library restatement: boolean mask built from the parent array, then a
    # softmax over the masked score matrix (float64).
    B, N, Hq, D = q.shape
    Lmax = k.shape[2]
    out = np.zeros((B, N, Hq, D))
    for b in range(B):
        L = int(kv_len[b])
        allow = np.zeros((N, Lmax), bool)
        allow[:, :L] = True
        for i in range(N):
            for m in _ancestors(parent, i):
                allow[i, L + m] = True
        for hq in range(Hq):
            hk = hq // group
            s = scale * q[b, :, hq, :] @ k[b, hk].T
            s = np.where(allow, s, -np.inf)
            p = np.exp(s - s.max(1, keepdims=True))
            p /= p.sum(1, keepdims=True)
            out[b, :, hq, :] = p @ v[b, hk]
    return out


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2)])
def test_matches_numpy_masked_softmax(Hq, Hkv):
    t = O.tree_layout(O.product_tree_paths((2, 3)), 2)
    B, N, D, Lmax = 3, t["N"], 16, 40
    x = W.attention_inputs(seed=5, B=B, N=N, Hq=Hq, Hkv=Hkv, D=D, Lmax=Lmax, dtype="f32")
    kv_len = np.array([0, 7, Lmax - N], np.int32)  # empty prefix, ragged, full
    scale = 1 / np.sqrt(D)
    got = O.tree_attention(x["q"], x["k_cache"], x["v_cache"], kv_len, t["mask"], "f32", scale)
    ref = _numpy_masked_attention(*(x[n].astype(np.float64) for n in ("q", "k_cache", "v_cache")),
                                  kv_len, t["parent"], scale, Hq // Hkv)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_row_list_matches_full():
    t = O.tree_layout(O.sparse_tree_paths(20, 4, 4, 0.6, 0.5), 4)
    B, N, Hq, D, Lmax = 2, t["N"], 3, 8, 64
    x = W.attention_inputs(seed=6, B=B, N=N, Hq=Hq, Hkv=Hq, D=D, Lmax=Lmax, dtype="bf16")
    kv_len = np.array([10, 33], np.int32)
    full = O.tree_attention(x["q"], x["k_cache"], x["v_cache"], kv_len, t["mask"], "bf16", 0.3)
    rows = np.array([[1, 5, 2], [0, 0, 0], [1, N - 1, 1]], np.int32)
    part = O.tree_attention(x["q"], x["k_cache"], x["v_cache"], kv_len, t["mask"], "bf16", 0.3,
                            rows=rows)
    for r, (b, i, h) in enumerate(rows):
        assert np.array_equal(part[r], full[b, i, h])


def test_root_only_tree_is_plain_decode_attention():
    # N = 1: the single query sees the L prefix keys and itself
    B, Hq, D, Lmax, L = 1, 2, 8, 30, 21
    x = W.attention_inputs(seed=7, B=B, N=1, Hq=Hq, Hkv=Hq, D=D, Lmax=Lmax, dtype="f32")
    mask = np.ones((1, 1), np.uint64)
    got = O.tree_attention(x["q"], x["k_cache"], x["v_cache"], np.array([L], np.int32), mask,
                           "f32", 0.5)
    for h in range(Hq):
        q = x["q"][0, 0, h].astype(np.float64)
        k = x["k_cache"][0, h, : L + 1].astype(np.float64)
        v = x["v_cache"][0, h, : L + 1].astype(np.float64)
        s = 0.5 * k @ q
        p = np.exp(s - s.max())
        np.testing.assert_allclose(got[0, 0, h], (p / p.sum()) @ v, atol=1e-12)


def test_uniform_scores_average_the_allowed_values():
    t = O.tree_layout(O.product_tree_paths((2, 2)), 2)
    B, N, Hq, D, Lmax, L = 1, t["N"], 1, 4, 16, 5
    x = W.attention_inputs(seed=8, B=B, N=N, Hq=Hq, Hkv=Hq, D=D, Lmax=Lmax, dtype="f32")
    q = np.zeros_like(x["q"])
    got = O.tree_attention(q, x["k_cache"], x["v_cache"], np.array([L], np.int32), t["mask"],
                           "f32", 1.0)
    for i in range(N):
        keys = list(range(L)) + [L + m for m in sorted(_ancestors(t["parent"], i))]
        np.testing.assert_allclose(got[0, i, 0], x["v_cache"][0, 0, keys].astype(np.float64).mean(0),
                                   atol=1e-12)


def test_rejects_overflowing_kv_len():
    t = O.tree_layout(O.product_tree_paths((2,)), 1)
    x = W.attention_inputs(seed=9, B=1, N=t["N"], Hq=1, Hkv=1, D=4, Lmax=8, dtype="f32")
    with pytest.raises(ValueError):
        O.tree_attention(x["q"], x["k_cache"], x["v_cache"], np.array([7], np.int32), t["mask"],
                         "f32", 1.0)
