"""GPU parity of medusa_tree_attention against the oracle (Medusa Heads glossary
page, "Tree attention and acceptance")."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import oracle as O
from util import oracle_attention_all, pool_map, to_dev, to_np

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _tree(kind):
    if kind == "c1":
        return O.tree_layout(O.product_tree_paths((2, 3)), 2)
    if kind == "sparse64":
        return O.tree_layout(O.sparse_tree_paths(64, 5, 8, 0.6, 0.5), 5)
    if kind == "dense":
        return O.tree_layout(O.product_tree_paths((4, 4, 4, 4)), 4)
    if kind == "small":
        return O.tree_layout(O.sparse_tree_paths(20, 4, 4, 0.6, 0.5), 4)
    if kind == "root":  # the root alone: plain decode attention over the prefix and itself
        return O.tree_layout(O.sparse_tree_paths(1, 4, 4, 0.6, 0.5), 4)
    if kind == "max512":  # the largest tree the entry point takes: 512 nodes, 8 mask words
        return O.tree_layout(O.sparse_tree_paths(512, 8, 8, 0.6, 0.5), 8)
    raise KeyError(kind)


def _run(M, x, kv_len, t, scale):
    out = M.tree_attention(to_dev(x["q"]), to_dev(x["k_cache"]), to_dev(x["v_cache"]),
                           to_dev(kv_len), to_dev(t["mask"]), scale=scale)
    torch.cuda.synchronize()
    return to_np(out)


@pytest.mark.parametrize("kind,B,Hq,Hkv,D,lens,Lmax,dtype", [
    ("c1", 1, 4, 4, 64, [128], 137, "f32"),
    ("small", 2, 3, 3, 128, [0, 33], 80, "f32"),
    ("sparse64", 3, 4, 4, 128, [0, 70, 500], 600, "bf16"),
    ("small", 2, 8, 2, 64, [5, 190], 240, "bf16"),
    ("dense", 1, 2, 2, 128, [300], 700, "bf16"),
    ("c1", 4, 4, 4, 64, [1, 63, 64, 65], 80, "bf16"),
    ("max512", 2, 2, 2, 128, [0, 200], 720, "bf16"),
    ("root", 2, 4, 4, 128, [0, 100], 110, "bf16"),
    ("root", 1, 8, 2, 64, [300], 310, "bf16"),
    ("max512", 1, 4, 2, 64, [129], 650, "f32"),
    # batch 1 with <= 64 query rows per block (rows spread over the four TMEM
    # lane quarters, split partials merged through the receive area), D 128
    # and 64, GQA, empty and long prefixes
    ("sparse64", 1, 4, 4, 128, [0], 80, "bf16"),
    ("c1", 1, 8, 2, 128, [500], 520, "bf16"),
    ("sparse64", 1, 2, 2, 64, [1000], 1100, "bf16"),
    ("small", 1, 6, 2, 128, [4000], 4100, "bf16"),
    # blocks of at most 64 rows with one key tile: the two-stream kernel with
    # rows spread over the TMEM lane quarters, query heads grouped 4 (TMA
    # query load) and 3 (rows gathered without TMA)
    ("c1", 2, 8, 2, 64, [20, 100], 110, "bf16"),
    ("c1", 2, 6, 2, 64, [20, 100], 110, "bf16"),
])
def test_attention_full_compare(medusa, kind, B, Hq, Hkv, D, lens, Lmax, dtype):
    t = _tree(kind)
    x = W.attention_inputs(seed=B + Hq + D, B=B, N=t["N"], Hq=Hq, Hkv=Hkv, D=D, Lmax=Lmax, dtype=dtype)
    kv_len = np.array(lens, np.int32)
    scale = float(np.float32(1 / np.sqrt(D)))
    got = _run(medusa, x, kv_len, t, scale)
    ref = oracle_attention_all(x["q"], x["k_cache"], x["v_cache"], kv_len, t["mask"], dtype, scale)
    assert np.abs(got - ref).max() <= TOL


@pytest.mark.parametrize("kind,B,Hq,Hkv,D,lens,Lmax", [
    # many (sequence, KV head, query block) units: odd block count (341 rows),
    # even count (512 rows x GQA 2), D 64 and 128, empty and ragged prefixes
    # (an empty prefix leaves a row a handful of keys, where the bf16 rounding
    # of the probabilities matters most)
    ("dense", 2, 38, 38, 128, [100, 300], 700),
    ("dense", 2, 38, 38, 64, [0, 250], 600),
    ("max512", 1, 76, 38, 64, [129], 650),
    # two-stream kernel (blocks of more than 64 rows, keys not split): one key
    # tile (the second stream empty), two and three tiles, and a group size of
    # 3 (query rows gathered without TMA)
    ("small", 4, 152, 38, 64, [0, 5, 108, 60], 128),
    ("small", 4, 152, 38, 128, [0, 200, 108, 350], 370),
    ("dense", 1, 156, 52, 64, [300], 700),
    # two-stream kernel over ragged lengths of 1 to 9 key tiles (single-tile
    # blocks leave the second stream empty) in more blocks than SMs
    ("small", 4, 160, 40, 128, [0, 300, 5, 1000], 1100),
])
def test_attention_many_blocks(medusa, kind, B, Hq, Hkv, D, lens, Lmax):
    t = _tree(kind)
    x = W.attention_inputs(seed=7 + B + D, B=B, N=t["N"], Hq=Hq, Hkv=Hkv, D=D, Lmax=Lmax, dtype="bf16")
    kv_len = np.array(lens, np.int32)
    scale = float(np.float32(1 / np.sqrt(D)))
    got = _run(medusa, x, kv_len, t, scale)
    ref = oracle_attention_all(x["q"], x["k_cache"], x["v_cache"], kv_len, t["mask"], "bf16", scale)
    assert np.abs(got - ref).max() <= TOL


def _sample_rows(B, N, Hq, n, seed):
    rng = np.random.default_rng(seed)
    rows = np.stack([rng.integers(0, B, n), rng.integers(0, N, n), rng.integers(0, Hq, n)], 1)
    rows[0] = [0, 0, 0]
    rows[1] = [B - 1, N - 1, Hq - 1]
    return rows.astype(np.int32)


def _full_size_rows(c, N, seed):
    """Rows compared at a workload's full size: at batch 1 every (node, query
    head); at larger batches every query row of one query head per sequence
    (the head rotating with the sequence, so all its KV-split CTAs and query
    blocks are met), plus 96 random rows and the first and last row."""
    B, Hq = c["B"], c["Hq"]
    if B == 1:
        n, h = np.meshgrid(np.arange(N), np.arange(Hq), indexing="ij")
        return np.stack([np.zeros(N * Hq, int), n.ravel(), h.ravel()], 1).astype(np.int32)
    full = [[b, i, (7 * b + 3) % Hq] for b in range(B) for i in range(N)]
    return np.concatenate([np.array(full, np.int32), _sample_rows(B, N, Hq, 96, seed)], 0)


@pytest.mark.parametrize("name,kind", [("h4096_b1_sparse64", "sparse64"), ("h5120_b8_ragged", "sparse64"),
                                       ("h4096_b4_kv8192", "dense"), ("h4096_b4_kv8192", "sparse64")])
def test_attention_full_size(medusa, name, kind):
    c = W.WORKLOADS[name]
    seed = c["seed"]
    t = _tree(kind)
    N = t["N"]
    kv_len = W.kv_lengths(seed, c["B"], c["L_lo"], c["L_hi"])
    Lmax = c["L_hi"] + N
    x = W.attention_inputs(seed=seed, B=c["B"], N=N, Hq=c["Hq"], Hkv=c["Hkv"], D=c["D"], Lmax=Lmax,
                           dtype=c["dtype"])
    scale = float(np.float32(1 / np.sqrt(c["D"])))
    got = _run(medusa, x, kv_len, t, scale)
    rows = _full_size_rows(c, N, seed)
    chunks = np.array_split(rows, 32)
    ref = np.concatenate(pool_map(lambda r: O.tree_attention(x["q"], x["k_cache"], x["v_cache"], kv_len,
                                                             t["mask"], c["dtype"], scale, rows=r), chunks), 0)
    sel = got[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert np.abs(sel - ref).max() <= TOL
    assert np.isfinite(got).all()


def test_out_of_range_kv_len_is_clamped(medusa):
    # kv_len beyond Lmax - N is clamped to Lmax - N (no read past the cache)
    t = _tree("c1")
    x = W.attention_inputs(seed=5, B=2, N=t["N"], Hq=2, Hkv=2, D=64, Lmax=100, dtype="bf16")
    scale = 0.125
    got = _run(medusa, x, np.array([10**6, -5], np.int32), t, scale)
    ref = O.tree_attention(x["q"], x["k_cache"], x["v_cache"], np.array([100 - t["N"], 0], np.int32),
                           t["mask"], "bf16", scale)
    assert np.abs(got - ref).max() <= TOL
