"""One whole Medusa decode step on the GPU (heads -> tree -> tree attention ->
acceptance -> KV compaction) against the same step in the oracle: the tiny fp32
workload and the Vicuna-7B-shaped batch-1 workload in full, the 13B-shaped
ragged batch-8 step (greedy) and the batch-4 KV-8192 dense-tree step (typical
acceptance), each with every output compared (attention on every row of one
query head per sequence plus sampled rows)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import oracle as O
from util import check_typical, pool_map, to_dev, to_np, topk_near_tie_ok

pytestmark = pytest.mark.gpu


def _tree(c):
    if c["tree"] in ("product", "dense"):
        paths = O.product_tree_paths(c["tree_ranks"])
        return O.tree_layout(paths, len(c["tree_ranks"]))
    return O.tree_layout(O.sparse_tree_paths(64, 5, 8, 0.6, 0.5), 5)


@pytest.mark.parametrize("name", ["tiny_h256_v1000_f32", "h4096_b1_sparse64"])
def test_full_step(medusa, name):
    M = medusa
    c = W.WORKLOADS[name]
    seed = c["seed"]
    t = _tree(c)
    N, Dmax = t["N"], t["max_depth"]
    dt = c["dtype"]
    heads = W.heads_inputs(seed, c["B"], c["H"], c["V"], c["K"], dt)
    kv_len = W.kv_lengths(seed, c["B"], c["L_lo"], c["L_hi"])
    Lmax = c["L_hi"] + N
    att = W.attention_inputs(seed, c["B"], N, c["Hq"], c["Hkv"], c["D"], Lmax, dt)
    ht = W.hidden_tree(seed, c["B"], N, c["H"], dt)
    root = W.root_tokens(seed, c["B"], c["V"])
    scale = float(np.float32(1 / np.sqrt(c["D"])))

    # oracle step
    ref_logits = O.heads_logits(heads["h"], heads["w1"], heads["b1"], heads["w2"], dt)
    ref_idx, _ = O.topk(ref_logits, c["topk"])
    ref_cand = O.build_tree(ref_idx, root, t["depth"], t["rank"])
    ref_att = O.tree_attention(att["q"], att["k_cache"], att["v_cache"], kv_len, t["mask"], dt, scale)
    vlogits = W.planted_logits(seed, ref_cand, t["parent"], c["V"], c["alpha"])
    ref_acc = O.verify_tree(vlogits, ref_cand, t["parent"], t["depth"], Dmax)
    ref_k, ref_v, ref_kl, ref_hn, ref_src = O.kv_compact(
        att["k_cache"], att["v_cache"], kv_len, ref_acc["path_nodes"], ref_acc["accept_len"],
        ref_acc["best_node"], ht, N, Dmax)

    # GPU step, all through the C ABI
    dev = {k: to_dev(v) for k, v in heads.items()}
    idx, val, _ = M.heads_topk(dev["h"], dev["w1"], dev["b1"], dev["w2"], c["topk"])
    cand = M.build_tree(idx, to_dev(root), to_dev(t["depth"]), to_dev(t["rank"]))
    kc, vc, kl = to_dev(att["k_cache"]), to_dev(att["v_cache"]), to_dev(kv_len)
    o = M.tree_attention(to_dev(att["q"]), kc, vc, kl, to_dev(t["mask"]), scale)
    acc = M.verify_accept_tree(to_dev(vlogits), cand, to_dev(t["parent"]), to_dev(t["depth"]), Dmax)
    h_next, src = M.kv_compact(kc, vc, kl, acc["path_nodes"], acc["accept_len"], acc["best_node"], N,
                               Dmax, hidden_tree=to_dev(ht))
    torch.cuda.synchronize()

    assert topk_near_tie_ok(to_np(idx), ref_idx, ref_logits) == 0
    assert np.array_equal(to_np(cand), ref_cand)
    assert np.abs(to_np(o) - ref_att).max() <= 1e-2
    for k in ("accept_len", "best_node", "path_nodes", "next_tok"):
        assert np.array_equal(to_np(acc[k]), ref_acc[k]), k
    assert np.array_equal(to_np(kc), ref_k) and np.array_equal(to_np(vc), ref_v)
    assert np.array_equal(to_np(kl), ref_kl)
    assert np.array_equal(to_np(h_next), ref_hn) and np.array_equal(to_np(src), ref_src)


def _att_rows(B, N, Hq, seed):
    rng = np.random.default_rng(seed)
    full = [[b, i, (7 * b + 3) % Hq] for b in range(B) for i in range(N)]
    extra = np.stack([rng.integers(0, B, 64), rng.integers(0, N, 64), rng.integers(0, Hq, 64)], 1)
    return np.concatenate([np.array(full), extra], 0).astype(np.int32)


@pytest.mark.parametrize("name", ["h5120_b8_ragged", "h4096_b4_kv8192"])
def test_full_step_batched(medusa, name):
    # 13B-shaped heads at batch 8 (tensor cores), the sparse 64-node tree per
    # sequence, 40-head attention over ragged KV lengths, greedy acceptance of
    # planted logits, compaction; or batch 4 with the dense 341-node tree, KV
    # 8192 and typical acceptance of N(0, 3) logits
    M = medusa
    c = W.WORKLOADS[name]
    seed = c["seed"]
    t = _tree(c)
    N, Dmax = t["N"], t["max_depth"]
    dt, B = c["dtype"], c["B"]
    typical = c["accept"] == "typical"
    heads = W.heads_inputs(seed, B, c["H"], c["V"], c["K"], dt)
    kv_len = W.kv_lengths(seed, B, c["L_lo"], c["L_hi"])
    Lmax = c["L_hi"] + N
    att = W.attention_inputs(seed, B, N, c["Hq"], c["Hkv"], c["D"], Lmax, dt)
    ht = W.hidden_tree(seed, B, N, c["H"], dt)
    root = W.root_tokens(seed, B, c["V"])
    scale = float(np.float32(1 / np.sqrt(c["D"])))

    # oracle: heads per sequence, candidates, verifier logits around them
    ref_logits = np.concatenate(pool_map(
        lambda b: O.heads_logits(heads["h"][b:b + 1], heads["w1"], heads["b1"], heads["w2"], dt), range(B)), 0)
    ref_idx, _ = O.topk(ref_logits, c["topk"])
    ref_cand = O.build_tree(ref_idx, root, t["depth"], t["rank"])
    if typical:
        vlogits = W.normal_logits(seed, B, N, c["V"], c["logit_std"])
    else:
        vlogits = W.planted_logits(seed, ref_cand, t["parent"], c["V"], c["alpha"])

    # GPU step through the C ABI
    dev = {k: to_dev(v) for k, v in heads.items()}
    idx, val, _ = M.heads_topk(dev["h"], dev["w1"], dev["b1"], dev["w2"], c["topk"])
    cand = M.build_tree(idx, to_dev(root), to_dev(t["depth"]), to_dev(t["rank"]))
    kc, vc, kl = to_dev(att["k_cache"]), to_dev(att["v_cache"]), to_dev(kv_len)
    o = M.tree_attention(to_dev(att["q"]), kc, vc, kl, to_dev(t["mask"]), scale)
    mode = "typical" if typical else "greedy"
    acc = M.verify_accept_tree(to_dev(vlogits), cand, to_dev(t["parent"]), to_dev(t["depth"]), Dmax, mode)
    h_next, src = M.kv_compact(kc, vc, kl, acc["path_nodes"], acc["accept_len"], acc["best_node"], N,
                               Dmax, hidden_tree=to_dev(ht))
    torch.cuda.synchronize()

    assert topk_near_tie_ok(to_np(idx), ref_idx, ref_logits) == 0
    assert np.array_equal(to_np(cand), ref_cand)
    rows = _att_rows(B, N, c["Hq"], seed)
    ref_att = np.concatenate(pool_map(
        lambda r: O.tree_attention(att["q"], att["k_cache"], att["v_cache"], kv_len, t["mask"], dt, scale, rows=r),
        np.array_split(rows, 32)), 0)
    got_att = to_np(o)
    assert np.abs(got_att[rows[:, 0], rows[:, 1], rows[:, 2]] - ref_att).max() <= 1e-2
    ref_acc = O.verify_tree(vlogits, ref_cand, t["parent"], t["depth"], Dmax, mode)
    got_acc = {k: to_np(v) for k, v in acc.items()}
    if typical:
        check_typical(got_acc, ref_acc, t["parent"], t["depth"])
    else:
        for k in ("accept_len", "best_node", "path_nodes", "next_tok"):
            assert np.array_equal(got_acc[k], ref_acc[k]), k
        assert len(set(got_acc["accept_len"].tolist())) > 1  # accepted lengths vary per sequence
    # compaction of the accepted branch the GPU reported (one of the allowed ones)
    ref_k, ref_v, ref_kl, ref_hn, ref_src = O.kv_compact(
        att["k_cache"], att["v_cache"], kv_len, got_acc["path_nodes"], got_acc["accept_len"],
        got_acc["best_node"], ht, N, Dmax)
    assert np.array_equal(to_np(kc), ref_k) and np.array_equal(to_np(vc), ref_v)
    assert np.array_equal(to_np(kl), ref_kl)
    assert np.array_equal(to_np(h_next), ref_hn) and np.array_equal(to_np(src), ref_src)
