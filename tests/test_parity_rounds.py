"""Chained decode rounds (Medusa Heads glossary page, "Tree attention and
acceptance": the longest accepted branch is kept and its last hidden state
feeds the heads of the next round; e-book page "Giai ma dau co", "Why a round
always yields exactly k + 1 tokens").

Round r + 1 starts from round r's results: its root token is round r's next
token, its heads read round r's h_next, and its KV prefix is round r's compacted
cache (kv_len grew by accept_len + 1).  Each round's new inputs (queries, the
tree's K/V rows written at slots [kv_len, kv_len + N), the tree hidden states
and the verifier logits planted around the round's candidates) come from the
seeded generator.  Three rounds on the GPU through the C ABI must equal three
oracle rounds: tokens, accepted paths and the compacted cache bit for bit."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import oracle as O
from util import to_dev, to_np, topk_near_tie_ok

pytestmark = pytest.mark.gpu


def _round_inputs(seed, r, B, N, Hq, Hkv, D, H, dt):
    s = 1000 * seed + r
    att = W.attention_inputs(s, B, N, Hq, Hkv, D, N, dt)  # q and the tree's own K/V rows
    return dict(q=att["q"], tk=att["k_cache"], tv=att["v_cache"], ht=W.hidden_tree(s, B, N, H, dt))


@pytest.mark.parametrize("name,rounds", [("tiny_h256_v1000_f32", 3), ("h4096_b1_sparse64", 3)])
def test_chained_rounds(medusa, name, rounds):
    M = medusa
    c = W.WORKLOADS[name]
    seed, dt, B = c["seed"], c["dtype"], c["B"]
    if c["tree"] == "product":
        t = O.tree_layout(O.product_tree_paths(c["tree_ranks"]), len(c["tree_ranks"]))
    else:
        t = O.tree_layout(O.sparse_tree_paths(64, 5, 8, 0.6, 0.5), 5)
    N, Dmax = t["N"], t["max_depth"]
    heads = W.heads_inputs(seed, B, c["H"], c["V"], c["K"], dt)
    kv_len = W.kv_lengths(seed, B, c["L_lo"], c["L_hi"])
    Lmax = c["L_hi"] + N + rounds * (Dmax + 1)
    cache = W.attention_inputs(seed, B, N, c["Hq"], c["Hkv"], c["D"], Lmax, dt)
    scale = float(np.float32(1 / np.sqrt(c["D"])))

    # oracle state and GPU state start equal
    o_h, o_root, o_kl = heads["h"], W.root_tokens(seed, B, c["V"]), kv_len.copy()
    o_k, o_v = cache["k_cache"].copy(), cache["v_cache"].copy()
    g = {k: to_dev(heads[k]) for k in ("w1", "b1", "w2")}
    g_h, g_root, g_kl = to_dev(o_h), to_dev(o_root), to_dev(kv_len)
    g_k, g_v = to_dev(o_k), to_dev(o_v)
    depth, rank, parent, mask = (to_dev(t[k]) for k in ("depth", "rank", "parent", "mask"))
    total_tokens = 0
    for r in range(rounds):
        x = _round_inputs(seed, r, B, N, c["Hq"], c["Hkv"], c["D"], c["H"], dt)
        # the backbone's part of the round: the tree's K/V rows enter the cache
        for b in range(B):
            L = int(o_kl[b])
            o_k[b, :, L:L + N] = x["tk"][b]
            o_v[b, :, L:L + N] = x["tv"][b]
            g_k[b, :, L:L + N] = to_dev(x["tk"][b])
            g_v[b, :, L:L + N] = to_dev(x["tv"][b])
        # oracle round
        ref_logits = O.heads_logits(o_h, heads["w1"], heads["b1"], heads["w2"], dt)
        ref_idx, _ = O.topk(ref_logits, c["topk"])
        ref_cand = O.build_tree(ref_idx, o_root, t["depth"], t["rank"])
        ref_att = O.tree_attention(x["q"], o_k, o_v, o_kl, t["mask"], dt, scale,
                                   rows=np.array([[b, i, h] for b in range(B) for i in range(N)
                                                  for h in range(0, c["Hq"], max(1, c["Hq"] // 4))], np.int32))
        vlog = W.planted_logits(1000 * seed + r, ref_cand, t["parent"], c["V"], c["alpha"])
        ref_acc = O.verify_tree(vlog, ref_cand, t["parent"], t["depth"], Dmax)
        o_k, o_v, o_kl, o_hn, _ = O.kv_compact(o_k, o_v, o_kl, ref_acc["path_nodes"], ref_acc["accept_len"],
                                               ref_acc["best_node"], x["ht"], N, Dmax)
        # GPU round, every step through the C ABI, chained on device buffers
        idx, _, _ = M.heads_topk(g_h, g["w1"], g["b1"], g["w2"], c["topk"])
        cand = M.build_tree(idx, g_root, depth, rank)
        att = M.tree_attention(to_dev(x["q"]), g_k, g_v, g_kl, mask, scale)
        acc = M.verify_accept_tree(to_dev(vlog), cand, parent, depth, Dmax)
        g_h, _ = M.kv_compact(g_k, g_v, g_kl, acc["path_nodes"], acc["accept_len"], acc["best_node"], N, Dmax,
                              hidden_tree=to_dev(x["ht"]))
        g_root = acc["next_tok"]
        torch.cuda.synchronize()

        assert topk_near_tie_ok(to_np(idx), ref_idx, ref_logits) == 0, r
        assert np.array_equal(to_np(cand), ref_cand), r
        a = to_np(att)
        rows = [[b, i, h] for b in range(B) for i in range(N) for h in range(0, c["Hq"], max(1, c["Hq"] // 4))]
        sel = np.array([a[b, i, h] for b, i, h in rows])
        assert np.abs(sel - ref_att).max() <= 1e-2, r
        for k in ("accept_len", "best_node", "path_nodes", "next_tok"):
            assert np.array_equal(to_np(acc[k]), ref_acc[k]), (r, k)
        assert np.array_equal(to_np(g_kl), o_kl), r
        assert np.array_equal(to_np(g_h), o_hn), r
        # the next round starts from this round's results
        o_h, o_root = o_hn, ref_acc["next_tok"]
        total_tokens += int(ref_acc["accept_len"].sum()) + B
    assert np.array_equal(to_np(g_k), o_k) and np.array_equal(to_np(g_v), o_v)
    assert int(o_kl.sum()) == int(kv_len.sum()) + total_tokens  # k + 1 tokens per round
