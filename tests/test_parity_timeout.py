"""The give-up path of the bounded device waits, made to run on purpose: with
the tensor-core kernels' first-wait limit lowered to a few clock cycles
(medusa_set_wait_limit), their waits for TMA tiles and MMA results run out
before the data arrives.  A kernel that gives up lets its own copies and MMAs
in flight land (those waits keep the default limit), frees its tensor memory
and marks its outputs; medusa_device_status then reports MEDUSA_ERR_TIMEOUT.
With the default limit restored the next calls are correct again (bitwise equal
to the calls made before) and the status is clear.

Covers the tensor-core paths: tree attention (bf16, a cluster of KV splits,
and the two-stream kernel of blocks of more than 64 rows with unsplit keys),
the heads at a bf16 batch on the tensor cores, and the fused verification
projection."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import oracle as O
from util import to_dev, to_np

pytestmark = pytest.mark.gpu


def _calls(M):
    t = O.tree_layout(O.sparse_tree_paths(64, 5, 8, 0.6, 0.5), 5)
    N = t["N"]
    att = W.attention_inputs(3, 1, N, 32, 32, 128, 2048 + N, "bf16")
    td = O.tree_layout(O.product_tree_paths((4, 4, 4, 4)), 4)  # 341 nodes
    att2 = W.attention_inputs(6, 2, td["N"], 76, 76, 64, 700, "bf16")
    x = W.heads_inputs(4, 4, 512, 3001, 5, "bf16")
    hid = W.hidden_tree(5, 2, N, 512, "bf16")
    lm = W.normal(5, "LMHEAD", (3001, 512), 0.02, "bf16")
    cand = O.build_tree(W.random_topk_lists(5, 2, 5, 8, 3001), W.root_tokens(5, 2, 3001), t["depth"], t["rank"])
    d = dict(q=to_dev(att["q"]), k=to_dev(att["k_cache"]), v=to_dev(att["v_cache"]),
             kl=to_dev(np.array([2048], np.int32)), mask=to_dev(t["mask"]),
             q2=to_dev(att2["q"]), k2=to_dev(att2["k_cache"]), v2=to_dev(att2["v_cache"]),
             kl2=to_dev(np.array([100, 300], np.int32)), mask2=to_dev(td["mask"]),
             h=[to_dev(x[n]) for n in ("h", "w1", "b1", "w2")],
             hid=to_dev(hid), lm=to_dev(lm), cand=to_dev(cand), parent=to_dev(t["parent"]),
             depth=to_dev(t["depth"]))

    def run():
        o = M.tree_attention(d["q"], d["k"], d["v"], d["kl"], d["mask"], 1 / np.sqrt(128))
        o2 = M.tree_attention(d["q2"], d["k2"], d["v2"], d["kl2"], d["mask2"], 1 / np.sqrt(64))
        idx, val, _ = M.heads_topk(*d["h"], 8)
        acc = M.verify_project_tree(d["hid"], d["lm"], d["cand"], d["parent"], d["depth"], t["max_depth"])
        torch.cuda.synchronize()
        return (to_np(o), to_np(o2)), to_np(idx), {k: to_np(v) for k, v in acc.items()}
    return run


def test_wait_give_up_is_reported_and_the_next_calls_are_correct(medusa):
    M = medusa
    run = _calls(M)
    M.device_status()  # clear whatever an earlier test left
    o0, idx0, acc0 = run()
    M.device_status()
    assert all(np.isfinite(o).all() for o in o0) and (idx0 >= 0).all() and (acc0["accept_len"] >= 0).all()
    try:
        M.set_wait_limit(4)
        o1, idx1, acc1 = run()
    finally:
        M.set_wait_limit(0)
    with pytest.raises(M.MedusaError) as e:
        M.device_status()
    assert e.value.code == -5
    # the outputs of the CTAs that gave up are marked, nothing else is invented
    for a, b in zip(o1, o0):
        assert np.isnan(a).any() and (np.isnan(a) | (a == b)).all()
    assert (idx1 == -1).any() and ((idx1 == -1) | (idx1 == idx0)).all()
    assert (acc1["accept_len"] == -1).all()
    # default limit again: same results as before, status clear
    o2, idx2, acc2 = run()
    M.device_status()
    assert all(np.array_equal(a, b) for a, b in zip(o2, o0)) and np.array_equal(idx2, idx0)
    for k in acc0:
        assert np.array_equal(acc2[k], acc0[k]), k
