"""GPU parity of medusa_heads_topk against the oracle (Medusa Heads glossary
page, "How heads predict later tokens")."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import oracle as O
from util import pool_map, to_dev, to_np, topk_near_tie_ok

pytestmark = pytest.mark.gpu


def _run(M, x, topk):
    idx, val, lg = M.heads_topk(to_dev(x["h"]), to_dev(x["w1"]), to_dev(x["b1"]), to_dev(x["w2"]),
                                topk, want_logits=True)
    torch.cuda.synchronize()
    return to_np(idx), to_np(val), to_np(lg)


@pytest.mark.parametrize("B,H,V,K,topk,dtype,tol", [
    # CUDA cores: float32 up to batch 8, bf16 at batch 1-2 or H % 128 != 0
    (1, 256, 1000, 3, 3, "f32", 1e-5),      # tiny fp32 step
    (1, 512, 3001, 5, 8, "bf16", 2e-2),     # several slices, ragged vocab tail
    (2, 512, 3001, 5, 8, "bf16", 2e-2),
    (3, 264, 3001, 5, 8, "bf16", 2e-2),
    (8, 264, 1000, 3, 8, "bf16", 2e-2),
    (5, 264, 777, 4, 5, "f32", 1e-5),
    (2, 16384, 300, 1, 4, "bf16", 2e-2),    # largest hidden size (B * H = 32768)
    (1, 128, 300, 64, 4, "bf16", 2e-2),     # largest head count
    (1, 8, 16, 1, 16, "f32", 1e-5),         # smallest hidden size, top-k of the whole vocab
    # bf16 batches 3-64 with H % 128 == 0 run on the tensor cores, the batch
    # padded to a multiple of 16 (planes at columns [0, Bp), [Bp, 2Bp),
    # [2Bp, 3Bp)): ragged vocab tiles, heads split across CTAs, runs that cross
    # heads, running per-sequence lists
    (3, 512, 3001, 5, 8, "bf16", 2e-2),
    (4, 256, 1000, 3, 8, "bf16", 2e-2),
    (5, 384, 1337, 4, 8, "bf16", 2e-2),
    (6, 640, 4099, 5, 8, "bf16", 2e-2),
    (7, 128, 300, 6, 4, "bf16", 2e-2),
    (8, 1024, 2000, 2, 16, "bf16", 2e-2),
    (9, 256, 1000, 3, 8, "bf16", 2e-2),
    (16, 384, 1337, 4, 8, "bf16", 2e-2),
    (20, 512, 3001, 5, 16, "bf16", 2e-2),
    (33, 128, 300, 2, 4, "bf16", 2e-2),
    (48, 256, 777, 3, 8, "bf16", 2e-2),
    (64, 256, 1000, 5, 8, "bf16", 2e-2),
    (3, 16384, 300, 1, 4, "bf16", 2e-2),    # largest hidden size on the tensor cores
    (4, 128, 300, 64, 4, "bf16", 2e-2),     # largest head count on the tensor cores
    (3, 128, 16, 2, 16, "bf16", 2e-2),      # vocab below one 128-row tile, top-k of all of it
])
def test_heads_small(medusa, B, H, V, K, topk, dtype, tol):
    x = W.heads_inputs(seed=B * 7 + K, B=B, H=H, V=V, K=K, dtype=dtype, b1_std=0.5)
    idx, val, lg = _run(medusa, x, topk)
    ref = O.heads_logits(x["h"], x["w1"], x["b1"], x["w2"], dtype)
    assert np.abs(lg - ref).max() <= tol
    ridx, rval = O.topk(ref, topk)
    topk_near_tie_ok(idx, ridx, ref)
    assert np.abs(val - rval).max() <= tol


def test_zero_init_heads_reproduce_lm_head(medusa):
    # hidden 256, vocab 1000, 3 heads, W1 = b1 = 0 and W2_k = lm_head: every head's
    # logits are bitwise equal on the GPU and match lm_head h from the oracle
    x = W.heads_inputs(seed=1, B=1, H=256, V=1000, K=3, dtype="f32", zero_init=True)
    idx, val, lg = _run(medusa, x, 3)
    assert [bool(np.array_equal(lg[:, k], lg[:, 0])) for k in range(3)] == [True, True, True]
    lm = O.lm_head_logits(x["h"], x["lm_head"], "f32")
    assert np.abs(lg[:, 0] - lm).max() <= 1e-5
    ridx, _ = O.topk(lm, 3)
    for k in range(3):
        topk_near_tie_ok(idx[:, k], ridx, lm)


def _oracle_rows(x, rows, dtype):
    """Oracle logits of the given sequences, one sequence per host core."""
    parts = pool_map(lambda b: O.heads_logits(x["h"][b:b + 1], x["w1"], x["b1"], x["w2"], dtype), rows)
    return np.concatenate(parts, 0)


@pytest.mark.parametrize("name", ["h4096_b1_sparse64", "h5120_b8_ragged", "h4096_b4_kv8192"])
def test_heads_full_size(medusa, name):
    # every sequence of the workload against the oracle
    c = W.WORKLOADS[name]
    x = W.heads_inputs(seed=c["seed"], B=c["B"], H=c["H"], V=c["V"], K=c["K"], dtype=c["dtype"])
    idx, val, lg = _run(medusa, x, c["topk"])
    rows = list(range(c["B"]))
    ref = _oracle_rows(x, rows, c["dtype"])
    assert np.abs(lg - ref).max() <= 2e-2
    ridx, rval = O.topk(ref, c["topk"])
    assert topk_near_tie_ok(idx, ridx, ref) == 0
    assert np.abs(val - rval).max() <= 2e-2


def test_heads_batch64_full_size(medusa):
    # Vicuna-7B-shaped heads at batch 64 (the top of the batch sweep); the oracle
    # checks 16 sequences spread over the batch (every tcgen05 accumulator
    # column group is met)
    x = W.heads_inputs(seed=64, B=64, H=4096, V=32000, K=5, dtype="bf16")
    idx, val, lg = _run(medusa, x, 8)
    rows = list(range(0, 64, 4))
    ref = _oracle_rows(x, rows, "bf16")
    assert np.abs(lg[rows] - ref).max() <= 2e-2
    ridx, _ = O.topk(ref, 8)
    topk_near_tie_ok(idx[rows], ridx, ref)


def test_wide_batch_limits(medusa):
    # batches above 8 exist only for bf16 with H % 128 == 0, up to 64
    for B, H, dt in ((9, 256, "f32"), (65, 256, "bf16"), (16, 264, "bf16")):
        x = W.heads_inputs(seed=5, B=B, H=H, V=300, K=2, dtype=dt)
        with pytest.raises(medusa.MedusaError) as e:
            medusa.heads_topk(to_dev(x["h"]), to_dev(x["w1"]), to_dev(x["b1"]), to_dev(x["w2"]), 4)
        assert e.value.code == -2


def test_workspace_and_alignment_errors(medusa):
    x = W.heads_inputs(seed=3, B=1, H=256, V=1000, K=3, dtype="f32")
    args = [to_dev(x[n]) for n in ("h", "w1", "b1", "w2")]
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(medusa.MedusaError) as e:
        medusa.heads_topk(*args, 3, ws=small)
    assert e.value.code == -3
    w2 = torch.empty(args[3].numel() + 1, dtype=torch.float32, device="cuda")[1:].view_as(args[3])
    with pytest.raises(medusa.MedusaError) as e:
        medusa.heads_topk(args[0], args[1], args[2], w2, 3)
    assert e.value.code == -1
