"""Helpers shared by the tests: numpy <-> torch transfers and tolerance checks."""
import numpy as np


def to_dev(a, device="cuda"):
    """numpy array -> torch tensor on device; uint16 arrays are bf16 bit patterns,
    uint64 arrays (tree masks) become int64 with the same bits."""
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    elif a.dtype == np.uint64:
        t = torch.from_numpy(a.view(np.int64))
    else:
        t = torch.from_numpy(a)
    return t.to(device)


def to_np(t):
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def topk_near_tie_ok(gpu_idx, ref_idx, ref_logits, band=1e-5):
    """GPU top-k indices equal the oracle's, except where the oracle's float64
    logits of the swapped tokens lie within `band` * max(1, |logit|) of each
    other (a near tie that float32 accumulation may order either way).
    Returns the number of tolerated near-tie positions; raises on a real mismatch."""
    gpu_idx = np.asarray(gpu_idx).reshape(-1, gpu_idx.shape[-1])
    ref_idx = np.asarray(ref_idx).reshape(-1, ref_idx.shape[-1])
    lg = np.asarray(ref_logits).reshape(-1, ref_logits.shape[-1])
    ties = 0
    for r in range(gpu_idx.shape[0]):
        if np.array_equal(gpu_idx[r], ref_idx[r]):
            continue
        k = gpu_idx.shape[1]
        vals_g = lg[r, gpu_idx[r]]
        vals_o = lg[r, ref_idx[r]]
        # same multiset of values up to the band, position by position
        scale = np.maximum(1.0, np.abs(vals_o))
        if not np.all(np.abs(vals_g - vals_o) <= band * scale):
            raise AssertionError(f"row {r}: gpu {gpu_idx[r].tolist()} vs oracle {ref_idx[r].tolist()}")
        ties += int(np.sum(gpu_idx[r] != ref_idx[r]))
        assert len(set(gpu_idx[r].tolist())) == k
    return ties


# ----------------------------------------------------------------------------
# oracle calls on independent units, spread over the host's cores (ctypes
# releases the interpreter lock while the C oracle runs)
def pool_map(fn, items):
    import concurrent.futures as cf
    import os
    items = list(items)
    n = max(1, min(len(items), len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                   else (os.cpu_count() or 1)))
    with cf.ThreadPoolExecutor(max_workers=n) as ex:
        return list(ex.map(fn, items))


# ----------------------------------------------------------------------------
# Typical acceptance where float32 and float64 may decide differently.
#
# The GPU decides P(cand) > tau in float32; the oracle in float64.  The
# relative difference of the two sides' P / tau is bounded by TYPICAL_BAND,
# which tests/test_parity_verify.py::test_typical_decision_error_is_within_band
# measures through the C ABI (the measured maximum must stay below half of it;
# on a GB300 it measured at most 2.7e-6 over 2048 rows of vocab 32000 at
# temperatures 1 and 0.7, in steps of 1e-6).
# A node whose oracle P(cand) lies within that band of its parent's tau is
# ambiguous: either decision is correct there.  Every other decision must
# match, so the GPU's outputs must equal the oracle's outputs under one of the
# resolutions of the ambiguous decisions.
TYPICAL_BAND = 1e-5


def typical_outcomes(ref, b, parent, depth, band=TYPICAL_BAND, max_amb=10):
    """All (accept_len, best_node, path_nodes, next_tok) that sequence b may
    produce: the oracle's pass decisions, with each ambiguous node (|P - tau| <=
    band * tau) taken both ways.  next_tok is the oracle's argmax of the best
    node's row.  Returns (outcomes, number of ambiguous nodes)."""
    import itertools
    N = len(parent)
    Dmax = ref["path_nodes"].shape[1] - 1
    tau = ref["tau"][b]
    pc = ref["pcand"][b]
    passes = np.zeros(N, bool)
    amb = []
    for j in range(1, N):
        t = tau[parent[j]]
        passes[j] = pc[j] > t
        if abs(pc[j] - t) <= band * t:
            amb.append(j)
    assert len(amb) <= max_amb, f"sequence {b}: {len(amb)} ambiguous nodes"
    outs = set()
    for flips in itertools.product((False, True), repeat=len(amb)):
        p = passes.copy()
        for j, f in zip(amb, flips):
            if f:
                p[j] = not p[j]
        acc = np.zeros(N, bool)
        acc[0] = True
        for j in range(1, N):  # parents precede children
            acc[j] = acc[parent[j]] and p[j]
        best = max((int(depth[j]), -j) for j in range(N) if acc[j])
        best = -best[1]
        path = [-1] * (Dmax + 1)
        u = best
        while u >= 0:
            path[depth[u]] = u
            u = parent[u] if u > 0 else -1
        outs.add((int(depth[best]), best, tuple(path), int(ref["argmax"][b, best])))
    return outs, len(amb)


def check_typical(got, ref, parent, depth, band=TYPICAL_BAND, next_tok=True):
    """Every sequence's GPU outputs equal one of its allowed outcomes.  Returns
    the number of ambiguous nodes met (usually 0)."""
    n_amb = 0
    for b in range(len(ref["accept_len"])):
        outs, na = typical_outcomes(ref, b, parent, depth, band)
        n_amb += na
        g = (int(got["accept_len"][b]), int(got["best_node"][b]), tuple(int(x) for x in got["path_nodes"][b]),
             int(got["next_tok"][b]))
        if not next_tok:
            g = g[:3]
            outs = {o[:3] for o in outs}
        assert g in outs, (b, g, sorted(outs))
    return n_amb


# ----------------------------------------------------------------------------
# The exponential race of the header's random-number contract, vectorised
# (SplitMix64 of Steele, Lea and Flood; entry 2m uses bits 40..63 and entry
# 2m+1 bits 16..39 of next(key, m + 1)).  Used where the GPU's best node differs
# from the oracle's at an ambiguous decision, to know the token the GPU must
# draw from its own best row.
_G = np.uint64(0x9E3779B97F4A7C15)


def _mix(z):
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def race_uniforms(key, V):
    with np.errstate(over="ignore"):
        m = np.arange((V + 1) // 2, dtype=np.uint64) + np.uint64(1)
        h = _mix(np.uint64(key) + m * _G)
    u = np.empty(2 * len(m), np.float64)
    u[0::2] = (h >> np.uint64(40)).astype(np.float64)
    u[1::2] = ((h >> np.uint64(16)) & np.uint64(0xFFFFFF)).astype(np.float64)
    return (u[:V] + 1.0) / 2.0 ** 24


def race_draw(w, key):
    """argmin over w_v > 0 of -ln U+_v / w_v (lowest v on ties), and the relative
    gap between the two best keys."""
    u = race_uniforms(key, len(w))
    with np.errstate(divide="ignore"):
        keys = np.where(w > 0, -np.log(u) / np.where(w > 0, w, 1.0), np.inf)
    order = np.argsort(keys, kind="stable")
    k1, k2 = keys[order[0]], keys[order[1]] if len(w) > 1 else np.inf
    return int(order[0]), (k2 - k1) / k1 if k1 > 0 else np.inf


# Relative error bound of the GPU's race keys for a sampled next token at
# temperature T: w_v = exp(x_v - m) with x = logit * (1/T) in float32 (argument
# error 2u|x| + 2u|m| when T != 1 from rounding 1/T and the product, plus u|x - m|
# for the subtraction), expf within 2 ulp (4u), -logf(U) within 1 ulp (2u), one
# rounding per cross-multiplied product (u); two keys are compared, so the sum
# of both keys' bounds.  u = 2^-24.  (Speculative-decoding e-book page, "Faster
# without changing the result": the draw follows the target distribution.)
def tree_race_band(row, T):
    u = 2.0 ** -24
    x = np.asarray(row, np.float64) / T
    m = x.max()
    ax = np.abs(x).max()
    arg = (2 * ax + 2 * abs(m)) if T != 1.0 else 0.0
    return 2 * u * (arg + (m - x.min()) + 4 + 2 + 1)


# Chain races draw from w = max(0, p - q) (one float32 rounding, u, against the
# oracle's exact double difference) or w = p (exact): per key u + 2u (logf) + u
# (product), two keys: 8u = 4.8e-7, so a band of 1e-6 holds with room.
CHAIN_RACE_BAND = 1e-6


def oracle_attention_all(q, k_cache, v_cache, kv_len, mask, dtype, scale):
    """The oracle's attention output [B,N,Hq,D] for every row, computed as row
    lists spread over the host's cores."""
    from oracle import oracle as O
    B, N, Hq, D = q.shape
    b, n, h = np.meshgrid(np.arange(B), np.arange(N), np.arange(Hq), indexing="ij")
    rows = np.stack([b.ravel(), n.ravel(), h.ravel()], 1).astype(np.int32)
    parts = pool_map(lambda r: O.tree_attention(q, k_cache, v_cache, kv_len, mask, dtype, scale, rows=r),
                     np.array_split(rows, 64))
    return np.concatenate(parts, 0).reshape(B, N, Hq, D)
