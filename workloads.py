"""Seeded synthetic inputs for the Medusa decode step.

This module is the one piece shared by the CUDA library's tests and bench and by
the CPU oracle's tests.  It only draws random numbers and lays them out: it holds
none of the method's arithmetic (no heads, no tree building, no attention, no
acceptance).  Inputs that depend on the method's own results (the verifier logits
are planted around the candidate tokens) take those results as arguments.

Every array comes from ``numpy.random.default_rng([seed, stream_id])`` with a
named stream, so each tensor can be regenerated on its own.  Normal draws are
made in float32; bf16 tensors are the float32 draws rounded to nearest-even and
are returned as their raw ``uint16`` bit patterns.

Shapes follow the five workloads of the method's pages (Medusa heads glossary,
"How heads predict later tokens" and "Tree attention and acceptance"; the
speculative-decoding e-book page, "Faster without changing the result"):

1. tiny fp32 step: hidden 256, vocab 1000, 3 heads, top-2 x top-3 tree;
2. Vicuna-7B-shaped bf16 step at batch 1: hidden 4096, vocab 32000, 5 heads,
   64-node sparse tree, 32 heads x 128 head dim, KV 2048;
3. 13B-shaped bf16 step at batch 8: hidden 5120, 40 heads, ragged KV in
   [1024, 4096];
4. dense (4x4x4x4, 341 nodes) and sparse trees at batch 4, KV 8192, verifier
   logits ~N(0, 3), typical acceptance;
5. speculative-sampling chains, batch 64, vocab 128256.
"""
from __future__ import annotations

import numpy as np

STREAMS = {
    "H": 1, "W1": 2, "B1": 3, "W2": 4, "LMHEAD": 5, "Q": 6, "K": 7, "V": 8,
    "HIDTREE": 9, "LOGITS": 10, "PLANT": 11, "KVLEN": 12, "ROOT": 13,
    "QL": 14, "NOISE": 15, "DRAFT": 16, "TOPK": 17,
}

# name -> shape and dtype of the five workloads.
# The workloads, named by shape; each draws its inputs from its own seed.
WORKLOADS = {
    "tiny_h256_v1000_f32": dict(seed=1, dtype="f32", B=1, H=256, V=1000, K=3, topk=3,
            tree="product", tree_ranks=(2, 3), Hq=4, Hkv=4, D=64,
            L_lo=128, L_hi=128, accept="greedy", alpha=0.8, w_std=0.02),
    "h4096_b1_sparse64": dict(seed=2, dtype="bf16", B=1, H=4096, V=32000, K=5, topk=8,
            tree="sparse64", Hq=32, Hkv=32, D=128, L_lo=2048, L_hi=2048,
            accept="greedy", alpha=0.8, w_std=0.02),
    "h5120_b8_ragged": dict(seed=3, dtype="bf16", B=8, H=5120, V=32000, K=5, topk=8,
            tree="sparse64", Hq=40, Hkv=40, D=128, L_lo=1024, L_hi=4096,
            accept="greedy", alpha=0.8, w_std=0.02),
    "h4096_b4_kv8192": dict(seed=4, dtype="bf16", B=4, H=4096, V=32000, K=5,
            topk=8, tree="dense", tree_ranks=(4, 4, 4, 4), Hq=32, Hkv=32, D=128,
            L_lo=8192, L_hi=8192, accept="typical", logit_std=3.0, w_std=0.02),
    "chain_b64_v128256": dict(seed=5, dtype="f32", B=64, V=128256, sigmas=(0.1, 0.5, 1.0),
            gamma_max=32, ql_std=2.0),
}


def rng(seed: int, stream: str) -> np.random.Generator:
    return np.random.default_rng([int(seed), STREAMS[stream]])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); return the uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (for building fixtures)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal(seed: int, stream: str, shape, std: float = 1.0, dtype: str = "f32",
           chunk: int = 1 << 24) -> np.ndarray:
    """N(0, std) draws of ``shape`` in float32, or bf16 bits when dtype == 'bf16'.

    Large tensors are drawn in chunks from one stream, so the result does not
    depend on the chunk size of the caller.
    """
    g = rng(seed, stream)
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32 if dtype == "f32" else np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        v = g.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        out[s:e] = v if dtype == "f32" else f32_to_bf16_bits(v)
    return out.reshape(shape)


# ----------------------------------------------------------------------------
# heads
# ----------------------------------------------------------------------------
def heads_inputs(seed: int, B: int, H: int, V: int, K: int, dtype: str,
                 w_std: float = 0.02, zero_init: bool = False, b1_std: float = 0.0) -> dict:
    """h [B,H], W1 [K,H,H] (row = output), b1 [K,H], W2 [K,V,H], lm_head [V,H].

    With ``zero_init`` W1 = b1 = 0 and every W2_k is a copy of lm_head, the
    initial state of the heads described on the Medusa heads page.
    """
    h = normal(seed, "H", (B, H), 1.0, dtype)
    lm = normal(seed, "LMHEAD", (V, H), w_std, dtype)
    if zero_init:
        zdt = np.float32 if dtype == "f32" else np.uint16
        w1 = np.zeros((K, H, H), dtype=zdt)
        b1 = np.zeros((K, H), dtype=zdt)
        w2 = np.ascontiguousarray(np.broadcast_to(lm, (K, V, H)))
    else:
        w1 = normal(seed, "W1", (K, H, H), w_std, dtype)
        if b1_std > 0:
            b1 = normal(seed, "B1", (K, H), b1_std, dtype)
        else:
            b1 = np.zeros((K, H), dtype=np.float32 if dtype == "f32" else np.uint16)
        w2 = normal(seed, "W2", (K, V, H), w_std, dtype)
    return dict(h=h, w1=w1, b1=b1, w2=w2, lm_head=lm)


def random_topk_lists(seed: int, B: int, K: int, topk: int, V: int) -> np.ndarray:
    """Synthetic per-head top-k token lists [B,K,topk]: distinct tokens per list."""
    g = rng(seed, "TOPK")
    out = np.empty((B, K, topk), dtype=np.int32)
    for b in range(B):
        for k in range(K):
            out[b, k] = g.choice(V, size=topk, replace=False)
    return out


def root_tokens(seed: int, B: int, V: int) -> np.ndarray:
    return rng(seed, "ROOT").integers(0, V, size=B, dtype=np.int32)


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------
def kv_lengths(seed: int, B: int, lo: int, hi: int) -> np.ndarray:
    """Prefix KV lengths L_b, uniform integers in [lo, hi]."""
    if lo == hi:
        return np.full(B, lo, dtype=np.int32)
    return rng(seed, "KVLEN").integers(lo, hi + 1, size=B, dtype=np.int32)


def attention_inputs(seed: int, B: int, N: int, Hq: int, Hkv: int, D: int,
                     Lmax: int, dtype: str) -> dict:
    """q [B,N,Hq,D]; K and V caches [B,Hkv,Lmax,D], all N(0,1).

    The caches are filled over their whole capacity, so the tree keys at slots
    [L_b, L_b + N) are already present whatever L_b is.
    """
    q = normal(seed, "Q", (B, N, Hq, D), 1.0, dtype)
    k = normal(seed, "K", (B, Hkv, Lmax, D), 1.0, dtype)
    v = normal(seed, "V", (B, Hkv, Lmax, D), 1.0, dtype)
    return dict(q=q, k_cache=k, v_cache=v)


def hidden_tree(seed: int, B: int, N: int, H: int, dtype: str) -> np.ndarray:
    return normal(seed, "HIDTREE", (B, N, H), 1.0, dtype)


# ----------------------------------------------------------------------------
# verifier logits
# ----------------------------------------------------------------------------
def planted_logits(seed: int, cand: np.ndarray, parent: np.ndarray, V: int,
                   alpha: float) -> np.ndarray:
    """Verifier logits [B,N,V] fp32 with planted argmaxes.

    Rows are N(0,1).  For each sequence and each node u that has children, a
    Bernoulli(alpha) draw decides the row's target token: on success the token
    of u's lowest-index child, otherwise the smallest token id that is none of
    u's children's tokens.  The target is then set to max(row) + 1, so it is the
    unique argmax.  Rows of leaves are left as drawn.
    """
    cand = np.asarray(cand, dtype=np.int32)
    parent = np.asarray(parent, dtype=np.int32)
    B, N = cand.shape
    logits = normal(seed, "LOGITS", (B, N, V), 1.0, "f32")
    g = rng(seed, "PLANT")
    children = [[] for _ in range(N)]
    for j in range(1, N):
        children[parent[j]].append(j)
    for b in range(B):
        for u in range(N):
            if not children[u]:
                continue
            hit = g.random() < alpha
            toks = {int(cand[b, j]) for j in children[u]}
            if hit:
                target = int(cand[b, min(children[u])])
            else:
                target = 0
                while target in toks:
                    target += 1
            row = logits[b, u]
            row[target] = row.max() + np.float32(1.0)
    return logits


def normal_logits(seed: int, B: int, N: int, V: int, std: float) -> np.ndarray:
    return normal(seed, "LOGITS", (B, N, V), std, "f32")


# ----------------------------------------------------------------------------
# speculative-sampling chains
# ----------------------------------------------------------------------------
def chain_inputs(seed: int, B: int, gamma: int, V: int, sigma: float,
                 ql_std: float = 2.0) -> dict:
    """Target p [B,gamma+1,V], draft q [B,gamma,V] (fp32) and drafts [B,gamma].

    Per row: ql ~ N(0, ql_std), q = softmax(ql), p = softmax(ql + N(0, sigma));
    row gamma of p (the bonus position) has its own ql.  Draft token i of a
    sequence is drawn from q_i by inverse CDF with a float64 uniform.
    """
    gq = rng(seed, "QL")
    gn = rng(seed, "NOISE")
    gd = rng(seed, "DRAFT")
    p = np.empty((B, gamma + 1, V), dtype=np.float32)
    q = np.empty((B, max(gamma, 0), V), dtype=np.float32)
    draft = np.empty((B, max(gamma, 0)), dtype=np.int32)
    for b in range(B):
        ql = gq.standard_normal((gamma + 1, V), dtype=np.float32) * np.float32(ql_std)
        noise = gn.standard_normal((gamma + 1, V), dtype=np.float32) * np.float32(sigma)
        for pos in range(gamma + 1):
            x = ql[pos].astype(np.float64)
            e = np.exp(x - x.max())
            qq = e / e.sum()
            y = x + noise[pos].astype(np.float64)
            e2 = np.exp(y - y.max())
            p[b, pos] = (e2 / e2.sum()).astype(np.float32)
            if pos < gamma:
                q[b, pos] = qq.astype(np.float32)
                c = np.cumsum(q[b, pos].astype(np.float64))
                u = gd.random() * c[-1]
                draft[b, pos] = min(int(np.searchsorted(c, u, side="right")), V - 1)
    return dict(p=p, q=q, draft=draft)
