"""The random-number contract that include/medusa.h states for speculative-
sampling acceptance (4b) and the sampled next token of typical acceptance
(4b'), implemented here in pure Python from that text alone, must reproduce the
oracle's draws token for token.  A caller who follows the header can then
replay any draw of the library (e-book page "Giai ma dau co", "Faster without
changing the result"; SplitMix64 of Steele, Lea and Flood, 2014)."""
import math

import numpy as np

import workloads as W
from oracle import oracle as O

MASK64 = (1 << 64) - 1
GOLDEN_GAMMA = 0x9E3779B97F4A7C15


def mix(z):
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def next_(s, n):  # the n-th output from state s
    return mix((s + n * GOLDEN_GAMMA) & MASK64)


def key(seed, stream, b, rnd, pos):
    f = lambda x: next_(x, 1)
    return f(f(f(f(f(seed) ^ stream) ^ b) ^ rnd) ^ pos)


def u_plus(k, v):  # entry 2m: bits 40..63, entry 2m+1: bits 16..39 of next(key, m + 1)
    h = next_(k, v // 2 + 1)
    bits = (h >> 16) & 0xFFFFFF if v & 1 else h >> 40
    return (bits + 1) / 2.0 ** 24


def race(w, p_fallback, k):
    best, bk = -1, math.inf
    for v, wv in enumerate(w):
        if wv > 0:
            kv = -math.log(u_plus(k, v)) / wv
            if kv < bk:
                best, bk = v, kv
    if best < 0:  # lowest v holding the largest p
        best = int(np.argmax(p_fallback))
    return best


def chain_from_header(p, q, draft, seed, rnd):
    B, g1, V = p.shape
    gamma = g1 - 1
    n_acc = np.zeros(B, np.int32)
    out = np.full((B, gamma + 1), -1, np.int32)
    for b in range(B):
        k = 0
        for i in range(1, gamma + 1):
            x = int(draft[b, i - 1])
            u = (next_(key(seed, 1, b, rnd, i), 1) >> 40) / 2.0 ** 24
            if u * float(q[b, i - 1, x]) < float(p[b, i - 1, x]):
                out[b, k] = x
                k += 1
                continue
            w = [max(0.0, float(pv) - float(qv)) for pv, qv in zip(p[b, i - 1], q[b, i - 1])]
            out[b, k] = race(w, p[b, i - 1], key(seed, 2, b, rnd, i))
            break
        else:
            out[b, gamma] = race([max(0.0, float(x)) for x in p[b, gamma]], p[b, gamma],
                                 key(seed, 3, b, rnd, gamma + 1))
        n_acc[b] = k
    return n_acc, out


def test_splitmix64_matches_oracle():
    for s in (0, 1, 1234567, MASK64):
        for n in (1, 2, 77):
            assert next_(s, n) == O.splitmix64(s, n)
    assert key(9, 2, 3, 4, 5) == O.row_key(9, 2, 3, 4, 5)


def test_chain_draws_from_the_header_text_match_the_oracle():
    rng = np.random.default_rng(5)
    for gamma, V in ((0, 11), (1, 9), (3, 13), (6, 7)):
        B = 12
        ql = rng.normal(0, 2, size=(B, gamma + 1, V))
        p = np.exp(ql + rng.normal(0, 0.7, size=ql.shape))
        p = (p / p.sum(-1, keepdims=True)).astype(np.float32)
        q = np.exp(ql[:, :gamma])
        q = (q / q.sum(-1, keepdims=True)).astype(np.float32) if gamma else np.zeros((B, 0, V), np.float32)
        draft = rng.integers(0, V, size=(B, gamma)).astype(np.int32)
        for rnd in range(3):
            n_acc, toks = chain_from_header(p, q, draft, 77, rnd)
            ref = O.verify_chain(p, q, draft, 77, rnd)
            assert np.array_equal(n_acc, ref["n_acc"])
            assert np.array_equal(toks, ref["out_tok"])


def test_sampled_next_token_from_the_header_text_matches_the_oracle():
    # 4b': the best node's row, w_v = exp(row_v / T - max / T), key stream 4 pos 0
    t = O.tree_layout(O.product_tree_paths((2, 3)), 2)
    B, V, T = 5, 23, 0.8
    cand = O.build_tree(W.random_topk_lists(8, B, 3, 3, V), W.root_tokens(8, B, V), t["depth"], t["rank"])
    logits = W.normal_logits(8, B, t["N"], V, 3.0)
    for rnd in range(3):
        ref = O.verify_tree_sample(logits, cand, t["parent"], t["depth"], t["max_depth"], 41, rnd, T)
        for b in range(B):
            row = logits[b, ref["best_node"][b]].astype(np.float64) / T
            w = np.exp(row - row.max())
            assert race(w, row, key(41, 4, b, rnd, 0)) == ref["next_tok"][b]
