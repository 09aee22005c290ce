"""ctypes wrapper of the C oracle -- TEST INFRASTRUCTURE ONLY.

Each function takes and returns numpy arrays and calls the float64 C routine of
the same name in medusa_oracle.c.  bf16 tensors are passed as their uint16 bit
patterns with dtype="bf16".
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        P = C.c_void_p
        i32, u64, dbl = C.c_int, C.c_uint64, C.c_double
        L.oracle_heads_logits.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P, P]
        L.oracle_lm_head_logits.argtypes = [P, P, i32, i32, i32, i32, P]
        L.oracle_topk.argtypes = [P, i32, i32, P, P]
        L.oracle_tree_layout.argtypes = [P, i32, i32, i32, i32, P, P, P, P, P, P, P, P]
        L.oracle_sparse_tree_paths.argtypes = [i32, i32, i32, dbl, dbl, P]
        L.oracle_build_tree.argtypes = [P, P, P, P, i32, i32, i32, i32, P]
        L.oracle_tree_attention.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                            dbl, P, i32, P]
        L.oracle_verify_tree.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, dbl, dbl, dbl,
                                         P, P, P, P, P, P, P, P]
        L.oracle_verify_chain.argtypes = [P, P, P, i32, i32, i32, u64, u64, P, P, P]
        L.oracle_verify_tree_sample.argtypes = [P, P, P, P, i32, i32, i32, i32, dbl, dbl, dbl, u64, u64,
                                                P, P, P, P, P]
        L.oracle_kv_compact.argtypes = [P, P, i32, P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                        i32, i32, P]
        L.oracle_splitmix64.argtypes = [u64, u64]
        L.oracle_splitmix64.restype = u64
        L.oracle_row_key.argtypes = [u64, u64, u64, u64, u64]
        L.oracle_row_key.restype = u64
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _dt(dtype: str) -> int:
    return {"f32": 0, "bf16": 1}[dtype]


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with status {rc}")


def _wdt(dtype):
    return np.float32 if dtype == "f32" else np.uint16


# ----------------------------------------------------------------------------
def heads_logits(h, w1, b1, w2, dtype, return_z=False):
    """Medusa head logits [B,K,V] in float64 (and z [B,K,H] if asked)."""
    wd = _wdt(dtype)
    h, w1, b1, w2 = (_c(x, wd) for x in (h, w1, b1, w2))
    B, H = h.shape
    K, V = w2.shape[0], w2.shape[1]
    out = np.zeros((B, K, V), dtype=np.float64)
    z = np.zeros((B, K, H), dtype=np.float64) if return_z else None
    _check(lib().oracle_heads_logits(_p(h), _p(w1), _p(b1), _p(w2), _dt(dtype), B, K, H, V,
                                     _p(z), _p(out)), "heads_logits")
    return (out, z) if return_z else out


def lm_head_logits(h, lm, dtype):
    wd = _wdt(dtype)
    h, lm = _c(h, wd), _c(lm, wd)
    B, H = h.shape
    V = lm.shape[0]
    out = np.zeros((B, V), dtype=np.float64)
    _check(lib().oracle_lm_head_logits(_p(h), _p(lm), _dt(dtype), B, H, V, _p(out)), "lm_head")
    return out


def lm_head_logits_matmul(h, lm, dtype):
    """lm_head . h for many rows at once: the same definition as lm_head_logits
    (bf16 decoded exactly, float64 arithmetic), with one float64 matrix product
    of the library (numpy) as the step, for row counts the C loop would take
    minutes over (e.g. 1364 tree rows x vocab 32000 x hidden 4096)."""
    def dec(a):
        if dtype == "f32":
            return np.asarray(a, np.float32).astype(np.float64)
        return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return dec(h) @ dec(lm).T


def topk(x, k):
    """Top-k of each row of x (float64): (idx int32, val float64), sorted."""
    x = _c(x, np.float64)
    shp = x.shape[:-1]
    n = x.shape[-1]
    rows = x.reshape(-1, n)
    idx = np.zeros((rows.shape[0], k), dtype=np.int32)
    val = np.zeros((rows.shape[0], k), dtype=np.float64)
    for r in range(rows.shape[0]):
        row = np.ascontiguousarray(rows[r])
        ii = np.zeros(k, dtype=np.int32)
        vv = np.zeros(k, dtype=np.float64)
        _check(lib().oracle_topk(_p(row), n, k, _p(ii), _p(vv)), "topk")
        idx[r], val[r] = ii, vv
    return idx.reshape(shp + (k,)), val.reshape(shp + (k,))


def heads_topk(h, w1, b1, w2, dtype, k):
    logits = heads_logits(h, w1, b1, w2, dtype)
    idx, val = topk(logits, k)
    return idx, val, logits


# ----------------------------------------------------------------------------
def tree_layout(paths, max_depth, cap_nodes=4096):
    """Node table of the candidate tree built from rank tuples (padded -1)."""
    paths = _c(paths, np.int32).reshape(-1, max_depth)
    P = paths.shape[0]
    cap_paths = cap_nodes
    parent = np.zeros(cap_nodes, np.int32)
    depth = np.zeros(cap_nodes, np.int32)
    rank = np.zeros(cap_nodes, np.int32)
    mask = np.zeros(cap_nodes * ((cap_nodes + 63) // 64), np.uint64)
    retrieve = np.zeros((cap_paths, max_depth + 1), np.int32)
    N, W, NP = C.c_int(), C.c_int(), C.c_int()
    _check(lib().oracle_tree_layout(_p(paths), P, max_depth, cap_nodes, cap_paths, _p(parent),
                                    _p(depth), _p(rank), _p(mask), _p(retrieve), C.byref(N),
                                    C.byref(W), C.byref(NP)), "tree_layout")
    n, w, npth = N.value, W.value, NP.value
    return dict(N=n, W=w, n_paths=npth, parent=parent[:n].copy(), depth=depth[:n].copy(),
                rank=rank[:n].copy(), mask=mask[: n * w].reshape(n, w).copy(),
                retrieve=retrieve[:npth].copy(), max_depth=max_depth)


def sparse_tree_paths(n_nodes, max_depth, max_rank, head_p, rank_p):
    out = np.zeros(((n_nodes - 1), max_depth), np.int32)
    _check(lib().oracle_sparse_tree_paths(n_nodes, max_depth, max_rank, head_p, rank_p, _p(out)),
           "sparse_tree_paths")
    return out


def product_tree_paths(ranks):
    """Rank tuples of the full Cartesian product of top-r_1 x ... x top-r_d."""
    grids = np.meshgrid(*[np.arange(r) for r in ranks], indexing="ij")
    return np.stack([g.reshape(-1) for g in grids], axis=1).astype(np.int32)


def build_tree(topk_idx, root_tok, depth, rank):
    topk_idx = _c(topk_idx, np.int32)
    root_tok = _c(root_tok, np.int32)
    depth, rank = _c(depth, np.int32), _c(rank, np.int32)
    B, K, k = topk_idx.shape
    N = depth.shape[0]
    cand = np.zeros((B, N), np.int32)
    _check(lib().oracle_build_tree(_p(topk_idx), _p(root_tok), _p(depth), _p(rank), B, K, k, N,
                                   _p(cand)), "build_tree")
    return cand


# ----------------------------------------------------------------------------
def tree_attention(q, k_cache, v_cache, kv_len, mask, dtype, scale, rows=None):
    """Masked attention output in float64: [B,N,Hq,D], or [n_rows,D] for a row list."""
    wd = _wdt(dtype)
    q, k_cache, v_cache = _c(q, wd), _c(k_cache, wd), _c(v_cache, wd)
    kv_len = _c(kv_len, np.int32)
    mask = _c(mask, np.uint64)
    B, N, Hq, D = q.shape
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    if rows is None:
        out = np.zeros((B, N, Hq, D), np.float64)
        nr = 0
        rp = None
    else:
        rows = _c(rows, np.int32).reshape(-1, 3)
        nr = rows.shape[0]
        out = np.zeros((nr, D), np.float64)
        rp = _p(rows)
    _check(lib().oracle_tree_attention(_p(q), _p(k_cache), _p(v_cache), _p(kv_len), _p(mask),
                                       _dt(dtype), B, N, Hq, Hkv, D, Lmax, float(scale), rp, nr,
                                       _p(out)), "tree_attention")
    return out


# ----------------------------------------------------------------------------
def verify_tree(logits, cand, parent, depth, max_depth, mode="greedy", T=1.0, eps=0.09,
                delta=0.3):
    logits = _c(logits, np.float32)
    cand, parent, depth = _c(cand, np.int32), _c(parent, np.int32), _c(depth, np.int32)
    B, N, V = logits.shape
    m = {"greedy": 0, "typical": 1}[mode]
    r = dict(accept_len=np.zeros(B, np.int32), best_node=np.zeros(B, np.int32),
             path_nodes=np.zeros((B, max_depth + 1), np.int32), next_tok=np.zeros(B, np.int32),
             argmax=np.zeros((B, N), np.int32), tau=np.zeros((B, N), np.float64),
             pcand=np.zeros((B, N), np.float64), accepted=np.zeros((B, N), np.uint8))
    _check(lib().oracle_verify_tree(_p(logits), _p(cand), _p(parent), _p(depth), B, N, V,
                                    max_depth, m, T, eps, delta, _p(r["accept_len"]),
                                    _p(r["best_node"]), _p(r["path_nodes"]), _p(r["next_tok"]),
                                    _p(r["argmax"]), _p(r["tau"]), _p(r["pcand"]),
                                    _p(r["accepted"])), "verify_tree")
    return r


def verify_chain(p, q, draft, seed, round_):
    p = _c(p, np.float32)
    B, g1, V = p.shape
    gamma = g1 - 1
    q = _c(q, np.float32) if gamma > 0 else np.zeros((B, 0, V), np.float32)
    draft = _c(draft, np.int32) if gamma > 0 else np.zeros((B, 0), np.int32)
    n_acc = np.zeros(B, np.int32)
    out = np.zeros((B, gamma + 1), np.int32)
    gap = np.zeros(B, np.float64)
    _check(lib().oracle_verify_chain(_p(p), _p(q) if gamma > 0 else None,
                                     _p(draft) if gamma > 0 else None, B, gamma, V,
                                     C.c_uint64(seed), C.c_uint64(round_), _p(n_acc), _p(out),
                                     _p(gap)), "verify_chain")
    return dict(n_acc=n_acc, out_tok=out, race_gap=gap)


def verify_tree_sample(logits, cand, parent, depth, max_depth, seed, round_, T=1.0, eps=0.09,
                       delta=0.3):
    """Typical acceptance; the next token drawn from softmax(row_best / T)."""
    logits = _c(logits, np.float32)
    cand, parent, depth = _c(cand, np.int32), _c(parent, np.int32), _c(depth, np.int32)
    B, N, V = logits.shape
    r = dict(accept_len=np.zeros(B, np.int32), best_node=np.zeros(B, np.int32),
             path_nodes=np.zeros((B, max_depth + 1), np.int32), next_tok=np.zeros(B, np.int32),
             race_gap=np.zeros(B, np.float64))
    _check(lib().oracle_verify_tree_sample(_p(logits), _p(cand), _p(parent), _p(depth), B, N, V,
                                           max_depth, T, eps, delta, C.c_uint64(seed),
                                           C.c_uint64(round_), _p(r["accept_len"]),
                                           _p(r["best_node"]), _p(r["path_nodes"]),
                                           _p(r["next_tok"]), _p(r["race_gap"])),
           "verify_tree_sample")
    return r


def splitmix64(state, n):
    return int(lib().oracle_splitmix64(C.c_uint64(state), C.c_uint64(n)))


def row_key(seed, stream, b, round_, pos):
    return int(lib().oracle_row_key(C.c_uint64(seed), C.c_uint64(stream), C.c_uint64(b),
                                    C.c_uint64(round_), C.c_uint64(pos)))


# ----------------------------------------------------------------------------
def kv_compact(k_cache, v_cache, kv_len, path_nodes, accept_len, best_node, hidden_tree, N,
               max_depth):
    """Returns new (k_cache, v_cache, kv_len, h_next, src_idx); inputs are not modified."""
    k = np.array(k_cache, copy=True, order="C")
    v = np.array(v_cache, copy=True, order="C")
    kl = np.array(kv_len, dtype=np.int32, copy=True)
    B, Hkv, Lmax, D = k.shape
    elem = k.dtype.itemsize
    H = hidden_tree.shape[-1] if hidden_tree is not None else 0
    ht = np.ascontiguousarray(hidden_tree) if hidden_tree is not None else None
    h_next = np.zeros((B, H), dtype=k.dtype) if hidden_tree is not None else None
    src = np.zeros((B, max_depth + 1), np.int32)
    _check(lib().oracle_kv_compact(_p(k), _p(v), elem, _p(kl), _p(_c(path_nodes, np.int32)),
                                   _p(_c(accept_len, np.int32)), _p(_c(best_node, np.int32)),
                                   _p(ht), _p(h_next), B, Hkv, D, Lmax, N, H, max_depth, _p(src)),
           "kv_compact")
    return k, v, kl, h_next, src
