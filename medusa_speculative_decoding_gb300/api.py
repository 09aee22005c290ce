"""Python binding of the C ABI (include/medusa.h) for torch tensors.

Argument marshalling only: checks device, dtype and contiguity, allocates the
outputs and workspaces with torch, and passes raw pointers plus the current CUDA
stream to libmedusa_gb300.so.  Every step of the computation runs in the
library's kernels.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from ._native import GREEDY, MEDUSA_BF16, MEDUSA_F32, TYPICAL, check, lib

_DT = {torch.float32: MEDUSA_F32, torch.bfloat16: MEDUSA_BF16}


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _need(t, name, dtype=None, cuda=True):
    if t is None:
        raise ValueError(f"{name} is required")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _dtype_of(t):
    if t.dtype not in _DT:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return _DT[t.dtype]


def _ws(nbytes, device):
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


# ----------------------------------------------------------------------------
def device_status(stream=None):
    """Synchronises the stream and raises MedusaError (code MEDUSA_ERR_TIMEOUT,
    -5) if a bounded wait of a tensor-core kernel on this device gave up since
    the previous check; returns None otherwise."""
    check(lib().medusa_device_status(_stream(stream)))


def set_wait_limit(cycles):
    """Test hook: limit (SM clock cycles) of the tensor-core kernels' first
    waits on the current device; cycles <= 0 restores the default."""
    check(lib().medusa_set_wait_limit(int(cycles)))


# ----------------------------------------------------------------------------
def heads_topk_workspace(B, K, H, V, topk):
    return int(lib().medusa_heads_topk_workspace(B, K, H, V, topk))


def heads_topk(h, w1, b1, w2, topk, want_logits=False, out=None, ws=None, stream=None):
    """Medusa heads + per-head top-k.  Returns (topk_idx [B,K,topk] int32,
    topk_val [B,K,topk] float32, logits [B,K,V] float32 or None)."""
    for n, t in (("h", h), ("w1", w1), ("b1", b1), ("w2", w2)):
        _need(t, n, h.dtype)
    B, H = h.shape
    K, V = w2.shape[0], w2.shape[1]
    dev = h.device
    if out is None:
        idx = torch.empty((B, K, topk), dtype=torch.int32, device=dev)
        val = torch.empty((B, K, topk), dtype=torch.float32, device=dev)
        lg = torch.empty((B, K, V), dtype=torch.float32, device=dev) if want_logits else None
    else:
        idx, val, lg = out
    need = heads_topk_workspace(B, K, H, V, topk)
    if ws is None:
        ws = _ws(need, dev)
    check(lib().medusa_heads_topk(_ptr(h), _ptr(w1), _ptr(b1), _ptr(w2), _dtype_of(h), B, K, H, V,
                                  topk, _ptr(idx), _ptr(val), _ptr(lg), _ptr(ws), ws.numel(),
                                  _stream(stream)))
    return idx, val, lg


HEADS_STATIC_SCRATCH_BYTES = 4 << 20


def heads_topk_static(h, w1, b1, w2, topk, want_logits=False, out=None, stream=None):
    """heads_topk without a workspace, for callers that cannot allocate device
    memory: the library's own 4 MiB device scratch array is used instead.  Calls
    share that array, so calls whose GPU work overlaps race; keep them on one
    stream."""
    for n, t in (("h", h), ("w1", w1), ("b1", b1), ("w2", w2)):
        _need(t, n, h.dtype)
    B, H = h.shape
    K, V = w2.shape[0], w2.shape[1]
    dev = h.device
    if out is None:
        idx = torch.empty((B, K, topk), dtype=torch.int32, device=dev)
        val = torch.empty((B, K, topk), dtype=torch.float32, device=dev)
        lg = torch.empty((B, K, V), dtype=torch.float32, device=dev) if want_logits else None
    else:
        idx, val, lg = out
    check(lib().medusa_heads_topk_static(_ptr(h), _ptr(w1), _ptr(b1), _ptr(w2), _dtype_of(h), B, K, H,
                                         V, topk, _ptr(idx), _ptr(val), _ptr(lg), _stream(stream)))
    return idx, val, lg


# ----------------------------------------------------------------------------
def sparse_tree_paths(n_nodes, max_depth, max_rank, head_p, rank_p):
    out = np.zeros((n_nodes - 1, max_depth), np.int32)
    check(lib().medusa_sparse_tree_paths(n_nodes, max_depth, max_rank, float(head_p), float(rank_p),
                                         out.ctypes.data_as(C.c_void_p)))
    return out


def tree_layout(paths, max_depth, cap_nodes=4096):
    """Host node table of the tree spanned by rank tuples (numpy in and out)."""
    paths = np.ascontiguousarray(paths, dtype=np.int32).reshape(-1, max_depth)
    P = paths.shape[0]
    W_cap = (cap_nodes + 63) // 64
    parent = np.zeros(cap_nodes, np.int32)
    depth = np.zeros(cap_nodes, np.int32)
    rank = np.zeros(cap_nodes, np.int32)
    mask = np.zeros(cap_nodes * W_cap, np.uint64)
    retrieve = np.zeros((cap_nodes, max_depth + 1), np.int32)
    N, W, NP = C.c_int(), C.c_int(), C.c_int()
    p = lambda a: a.ctypes.data_as(C.c_void_p)
    check(lib().medusa_tree_layout(p(paths), P, max_depth, cap_nodes, cap_nodes, p(parent),
                                   p(depth), p(rank), p(mask), p(retrieve), C.byref(N), C.byref(W),
                                   C.byref(NP)))
    n, w, npth = N.value, W.value, NP.value
    return dict(N=n, W=w, n_paths=npth, parent=parent[:n].copy(), depth=depth[:n].copy(),
                rank=rank[:n].copy(), mask=mask[: n * w].reshape(n, w).copy(),
                retrieve=retrieve[:npth].copy(), max_depth=max_depth)


def build_tree(topk_idx, root_tok, depth, rank, out=None, stream=None):
    _need(topk_idx, "topk_idx", torch.int32)
    _need(root_tok, "root_tok", torch.int32)
    _need(depth, "depth", torch.int32)
    _need(rank, "rank", torch.int32)
    B, K, k = topk_idx.shape
    N = depth.shape[0]
    cand = out if out is not None else torch.empty((B, N), dtype=torch.int32, device=topk_idx.device)
    check(lib().medusa_build_tree(_ptr(topk_idx), _ptr(root_tok), _ptr(depth), _ptr(rank), B, K, k,
                                  N, _ptr(cand), _stream(stream)))
    return cand


# ----------------------------------------------------------------------------
def tree_attention_workspace(B, N, Hq, Hkv, D, Lmax):
    return int(lib().medusa_tree_attention_workspace(B, N, Hq, Hkv, D, Lmax))


def tree_attention(q, k_cache, v_cache, kv_len, mask, scale, out=None, ws=None, stream=None):
    """Tree attention; `scale` multiplies q.k inside the softmax (the model's
    choice, usually 1/sqrt(head dim)); it is passed to the library as given."""
    _need(q, "q")
    _need(k_cache, "k_cache", q.dtype)
    _need(v_cache, "v_cache", q.dtype)
    _need(kv_len, "kv_len", torch.int32)
    _need(mask, "mask", torch.int64)
    B, N, Hq, D = q.shape
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    o = out if out is not None else torch.empty((B, N, Hq, D), dtype=torch.float32, device=q.device)
    need = tree_attention_workspace(B, N, Hq, Hkv, D, Lmax)
    if ws is None:
        ws = _ws(need, q.device)
    check(lib().medusa_tree_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len),
                                      _ptr(mask), _dtype_of(q), B, N, Hq, Hkv, D, Lmax,
                                      float(scale), _ptr(o), _ptr(ws), ws.numel(), _stream(stream)))
    return o


# ----------------------------------------------------------------------------
def verify_accept_workspace(B, N, V):
    return int(lib().medusa_verify_accept_workspace(B, N, V))


def verify_accept_tree(logits, cand, parent, depth, max_depth, mode="greedy", temperature=1.0,
                       eps=0.09, delta=0.3, out=None, ws=None, stream=None):
    _need(logits, "logits", torch.float32)
    _need(cand, "cand", torch.int32)
    _need(parent, "parent", torch.int32)
    _need(depth, "depth", torch.int32)
    B, N, V = logits.shape
    dev = logits.device
    if out is None:
        out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                   best_node=torch.empty(B, dtype=torch.int32, device=dev),
                   path_nodes=torch.empty((B, max_depth + 1), dtype=torch.int32, device=dev),
                   next_tok=torch.empty(B, dtype=torch.int32, device=dev))
    if ws is None:
        ws = _ws(verify_accept_workspace(B, N, V), dev)
    m = {"greedy": GREEDY, "typical": TYPICAL}[mode]
    check(lib().medusa_verify_accept_tree(_ptr(logits), _ptr(cand), _ptr(parent), _ptr(depth), B,
                                          N, V, max_depth, m, float(temperature), float(eps),
                                          float(delta), _ptr(out["accept_len"]),
                                          _ptr(out["best_node"]), _ptr(out["path_nodes"]),
                                          _ptr(out["next_tok"]), _ptr(ws), ws.numel(),
                                          _stream(stream)))
    return out


def verify_sample_workspace(B, N, V):
    return int(lib().medusa_verify_sample_workspace(B, N, V))


def verify_accept_tree_sample(logits, cand, parent, depth, max_depth, seed, round_, temperature=1.0,
                              eps=0.09, delta=0.3, out=None, ws=None, stream=None):
    """Typical acceptance; the next token drawn from the best node's softmax."""
    _need(logits, "logits", torch.float32)
    _need(cand, "cand", torch.int32)
    _need(parent, "parent", torch.int32)
    _need(depth, "depth", torch.int32)
    B, N, V = logits.shape
    dev = logits.device
    if out is None:
        out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                   best_node=torch.empty(B, dtype=torch.int32, device=dev),
                   path_nodes=torch.empty((B, max_depth + 1), dtype=torch.int32, device=dev),
                   next_tok=torch.empty(B, dtype=torch.int32, device=dev))
    if ws is None:
        ws = _ws(verify_sample_workspace(B, N, V), dev)
    check(lib().medusa_verify_accept_tree_sample(_ptr(logits), _ptr(cand), _ptr(parent), _ptr(depth), B, N,
                                                 V, max_depth, float(temperature), float(eps), float(delta),
                                                 C.c_uint64(seed), C.c_uint64(round_),
                                                 _ptr(out["accept_len"]), _ptr(out["best_node"]),
                                                 _ptr(out["path_nodes"]), _ptr(out["next_tok"]), _ptr(ws),
                                                 ws.numel(), _stream(stream)))
    return out


def verify_project_workspace(B, N, H, V):
    return int(lib().medusa_verify_project_workspace(B, N, H, V))


def verify_project_tree(hidden_tree, lm_head, cand, parent, depth, max_depth, mode="greedy",
                        temperature=1.0, eps=0.09, delta=0.3, out=None, ws=None, stream=None):
    """verify_accept_tree with the verifier logits defined as lm_head . hidden_tree,
    computed and reduced on the GPU without materialising them."""
    _need(hidden_tree, "hidden_tree", torch.bfloat16)
    _need(lm_head, "lm_head", torch.bfloat16)
    _need(cand, "cand", torch.int32)
    _need(parent, "parent", torch.int32)
    _need(depth, "depth", torch.int32)
    B, N, H = hidden_tree.shape
    V = lm_head.shape[0]
    dev = hidden_tree.device
    if out is None:
        out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                   best_node=torch.empty(B, dtype=torch.int32, device=dev),
                   path_nodes=torch.empty((B, max_depth + 1), dtype=torch.int32, device=dev),
                   next_tok=torch.empty(B, dtype=torch.int32, device=dev))
    if ws is None:
        ws = _ws(verify_project_workspace(B, N, H, V), dev)
    m = {"greedy": GREEDY, "typical": TYPICAL}[mode]
    check(lib().medusa_verify_project_tree(_ptr(hidden_tree), _ptr(lm_head), _dtype_of(hidden_tree),
                                           _ptr(cand), _ptr(parent), _ptr(depth), B, N, H, V,
                                           max_depth, m, float(temperature), float(eps),
                                           float(delta), _ptr(out["accept_len"]),
                                           _ptr(out["best_node"]), _ptr(out["path_nodes"]),
                                           _ptr(out["next_tok"]), _ptr(ws), ws.numel(),
                                           _stream(stream)))
    return out


def verify_chain_workspace(B, gamma, V):
    return int(lib().medusa_verify_chain_workspace(B, gamma, V))


def verify_accept_chain(p, q, draft, seed, round_, out=None, ws=None, stream=None):
    _need(p, "p", torch.float32)
    B, g1, V = p.shape
    gamma = g1 - 1
    if gamma > 0:
        _need(q, "q", torch.float32)
        _need(draft, "draft", torch.int32)
    dev = p.device
    if out is None:
        out = (torch.empty(B, dtype=torch.int32, device=dev),
               torch.empty((B, gamma + 1), dtype=torch.int32, device=dev))
    if ws is None:
        ws = _ws(verify_chain_workspace(B, gamma, V), dev)
    n_acc, out_tok = out
    check(lib().medusa_verify_accept_chain(_ptr(p), _ptr(q) if gamma > 0 else None,
                                           _ptr(draft) if gamma > 0 else None, B, gamma, V,
                                           C.c_uint64(seed), C.c_uint64(round_), _ptr(n_acc),
                                           _ptr(out_tok), _ptr(ws), ws.numel(), _stream(stream)))
    return n_acc, out_tok


# ----------------------------------------------------------------------------
def kv_compact(k_cache, v_cache, kv_len, path_nodes, accept_len, best_node, N, max_depth,
               hidden_tree=None, h_next=None, src_idx=None, stream=None):
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache", k_cache.dtype)
    _need(kv_len, "kv_len", torch.int32)
    for n, t in (("path_nodes", path_nodes), ("accept_len", accept_len), ("best_node", best_node)):
        _need(t, n, torch.int32)
    B, Hkv, Lmax, D = k_cache.shape
    H = 0
    if hidden_tree is not None:
        _need(hidden_tree, "hidden_tree", k_cache.dtype)
        H = hidden_tree.shape[-1]
        if h_next is None:
            h_next = torch.empty((B, H), dtype=k_cache.dtype, device=k_cache.device)
    if src_idx is None:
        src_idx = torch.empty((B, max_depth + 1), dtype=torch.int32, device=k_cache.device)
    check(lib().medusa_kv_compact(_ptr(k_cache), _ptr(v_cache), _ptr(kv_len), _ptr(path_nodes),
                                  _ptr(accept_len), _ptr(best_node), _ptr(hidden_tree),
                                  _ptr(h_next), _dtype_of(k_cache), B, Hkv, D, Lmax, N, H,
                                  max_depth, _ptr(src_idx), _stream(stream)))
    return h_next, src_idx
