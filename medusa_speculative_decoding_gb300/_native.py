"""ctypes loader of libmedusa_gb300.so, the library every call goes through.

There is no fallback: if the library is missing or fails to load, importing the
binding raises, so a CUDA-less or unbuilt install fails loudly instead of
computing anything elsewhere.
"""
from __future__ import annotations

import ctypes as C
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmedusa_gb300.so")

MEDUSA_F32, MEDUSA_BF16 = 0, 1
MEDUSA_ERR_TIMEOUT = -5
GREEDY, TYPICAL = 0, 1

# every symbol include/medusa.h declares
EXPORTS = (
    "medusa_last_error", "medusa_abi_version", "medusa_device_status", "medusa_set_wait_limit",
    "medusa_heads_topk_workspace", "medusa_heads_topk", "medusa_heads_topk_static",
    "medusa_sparse_tree_paths", "medusa_tree_layout", "medusa_build_tree",
    "medusa_tree_attention_workspace", "medusa_tree_attention",
    "medusa_verify_accept_workspace", "medusa_verify_accept_tree",
    "medusa_verify_project_workspace", "medusa_verify_project_tree",
    "medusa_verify_sample_workspace", "medusa_verify_accept_tree_sample",
    "medusa_verify_chain_workspace", "medusa_verify_accept_chain",
    "medusa_kv_compact",
)


class MedusaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"medusa error {code}: {msg}")
        self.code = code


_lib = None


def lib() -> C.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run medusa_speculative_decoding_gb300.build.build()")
    L = C.CDLL(LIB_PATH)
    P, i32, u64, f32, f64, sz = C.c_void_p, C.c_int, C.c_uint64, C.c_float, C.c_double, C.c_size_t
    L.medusa_last_error.restype = C.c_char_p
    L.medusa_abi_version.restype = i32
    L.medusa_device_status.argtypes = [P]
    L.medusa_set_wait_limit.argtypes = [C.c_longlong]
    L.medusa_heads_topk_workspace.argtypes = [i32] * 5
    L.medusa_heads_topk_workspace.restype = sz
    L.medusa_heads_topk.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, P, P, P, P, sz, P]
    L.medusa_heads_topk_static.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, P, P, P, P]
    L.medusa_sparse_tree_paths.argtypes = [i32, i32, i32, f64, f64, P]
    L.medusa_tree_layout.argtypes = [P, i32, i32, i32, i32, P, P, P, P, P, P, P, P]
    L.medusa_build_tree.argtypes = [P, P, P, P, i32, i32, i32, i32, P, P]
    L.medusa_tree_attention_workspace.argtypes = [i32] * 6
    L.medusa_tree_attention_workspace.restype = sz
    L.medusa_tree_attention.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, f32, P,
                                        P, sz, P]
    L.medusa_verify_accept_workspace.argtypes = [i32] * 3
    L.medusa_verify_accept_workspace.restype = sz
    L.medusa_verify_accept_tree.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, f32, f32, f32,
                                            P, P, P, P, P, sz, P]
    L.medusa_verify_project_workspace.argtypes = [i32] * 4
    L.medusa_verify_project_workspace.restype = sz
    L.medusa_verify_project_tree.argtypes = [P, P, i32, P, P, P, i32, i32, i32, i32, i32, i32, f32,
                                             f32, f32, P, P, P, P, P, sz, P]
    L.medusa_verify_sample_workspace.argtypes = [i32] * 3
    L.medusa_verify_sample_workspace.restype = sz
    L.medusa_verify_accept_tree_sample.argtypes = [P, P, P, P, i32, i32, i32, i32, f32, f32, f32, u64, u64,
                                                   P, P, P, P, P, sz, P]
    L.medusa_verify_chain_workspace.argtypes = [i32] * 3
    L.medusa_verify_chain_workspace.restype = sz
    L.medusa_verify_accept_chain.argtypes = [P, P, P, i32, i32, i32, u64, u64, P, P, P, sz, P]
    L.medusa_kv_compact.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                    P, P]
    _lib = L
    return L


def check(rc: int) -> None:
    if rc != 0:
        msg = lib().medusa_last_error().decode(errors="replace")
        raise MedusaError(rc, msg)
