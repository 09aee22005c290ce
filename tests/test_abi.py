"""The C-ABI library builds, loads and exports every symbol include/medusa.h
declares; host-only entry points (tree construction) agree with the oracle
bit for bit; argument errors are reported before any device work.  No test
here launches a kernel."""
import ctypes as C
import os
import re

import numpy as np
import pytest

from oracle import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def M():
    from medusa_speculative_decoding_gb300 import build
    build.build()
    import medusa_speculative_decoding_gb300 as M
    return M


def _declared():
    src = open(os.path.join(ROOT, "include", "medusa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(medusa_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(M):
    from medusa_speculative_decoding_gb300 import _native
    names = _declared()
    assert len(names) >= 14
    L = C.CDLL(_native.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n
    assert sorted(_native.EXPORTS) == names
    assert M.lib().medusa_abi_version() == 1


def test_library_has_no_oracle_dependency():
    # the product library shares nothing with the oracle: no symbol, no link
    from medusa_speculative_decoding_gb300 import _native
    data = open(_native.LIB_PATH, "rb").read()
    assert b"oracle_" not in data and b"libmedusa_oracle" not in data


@pytest.mark.parametrize("n,d,r", [(64, 5, 8), (2, 3, 3), (30, 4, 3), (100, 5, 6)])
def test_sparse_paths_match_oracle(M, n, d, r):
    assert np.array_equal(M.sparse_tree_paths(n, d, r, 0.6, 0.5), O.sparse_tree_paths(n, d, r, 0.6, 0.5))


@pytest.mark.parametrize("kind", ["c1", "dense", "sparse64", "random"])
def test_tree_layout_matches_oracle(M, kind):
    if kind == "c1":
        paths, md = O.product_tree_paths((2, 3)), 2
    elif kind == "dense":
        paths, md = O.product_tree_paths((4, 4, 4, 4)), 4
    elif kind == "sparse64":
        paths, md = O.sparse_tree_paths(64, 5, 8, 0.6, 0.5), 5
    else:
        rng = np.random.default_rng(40)
        md = 4
        paths = np.full((25, md), -1, np.int32)
        for i in range(25):
            dd = int(rng.integers(1, md + 1))
            paths[i, :dd] = rng.integers(0, 5, size=dd)
    a = M.tree_layout(paths, md)
    b = O.tree_layout(paths, md)
    for k in ("N", "W", "n_paths"):
        assert a[k] == b[k]
    for k in ("parent", "depth", "rank", "mask", "retrieve"):
        assert np.array_equal(a[k], b[k]), k


def test_layout_rejects_malformed(M):
    with pytest.raises(M.MedusaError) as e:
        M.tree_layout(np.array([[0, -1, 2]], np.int32), 3)
    assert e.value.code == -1


def test_host_side_argument_errors(M):
    L = M.lib()
    # null inputs: rejected before any device work
    rc = L.medusa_heads_topk(None, None, None, None, 1, 1, 5, 4096, 32000, 8, None, None, None,
                             None, 0, None)
    assert rc == -1 and b"null" in L.medusa_last_error()
    # unsupported shapes
    assert L.medusa_heads_topk(None, None, None, None, 1, 65, 5, 4096, 32000, 8, None, None, None,
                               None, 0, None) == -2
    assert L.medusa_heads_topk(None, None, None, None, 0, 9, 5, 4096, 32000, 8, None, None, None,
                               None, 0, None) == -2
    assert L.medusa_heads_topk(None, None, None, None, 1, 1, 5, 4095, 32000, 8, None, None, None,
                               None, 0, None) == -2
    assert L.medusa_heads_topk_workspace(1, 5, 4096, 32000, 17) == 0
    assert L.medusa_tree_attention(None, None, None, None, None, 1, 1, 64, 32, 32, 96, 2112,
                                   C.c_float(0.1), None, None, 0, None) == -2
    assert L.medusa_tree_attention(None, None, None, None, None, 1, 1, 64, 32, 32, 128, 2112,
                                   C.c_float(0.1), None, None, 0, None) == -1
    assert L.medusa_verify_accept_tree(None, None, None, None, 1, 64, 100, 4, 0, C.c_float(1),
                                       C.c_float(0), C.c_float(0), None, None, None, None, None, 0,
                                       None) == -1
    assert L.medusa_verify_accept_chain(None, None, None, 1, 2, 10, 0, 0, None, None, None, 0,
                                        None) == -1
    assert L.medusa_kv_compact(None, None, None, None, None, None, None, None, 1, 1, 1, 128, 10,
                               2, 0, 1, None, None) == -1
    assert L.medusa_build_tree(None, None, None, None, 1, 1, 1, 1, None, None) == -1
    f0 = C.c_float(0)
    assert L.medusa_verify_project_tree(None, None, 1, None, None, None, 1, 64, 4096, 32000, 4, 0,
                                        C.c_float(1), f0, f0, None, None, None, None, None, 0,
                                        None) == -1
    assert L.medusa_verify_project_workspace(1, 64, 4100, 32000) == 0   # H % 8 != 0
    assert L.medusa_verify_project_workspace(1, 513, 4096, 32000) == 0  # N above 512


def test_product_path_has_no_cpu_fallback():
    # the binding refuses to run without the CUDA library instead of computing elsewhere
    from medusa_speculative_decoding_gb300 import api
    src = open(api.__file__).read()
    assert "oracle" not in src and "numpy.linalg" not in src


def test_device_status_calls_report_a_missing_device(M):
    # medusa_device_status / medusa_set_wait_limit touch the device; without one
    # they return MEDUSA_ERR_CUDA with a message instead of crashing
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present: tests/test_parity_timeout.py covers these calls")
    L = M.lib()
    assert L.medusa_device_status(None) == -4
    assert L.medusa_last_error()
    assert L.medusa_set_wait_limit(5) == -4
