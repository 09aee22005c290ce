"""medusa_heads_topk_static: the heads entry point for callers that cannot call
cudaMalloc (an operator inside a host engine that owns all device memory and
gives its operators no workspace, or a process whose device memory is fully
reserved by a pool).  It takes its scratch from the library's own fixed device
array.  Its results must equal those of medusa_heads_topk with a caller
workspace, call after call, whatever the previous call left in the array.

The file name sorts last so that a run stopping at its first failure has run
every other test before this one."""
import ctypes as C

import numpy as np
import pytest
import torch

import workloads as W
from util import to_dev, to_np

pytestmark = pytest.mark.gpu


def _static_call(M, dev, topk):
    """Direct C-ABI call of medusa_heads_topk_static; returns (rc, idx, val, logits)."""
    h, w1, b1, w2 = dev
    B, H = h.shape
    K, V = w2.shape[0], w2.shape[1]
    idx = torch.full((B, K, topk), -7, dtype=torch.int32, device="cuda")
    val = torch.full((B, K, topk), float("nan"), dtype=torch.float32, device="cuda")
    lg = torch.full((B, K, V), float("nan"), dtype=torch.float32, device="cuda")
    dt = 1 if h.dtype == torch.bfloat16 else 0
    p = lambda t: C.c_void_p(t.data_ptr())
    rc = M.lib().medusa_heads_topk_static(p(h), p(w1), p(b1), p(w2), dt, B, K, H, V, topk, p(idx),
                                          p(val), p(lg),
                                          C.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return rc, to_np(idx), to_np(val), to_np(lg)


@pytest.mark.parametrize("cases", [
    # two calls in a row with different shapes and inputs
    [dict(seed=1, B=1, H=4096, V=32000, K=5, topk=8, dtype="bf16", tol=2e-2),
     dict(seed=2, B=3, H=512, V=3001, K=4, topk=5, dtype="bf16", tol=2e-2)],
    [dict(seed=3, B=1, H=256, V=1000, K=3, topk=3, dtype="f32", tol=1e-5),
     dict(seed=4, B=1, H=256, V=1000, K=3, topk=3, dtype="f32", tol=1e-5)],
])
def test_static_scratch_matches_workspace_entry(medusa, cases):
    for c in cases:
        x = W.heads_inputs(c["seed"], c["B"], c["H"], c["V"], c["K"], c["dtype"], b1_std=0.3)
        dev = [to_dev(x[n]) for n in ("h", "w1", "b1", "w2")]
        rc, idx, val, lg = _static_call(medusa, dev, c["topk"])
        assert rc == 0, medusa.lib().medusa_last_error()
        ridx, rval, rlg = medusa.heads_topk(*dev, c["topk"], want_logits=True)
        torch.cuda.synchronize()
        assert np.array_equal(idx, to_np(ridx))
        assert np.abs(val - to_np(rval)).max() <= c["tol"]
        assert np.abs(lg - to_np(rlg)).max() <= c["tol"]


def test_static_scratch_rejects_shapes_beyond_its_maximum(medusa):
    # B=8, K=64, H=4096 needs far more than the 4 MiB maximum (25 MB of z planes
    # on the tensor cores, 8 MiB of float32 z on CUDA cores): refused, nothing
    # launched
    L = medusa.lib()
    rc = L.medusa_heads_topk_static(None, None, None, None, 1, 8, 64, 4096, 32000, 8, None, None,
                                    None, None)
    assert rc == -2
    assert b"static" in L.medusa_last_error()
