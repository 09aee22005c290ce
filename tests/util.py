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
