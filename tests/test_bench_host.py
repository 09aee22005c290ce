"""Host-side helpers of bench.py that run without a GPU: the packed transfer
buffers of the end-to-end loop and the algorithmic byte counts behind the
roofline figures."""
import numpy as np
import torch

import bench
import workloads as W


def test_pack_keeps_contents_shapes_and_alignment():
    ts = [torch.arange(7, dtype=torch.int32), torch.randn(3, 5).to(torch.bfloat16),
          torch.randn(2, 3, 4), torch.tensor([1, 2], dtype=torch.int64)]
    buf, views = bench._pack(ts, "cpu")
    assert buf.dtype == torch.uint8
    base = buf.data_ptr()
    for t, v in zip(ts, views):
        assert v.dtype == t.dtype and v.shape == t.shape
        assert torch.equal(v, t)
        assert (v.data_ptr() - base) % 256 == 0          # 256-byte aligned offsets
        assert v.data_ptr() + v.numel() * v.element_size() <= base + buf.numel()
    # the views share the buffer: writing through one changes the packed bytes
    views[0].fill_(-1)
    assert torch.equal(buf[:4], torch.full((4,), 255, dtype=torch.uint8))
    # the views do not overlap
    spans = sorted((v.data_ptr(), v.data_ptr() + v.numel() * v.element_size()) for v in views)
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))


def test_algorithmic_bytes_of_the_batch1_step():
    c = W.WORKLOADS["h4096_b1_sparse64"]
    heads, att, verify = bench.algorithmic_bytes(c, 64, 2048 + 64)
    K, H, V = c["K"], c["H"], c["V"]
    # bf16 weights read once: K (H*H + H + V*H) elements, plus h and the top-k lists
    assert heads == K * (H * H + H + V * H) * 2 + H * 2 + K * c["topk"] * 8
    assert abs(heads - 1.4785e9) < 1e6
    # keys and values of 32 heads over 2112 slots, queries in bf16, outputs in float32
    assert att == 2 * 32 * 2112 * 128 * 2 + 64 * 32 * 128 * 6
    assert abs(att - 36.18e6) < 0.01e6
    assert verify == 64 * V * 4 + 64 * 4


def test_workloads_have_distinct_seeds():
    seeds = [w["seed"] for w in W.WORKLOADS.values()]
    assert len(seeds) == len(set(seeds)) == 5
    assert np.all(np.array(seeds) > 0)


def test_expected_tokens_of_the_sweep_report():
    # the sweep's E(alpha, gamma) is the cost model's closed form (the oracle's
    # analytic module, pinned to the page's printed numbers)
    from oracle import analytic as A
    for a in (0.0, 0.3, 0.8, 0.99, 1.0):
        for g in (0, 1, 4, 32):
            assert abs(bench.expected_tokens(a, g) - A.expected_tokens(a, g)) < 1e-12
    assert abs(bench.expected_tokens(0.8, 4) - 3.3616) < 1e-12


def test_host_description():
    assert bench.host_cores() >= 1
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
