"""The end-to-end loop of bench.py moves real results: with one step at a
time and with two steps in flight (inputs copied and results read back on
streams of their own), every result buffer read back to the host holds what a
direct run of the same step produces."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_e2e_loop_reads_back_every_step_result(medusa):
    import bench
    dev = torch.device("cuda", 0)
    step = bench.Step(bench.make_inputs(), dev)
    step.run()
    torch.cuda.synchronize()
    ref = [step.acc[n].cpu() for n in ("accept_len", "best_node", "path_nodes", "next_tok")] + [step.h_next.cpu()]
    assert int(ref[0][0]) >= 0  # a real acceptance, not a failure marker
    for pipelined in (False, True):
        dt, h2d, d2h, got = bench.run_e2e(step, 5, 3, pipelined=pipelined, host_results=True)
        assert dt > 0 and h2d > 10_000_000 and d2h > 0
        assert len(got) == (2 if pipelined else 1)
        for segs in got:
            for g, r in zip(segs, ref):
                assert g.dtype == r.dtype and g.shape == r.shape
                assert torch.equal(g, r)
