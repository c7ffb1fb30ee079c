"""The benchmark's end-to-end pipeline moves and computes every step.

bench.time_e2e times the hot path with host buffers: each step uploads all of
its inputs from pinned host memory, runs both calls and downloads all of its
outputs, on three streams and three device buffer sets.  Here it runs on small
shapes, and the outputs that reached the host must be bit-identical to a
direct device run of the same step (both calls are deterministic).
"""
import pytest
import torch

import bench
import mc2_inputs
from parity import assert_bits_equal

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("ag_name,a2a_name", [("ag-tiny", "a2a-dyn-small")])
def test_e2e_outputs_match_a_device_run(ag_name, a2a_name):
    dev = torch.device("cuda")
    ag_s, a2a_s = mc2_inputs.WORKLOADS[ag_name], mc2_inputs.WORKLOADS[a2a_name]
    ref_step = bench.Step(dev, ag_s, a2a_s, seed=3)
    ref_step.run()
    torch.cuda.synchronize()
    ref = [t.cpu() for t in ref_step.outputs()]
    step = bench.Step(dev, ag_s, a2a_s, host=ref_step.host)
    ms, h2d, d2h, got = bench.time_e2e(step, 4, 1, dev, return_outputs=True)
    assert ms > 0
    assert h2d >= sum(t.numel() * t.element_size() for t in bench._ag_host_tensors(ref_step.host["ag"]))
    assert d2h >= sum(t.numel() * t.element_size() for t in ref)
    assert len(got) == len(ref)
    for i, (g, r) in enumerate(zip(got, ref)):
        assert_bits_equal(g, r, f"e2e output {i}")
