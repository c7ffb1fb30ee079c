"""The C ABI called from several host threads at once, each on its own stream.

The library keeps per-device caches (occupancy, the status word's address, the
driver's tensor-map entry point) that the first calls fill; calls that race to
fill them must still launch correctly.  Every thread runs both hot-path calls
(AllGatherMatmul and the dynamic-quant AlltoAllQuantMatmul) on its own stream
and its own buffers, and every result must equal, bit for bit, the result of
the same call made alone.  The kernels are deterministic: the float GEMMs
compute every tile whole, and the integer GEMM's stream-K tail, which meets
its partial sums through workspace flags and atomics, adds exact int32 values,
so the order in which the parts finish does not change the bits.
"""
import threading

import pytest
import torch

import mc2_inputs
import quantized_gemm_rank_gb300 as mc2

pytestmark = pytest.mark.gpu

AG = mc2_inputs.AGShape(world_size=4, m_local=200, k=640, n=392, x2_is_nk=True, bias=True)
A2A = mc2_inputs.A2AShape(rank_size=4, bs_local=300, h=256, n=528, quant_mode=7)
THREADS = 6
REPEATS = 4


def _device_inputs():
    dev = torch.device("cuda")
    ag = mc2_inputs.ag_inputs(AG, seed=11)
    a2a = mc2_inputs.a2a_inputs(A2A, seed=12)
    return ({"chunks": [c.to(dev) for c in ag["chunks"]], "x2": ag["x2"].to(dev), "bias": ag["bias"].to(dev)},
            {"chunks": [c.to(dev) for c in a2a["chunks"]], "x1_scale": a2a["x1_scale"].to(dev),
             "x2": a2a["x2"].to(dev), "x2_scale": a2a["x2_scale"].to(dev), "bias": a2a["bias"].to(dev)})


def _run(ag, a2a, stream):
    with torch.cuda.stream(stream):
        out, gathered = mc2.mc2_all_gather_mm(ag["chunks"], ag["x2"], x2_is_nk=True, bias=ag["bias"], stream=stream)
        res = mc2.mc2_alltoall_quant_mm(a2a["chunks"], a2a["x2"], a2a["x2_scale"], a2a["bias"], x1_quant_mode=7,
                                        x1_scale=a2a["x1_scale"], stream=stream)
    stream.synchronize()
    return out.cpu(), gathered.cpu(), res["out"].cpu()


def test_concurrent_host_threads_match_a_lone_call():
    ag, a2a = _device_inputs()
    ref = _run(ag, a2a, torch.cuda.Stream())
    results, errors = {}, []
    start = threading.Barrier(THREADS)

    def worker(t):
        try:
            s = torch.cuda.Stream()
            start.wait()
            results[t] = [_run(ag, a2a, s) for _ in range(REPEATS)]
        except Exception as e:  # reported below, with the thread
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(THREADS)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not errors, errors
    assert sorted(results) == list(range(THREADS))
    assert mc2.mc2_device_status() == mc2.MC2_OK
    for t, runs in results.items():
        for i, got in enumerate(runs):
            for name, a, b in zip(("ag out", "gathered", "a2a out"), got, ref):
                assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"thread {t} run {i}: {name}"
