"""Bounded device waits and their status, made to run out on purpose.

"aclnnAlltoAllQuantMatmul" (函数原型 / 返回值) returns a status from the op.
Every wait inside this library's kernels has a time limit; when one runs out
the kernel skips the rest of its work, raises a device status word and
returns, so the context stays usable, and mc2_device_status() reports
MC2_ERR_TIMEOUT.  The test hook mc2_test_expire_next_flag_waits makes every
stream-K finishing part of the next call's GEMM expect one partial sum more
than any part writes, so its wait on the tile's flag (a flag that nothing will
set) runs out after a short limit.  Nothing faults, traps or hangs: the waits
end by their own clock.  Also here: the launch-event hook that the benchmark
uses to time each kernel of a call.
"""
import pytest
import torch

import mc2_inputs
import oracle
import quantized_gemm_rank_gb300 as mc2
from parity import assert_bits_equal

pytestmark = pytest.mark.gpu

# 5 x 8 tiles of 2 K blocks: every tile goes through the stream-K tail
SK_SHAPE = mc2_inputs.A2AShape(rank_size=8, bs_local=1100, h=256, n=2048, quant_mode=7)


def _inputs(shape, seed):
    dev = torch.device("cuda")
    inp = mc2_inputs.a2a_inputs(shape, seed=seed)
    d = {"chunks": [c.to(dev) for c in inp["chunks"]], "x1_scale": inp["x1_scale"].to(dev),
         "x2": inp["x2"].to(dev), "x2_scale": inp["x2_scale"].to(dev), "bias": inp["bias"].to(dev)}
    return inp, d


def _call(shape, d, ws=None, **outs):
    return mc2.mc2_alltoall_quant_mm(d["chunks"], d["x2"], d["x2_scale"], d["bias"], x1_quant_mode=shape.quant_mode,
                                     x1_scale=d["x1_scale"], workspace=ws, **outs)


def test_expired_flag_wait_reports_timeout_and_device_stays_usable():
    shape = SK_SHAPE
    inp, d = _inputs(shape, seed=60)
    dev = torch.device("cuda")
    ws = torch.empty(mc2.mc2_alltoall_quant_mm_workspace(shape.rank_size, shape.bs_local, shape.h, shape.n, 7,
                                                         torch.bfloat16), dtype=torch.uint8, device=dev)
    assert mc2.mc2_device_status() == mc2.MC2_OK
    # 20 ms instead of 2 s: every finishing part gives up after that
    mc2.mc2_test_expire_next_flag_waits(20_000_000)
    _call(shape, d, ws)
    assert mc2.mc2_device_status() == mc2.MC2_ERR_TIMEOUT
    assert "gave up" in mc2.last_error()
    # the status was read and cleared; the hook was one-shot
    assert mc2.mc2_device_status() == mc2.MC2_OK
    # the same workspace (its flags left by the aborted launch) and a new input:
    # the next call is whole and exact
    inp, d = _inputs(shape, seed=61)
    acc = torch.empty((shape.bs_local, shape.n), dtype=torch.int32, device=dev)
    res = _call(shape, d, ws, acc_out=acc)
    torch.cuda.synchronize()
    assert mc2.mc2_device_status() == mc2.MC2_OK
    ref = oracle.alltoall_quant_mm(inp["chunks"], inp["x2"], inp["x2_scale"], inp["bias"], quant_mode=7,
                                   x1_scale=inp["x1_scale"])
    assert_bits_equal(acc.cpu(), ref["acc"], "after the timeout: acc")
    assert_bits_equal(res["out"].cpu(), ref["out"], "after the timeout: out")


def test_launch_events_time_each_kernel_of_a_call():
    """Mode 3 with h % 64 == 0 launches two kernels (the chunks and x2 widened in
    one pass, then the GEMM): three events bracket them, in stream order, each
    interval positive; a fourth event installed past the last launch is not
    recorded by the call."""
    shape = mc2_inputs.A2AShape(rank_size=4, bs_local=512, h=512, n=1024, quant_mode=3)
    inp, d = _inputs(shape, seed=62)
    stream = torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for e in evs:
        e.record(stream)
    torch.cuda.synchronize()
    mc2.mc2_set_launch_events(evs[:4])
    try:
        res = _call(shape, d)
    finally:
        mc2.mc2_set_launch_events(None)
    evs[4].record(stream)
    torch.cuda.synchronize()
    gaps = [evs[i].elapsed_time(evs[i + 1]) for i in range(2)]
    assert all(g > 0 for g in gaps), gaps
    assert evs[2].elapsed_time(evs[4]) >= 0
    # events[3] kept the time it was recorded at before the call (before events[0])
    assert evs[3].elapsed_time(evs[0]) > 0
    ref = oracle.alltoall_quant_mm(inp["chunks"], inp["x2"], inp["x2_scale"], inp["bias"], quant_mode=3,
                                   x1_scale=inp["x1_scale"])
    assert_bits_equal(res["out"].cpu(), ref["out"], "with launch events: out")
    assert mc2.mc2_device_status() == mc2.MC2_OK
