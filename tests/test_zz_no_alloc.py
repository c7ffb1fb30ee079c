"""The AlltoAllQuantMatmul entry point that allocates nothing.

Some callers cannot hand the library a workspace: a C or Fortran host program
with no device allocator of its own, or a plugin inside a framework that owns
all device memory and forbids cudaMalloc.  mc2_alltoall_quant_mm_no_alloc
serves them from a scratch array built into the library.  These tests call it
through the C ABI and compare every output (out, q, x1_scale and the int32
accumulators) bit for bit with the CPU oracle and with mc2_alltoall_quant_mm
(the rule every AlltoAllQuantMatmul parity test here uses), on calls in a row
with different inputs, so that what one call leaves in the shared scratch
cannot leak into the next.  One shape's GEMM runs a stream-K tail, so the
scratch's partial-sum slots and flags are used too.  The file is named to be
collected last.
"""
import ctypes

import pytest
import torch

import mc2_inputs
import oracle
import quantized_gemm_rank_gb300 as mc2
from parity import assert_bits_equal

A2A = mc2_inputs.A2AShape
# ragged tiles with dynamic quant; 4 K blocks of pre-quantised int8; and a
# stream-K shape: 5 x 8 tiles of 2 K blocks, split over every co-resident CTA
# pair (partial slots and flags in the scratch), 31.3 MiB of the 32 MiB
SHAPES = {
    "dyn-ragged": A2A(rank_size=4, bs_local=300, h=256, n=528, quant_mode=7),
    "full-4kblocks": A2A(rank_size=8, bs_local=520, h=512, n=1024, quant_mode=3),
    "dyn-stream-k": A2A(rank_size=8, bs_local=1100, h=256, n=2048, quant_mode=7),
}
KEYS = ("out", "q_out", "x1_scale_out", "acc_out")
ORACLE_KEYS = {"out": "out", "q_out": "q", "x1_scale_out": "x1_scale", "acc_out": "acc"}


def _device_inputs(shape, seed):
    dev = torch.device("cuda")
    inp = mc2_inputs.a2a_inputs(shape, seed=seed)
    d = {"chunks": [c.to(dev) for c in inp["chunks"]],
         "x1_scale": None if inp["x1_scale"] is None else inp["x1_scale"].to(dev),
         "x2": inp["x2"].to(dev), "x2_scale": inp["x2_scale"].to(dev), "bias": inp["bias"].to(dev)}
    K = shape.rank_size * shape.h

    def outs():
        return {"out": torch.empty((shape.bs_local, shape.n), dtype=torch.bfloat16, device=dev),
                "q_out": torch.empty((shape.bs_local, K), dtype=torch.int8, device=dev),
                "x1_scale_out": torch.empty((shape.bs_local,), dtype=torch.float32, device=dev),
                "acc_out": torch.empty((shape.bs_local, shape.n), dtype=torch.int32, device=dev)}
    return inp, d, outs


def _no_alloc(shape, d, o):
    mc2.mc2_alltoall_quant_mm_no_alloc(d["chunks"], d["x2"], d["x2_scale"], d["bias"],
                                       x1_quant_mode=shape.quant_mode, x1_scale=d["x1_scale"], **o)


def _check(shape, inp, o_new, o_ref, what):
    ref = oracle.alltoall_quant_mm(inp["chunks"], inp["x2"], inp["x2_scale"], inp["bias"],
                                   quant_mode=shape.quant_mode, x1_scale=inp["x1_scale"])
    for key in KEYS:
        assert_bits_equal(o_new[key], ref[ORACLE_KEYS[key]], f"{what}: {key} vs the oracle")
        assert_bits_equal(o_new[key], o_ref[key], f"{what}: {key} vs the workspace entry point")


@pytest.mark.gpu
def test_no_alloc_matches_oracle_and_workspace_entry_point():
    """Every shape, one call each in a row (the layouts differ from call to
    call), checked against the oracle and the workspace entry point."""
    for i, (name, shape) in enumerate(SHAPES.items()):
        inp, d, outs = _device_inputs(shape, seed=40 + i)
        o_ref, o_new = outs(), outs()
        mc2.mc2_alltoall_quant_mm(d["chunks"], d["x2"], d["x2_scale"], d["bias"], x1_quant_mode=shape.quant_mode,
                                  x1_scale=d["x1_scale"], **o_ref)
        _no_alloc(shape, d, o_new)
        torch.cuda.synchronize()
        assert mc2.mc2_device_status() == mc2.MC2_OK
        _check(shape, inp, o_new, o_ref, f"no-alloc {name}")


@pytest.mark.gpu
def test_no_alloc_stream_k_twice_in_a_row_allocates_nothing():
    """Two stream-K calls back to back on the shared scratch with the same
    layout and different inputs: the second reads flags and partial slots
    that the first left behind, which must count for nothing.  Around the
    second call (the first has loaded the library's device code) the device's
    free memory, as the driver reports it, must not change."""
    shape = SHAPES["dyn-stream-k"]
    runs = []
    for seed in (50, 51):
        inp, d, outs = _device_inputs(shape, seed=seed)
        o_ref, o_new = outs(), outs()
        mc2.mc2_alltoall_quant_mm(d["chunks"], d["x2"], d["x2_scale"], d["bias"], x1_quant_mode=shape.quant_mode,
                                  x1_scale=d["x1_scale"], **o_ref)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        allocated_before = torch.cuda.memory_allocated()
        _no_alloc(shape, d, o_new)
        torch.cuda.synchronize()
        if seed == 51:
            assert torch.cuda.mem_get_info()[0] == free_before
        assert torch.cuda.memory_allocated() == allocated_before
        runs.append((inp, o_new, o_ref))
    assert mc2.mc2_device_status() == mc2.MC2_OK
    for k, (inp, o_new, o_ref) in enumerate(runs):
        _check(shape, inp, o_new, o_ref, f"no-alloc stream-K call {k}")


def test_no_alloc_refuses_sizes_beyond_its_scratch():
    # a2a-dyn needs ~128 MiB of scratch, four times the built-in 32 MiB: refused on
    # the host before any device work (so this also runs without a GPU)
    s = mc2_inputs.WORKLOADS["a2a-dyn"]
    need = mc2.mc2_alltoall_quant_mm_workspace(s.rank_size, s.bs_local, s.h, s.n, 7, torch.bfloat16)
    assert need > mc2.NO_ALLOC_SCRATCH_BYTES
    fake = 0x10000
    arr = (ctypes.c_void_p * 8)(*([fake] * 8))
    st = mc2.lib().mc2_alltoall_quant_mm_no_alloc(arr, 8, s.bs_local, s.h, mc2.MC2_BF16, None, fake, fake, fake,
                                                  mc2.MC2_F32, 7, 2, s.n, fake, None, None, None, None, None)
    assert st == mc2.MC2_ERR_WORKSPACE
    assert "built-in scratch" in mc2.last_error()


def test_stream_k_shape_fits_the_scratch():
    # the stream-K shape above must fit the built-in scratch (host-side query only)
    s = SHAPES["dyn-stream-k"]
    need = mc2.mc2_alltoall_quant_mm_workspace(s.rank_size, s.bs_local, s.h, s.n, 7, torch.bfloat16)
    assert 24 << 20 < need <= mc2.NO_ALLOC_SCRATCH_BYTES
