"""The AlltoAllQuantMatmul entry point that allocates nothing.

Some callers cannot hand the library a workspace: a C or Fortran host program
with no device allocator of its own, or a plugin inside a framework that owns
all device memory and forbids cudaMalloc.  mc2_alltoall_quant_mm_no_alloc
serves them from a scratch array built into the library.  These tests call it
through the C ABI and compare it with mc2_alltoall_quant_mm (bit for bit, the
rule every AlltoAllQuantMatmul parity test here uses), on two calls in a row
with different inputs, so that what the first call leaves in the shared
scratch cannot leak into the second.  The file is named to be collected last.
"""
import pytest
import torch

import mc2_inputs
import quantized_gemm_rank_gb300 as mc2
from parity import assert_bits_equal

A2A = mc2_inputs.A2AShape
SHAPES = [
    A2A(rank_size=4, bs_local=300, h=256, n=528, quant_mode=7),          # ragged tiles, dynamic quant
    A2A(rank_size=8, bs_local=520, h=512, n=1024, quant_mode=3),         # 4 K blocks, pre-quantised int8
]


def _device_inputs(shape, seed):
    dev = torch.device("cuda")
    inp = mc2_inputs.a2a_inputs(shape, seed=seed)
    d = {"chunks": [c.to(dev) for c in inp["chunks"]],
         "x1_scale": None if inp["x1_scale"] is None else inp["x1_scale"].to(dev),
         "x2": inp["x2"].to(dev), "x2_scale": inp["x2_scale"].to(dev), "bias": inp["bias"].to(dev)}
    K = shape.rank_size * shape.h
    outs = lambda: {"out": torch.empty((shape.bs_local, shape.n), dtype=torch.bfloat16, device=dev),  # noqa: E731
                    "q_out": torch.empty((shape.bs_local, K), dtype=torch.int8, device=dev),
                    "x1_scale_out": torch.empty((shape.bs_local,), dtype=torch.float32, device=dev),
                    "acc_out": torch.empty((shape.bs_local, shape.n), dtype=torch.int32, device=dev)}
    return d, outs


@pytest.mark.gpu
def test_no_alloc_matches_workspace_entry_point_twice():
    runs = []
    for i, shape in enumerate(SHAPES):
        d, outs = _device_inputs(shape, seed=40 + i)
        o_ref, o_new = outs(), outs()
        mc2.mc2_alltoall_quant_mm(d["chunks"], d["x2"], d["x2_scale"], d["bias"], x1_quant_mode=shape.quant_mode,
                                  x1_scale=d["x1_scale"], **o_ref)
        torch.cuda.synchronize()
        before = torch.cuda.memory_allocated()
        mc2.mc2_alltoall_quant_mm_no_alloc(d["chunks"], d["x2"], d["x2_scale"], d["bias"],
                                           x1_quant_mode=shape.quant_mode, x1_scale=d["x1_scale"], **o_new)
        torch.cuda.synchronize()
        assert torch.cuda.memory_allocated() == before
        runs.append((shape, o_ref, o_new))
    assert mc2.mc2_device_status() == mc2.MC2_OK
    for shape, o_ref, o_new in runs:
        for key in ("out", "q_out", "x1_scale_out", "acc_out"):
            assert_bits_equal(o_new[key], o_ref[key], f"no-alloc mode {shape.quant_mode}: {key}")


def test_no_alloc_refuses_sizes_beyond_its_scratch():
    # a2a-dyn needs ~128 MiB of scratch, four times the built-in 32 MiB: refused on
    # the host before any device work (so this also runs without a GPU)
    s = mc2_inputs.WORKLOADS["a2a-dyn"]
    need = mc2.mc2_alltoall_quant_mm_workspace(s.rank_size, s.bs_local, s.h, s.n, 7, torch.bfloat16)
    assert need > mc2.NO_ALLOC_SCRATCH_BYTES
    import ctypes
    fake = 0x10000
    arr = (ctypes.c_void_p * 8)(*([fake] * 8))
    st = mc2.lib().mc2_alltoall_quant_mm_no_alloc(arr, 8, s.bs_local, s.h, mc2.MC2_BF16, None, fake, fake, fake,
                                                  mc2.MC2_F32, 7, 2, s.n, fake, None, None, None, None, None)
    assert st == mc2.MC2_ERR_WORKSPACE
    assert "built-in scratch" in mc2.last_error()
