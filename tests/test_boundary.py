"""The C-ABI boundary without a GPU: the library loads, exports every function
that include/*.h declares, and rejects each violated constraint with the right
status before touching CUDA.

Constraints come from "torch_npu.npu_all_gather_base_mm" (参数说明/约束说明:
world_size 2/4/8, k in [256, 65535), 2-D fp16/bf16 operands of one dtype) and
"aclnnAlltoAllQuantMatmul" (约束说明: rankSize 2/4/8, BS and N <= INT32_MAX, no
empty tensors, non-null x1/x2/x2Scale/output/bias, x1QuantMode 3 or 7,
x2QuantMode 2, rankSize*H a multiple of 16 in [1, 35000]) and "QuantAllReduce"
(参数说明/约束说明: ranks 2/4/8, x int8 or fp8, scales fp32 or e8m0 with e8m0
only for fp8 x, output fp32/fp16/bf16, H in [1024, 8192] and 128-aligned, no
empty tensors).
"""
import ctypes
import glob
import os
import re

import pytest
import torch

import quantized_gemm_rank_gb300 as mc2

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000  # a 16-byte-aligned non-null address; validation must never dereference it


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(mc2_\w+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    L = mc2.lib()
    names = declared_functions()
    assert "mc2_all_gather_mm" in names and "mc2_alltoall_quant_mm" in names
    for name in names:
        assert hasattr(L, name), name


def test_calibration_probe_is_not_in_the_operations_library():
    """The mma.sync calibration probe lives in its own library that only the
    benchmark loads; it rejects bad arguments before launching."""
    from quantized_gemm_rank_gb300 import build
    assert not hasattr(mc2.lib(), "mc2_calib_mma_sync")
    C = ctypes.CDLL(build.build_calib())
    C.mc2_calib_mma_sync.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.POINTER(ctypes.c_double)]
    ops = ctypes.c_double(-1.0)
    fake = ctypes.c_void_p(256)   # never dereferenced: validation fails first
    assert C.mc2_calib_mma_sync(0, 16, 4, None, None, ctypes.byref(ops)) == -1
    assert C.mc2_calib_mma_sync(0, 16, 4, fake, None, None) == -1
    assert C.mc2_calib_mma_sync(2, 16, 4, fake, None, ctypes.byref(ops)) == -2
    assert C.mc2_calib_mma_sync(0, 0, 4, fake, None, ctypes.byref(ops)) == -2
    assert C.mc2_calib_mma_sync(1, 16, 0, fake, None, ctypes.byref(ops)) == -2
    assert ops.value == -1.0


def test_launch_events_and_test_hook_validate_their_arguments():
    L = mc2.lib()
    assert L.mc2_set_launch_events(None, 0) == mc2.MC2_OK
    assert L.mc2_set_launch_events(None, 2) == mc2.MC2_ERR_NULL
    assert L.mc2_set_launch_events(None, 9) == mc2.MC2_ERR_SHAPE
    assert L.mc2_set_launch_events(None, -1) == mc2.MC2_ERR_SHAPE
    arr = (ctypes.c_void_p * 2)(FAKE, None)
    assert L.mc2_set_launch_events(arr, 2) == mc2.MC2_ERR_NULL
    assert "events[1]" in mc2.last_error()
    # out-of-range limits are refused (and arm nothing)
    assert L.mc2_test_expire_next_flag_waits(0) == mc2.MC2_ERR_SHAPE
    assert L.mc2_test_expire_next_flag_waits(2_000_000_001) == mc2.MC2_ERR_SHAPE


def test_status_strings():
    assert mc2.status_str(0) == "MC2_OK"
    assert mc2.status_str(mc2.MC2_ERR_TIMEOUT) == "MC2_ERR_TIMEOUT"
    assert mc2.status_str(-99) == "MC2_ERR_UNKNOWN"


def ag_call(world_size=2, m_local=16, k=256, n=64, x2_is_nk=0, bias=None, dtype=mc2.MC2_BF16, gather=1,
            chunks=None, x2=FAKE, out=FAKE, gathered=FAKE):
    if chunks is None:
        chunks = [FAKE] * max(world_size, 1)
    arr = (ctypes.c_void_p * len(chunks))(*chunks)
    return mc2.lib().mc2_all_gather_mm(arr, world_size, m_local, k, x2, n, x2_is_nk, bias, dtype, gather, out,
                                       gathered if gather else None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(world_size=3), mc2.MC2_ERR_SHAPE),
    (dict(world_size=1), mc2.MC2_ERR_SHAPE),
    (dict(world_size=16), mc2.MC2_ERR_SHAPE),
    (dict(k=255), mc2.MC2_ERR_SHAPE),
    (dict(k=65535), mc2.MC2_ERR_SHAPE),
    (dict(m_local=0), mc2.MC2_ERR_SHAPE),
    (dict(n=0), mc2.MC2_ERR_SHAPE),
    (dict(dtype=mc2.MC2_F32), mc2.MC2_ERR_DTYPE),
    (dict(dtype=mc2.MC2_I8), mc2.MC2_ERR_DTYPE),
    (dict(x2=None), mc2.MC2_ERR_NULL),
    (dict(out=None), mc2.MC2_ERR_NULL),
    (dict(chunks=[FAKE, None]), mc2.MC2_ERR_NULL),
    (dict(gathered=None), mc2.MC2_ERR_NULL),
    (dict(m_local=12), mc2.MC2_ERR_UNSUPPORTED),
    (dict(k=260), mc2.MC2_ERR_UNSUPPORTED),
    (dict(n=60), mc2.MC2_ERR_UNSUPPORTED),
    (dict(x2=FAKE + 8), mc2.MC2_ERR_UNSUPPORTED),
    (dict(chunks=[FAKE, FAKE + 2]), mc2.MC2_ERR_UNSUPPORTED),
])
def test_all_gather_rejects(kw, status):
    assert ag_call(**kw) == status
    assert mc2.last_error() != ""


def test_all_gather_k_bounds_accepted_by_validation():
    # k = 256 and k = 65528 (< 65535, multiple of 8) pass validation; without a GPU the
    # call then fails at the first CUDA call, never earlier.
    if torch.cuda.is_available():
        pytest.skip("would launch on a real device with fake pointers")
    for k in (256, 65528):
        assert ag_call(k=k) == mc2.MC2_ERR_CUDA, mc2.last_error()


def test_all_gather_gather_flag_consistency():
    arr = (ctypes.c_void_p * 2)(FAKE, FAKE)
    st = mc2.lib().mc2_all_gather_mm(arr, 2, 16, 256, FAKE, 64, 0, None, mc2.MC2_BF16, 0, FAKE, FAKE, None)
    assert st == mc2.MC2_ERR_SHAPE


def mmrs_call(world_size=2, m=16, k_local=256, n=64, w_is_nk=1, bias=None, dtype=mc2.MC2_BF16, xs=None, ws=None,
              outs=None):
    xs = [FAKE] * max(world_size, 1) if xs is None else xs
    ws = [FAKE] * max(world_size, 1) if ws is None else ws
    outs = [FAKE] * max(world_size, 1) if outs is None else outs
    arr = lambda v: (ctypes.c_void_p * len(v))(*v)
    return mc2.lib().mc2_matmul_reduce_scatter(arr(xs), arr(ws), world_size, m, k_local, n, w_is_nk, bias, dtype,
                                               arr(outs), None)


@pytest.mark.parametrize("kw,status", [
    (dict(world_size=3), mc2.MC2_ERR_SHAPE),
    (dict(world_size=1), mc2.MC2_ERR_SHAPE),
    (dict(m=17), mc2.MC2_ERR_SHAPE),                    # m not divisible by world_size
    (dict(m=0), mc2.MC2_ERR_SHAPE),
    (dict(n=0), mc2.MC2_ERR_SHAPE),
    (dict(k_local=255), mc2.MC2_ERR_SHAPE),
    (dict(k_local=65535), mc2.MC2_ERR_SHAPE),
    (dict(dtype=mc2.MC2_F32), mc2.MC2_ERR_DTYPE),
    (dict(xs=[FAKE, None]), mc2.MC2_ERR_NULL),
    (dict(ws=[None, FAKE]), mc2.MC2_ERR_NULL),
    (dict(outs=[FAKE, None]), mc2.MC2_ERR_NULL),
    (dict(k_local=328), mc2.MC2_ERR_UNSUPPORTED),       # a k-tile would straddle two ranks
    (dict(n=60), mc2.MC2_ERR_UNSUPPORTED),
    (dict(ws=[FAKE, FAKE + 8]), mc2.MC2_ERR_UNSUPPORTED),
    (dict(bias=FAKE + 2), mc2.MC2_ERR_UNSUPPORTED),
])
def test_matmul_reduce_scatter_rejects(kw, status):
    assert mmrs_call(**kw) == status, mc2.last_error()
    assert mc2.last_error() != ""


def test_matmul_reduce_scatter_null_arrays():
    L = mc2.lib()
    arr = (ctypes.c_void_p * 2)(FAKE, FAKE)
    assert L.mc2_matmul_reduce_scatter(None, arr, 2, 16, 256, 64, 1, None, mc2.MC2_BF16, arr, None) == mc2.MC2_ERR_NULL
    assert L.mc2_matmul_reduce_scatter(arr, arr, 2, 16, 256, 64, 1, None, mc2.MC2_BF16, None, None) == mc2.MC2_ERR_NULL


def test_matmul_reduce_scatter_bounds_accepted_by_validation():
    if torch.cuda.is_available():
        pytest.skip("would launch on a real device with fake pointers")
    for kl in (256, 65472):
        assert mmrs_call(k_local=kl) == mc2.MC2_ERR_CUDA, mc2.last_error()


def wg_call(m=64, n=64, k=64, dtype=mc2.MC2_BF16, dy=FAKE, x=FAKE, dw=FAKE, db=None):
    return mc2.lib().mc2_matmul_weight_grad(dy, m, n, x, k, dtype, dw, db, None)


@pytest.mark.parametrize("kw,status", [
    (dict(dy=None), mc2.MC2_ERR_NULL),
    (dict(x=None), mc2.MC2_ERR_NULL),
    (dict(dw=None), mc2.MC2_ERR_NULL),
    (dict(dtype=mc2.MC2_I8), mc2.MC2_ERR_DTYPE),
    (dict(m=0), mc2.MC2_ERR_SHAPE),
    (dict(n=0), mc2.MC2_ERR_SHAPE),
    (dict(k=2 ** 31), mc2.MC2_ERR_SHAPE),
    (dict(n=60), mc2.MC2_ERR_UNSUPPORTED),
    (dict(k=12), mc2.MC2_ERR_UNSUPPORTED),
    (dict(db=FAKE + 2), mc2.MC2_ERR_UNSUPPORTED),
])
def test_weight_grad_rejects(kw, status):
    assert wg_call(**kw) == status, mc2.last_error()
    assert mc2.last_error() != ""


def a2a_call(rank_size=2, bs_local=16, h=64, x1_dtype=mc2.MC2_BF16, x1_scale=None, x2=FAKE, x2_scale=FAKE,
             bias=FAKE, bias_dtype=mc2.MC2_F32, mode=7, mode2=2, n=64, out=FAKE, ws=FAKE, ws_bytes=1 << 40,
             chunks=None, a2a_out=None):
    if chunks is None:
        chunks = [FAKE] * max(rank_size, 1)
    arr = (ctypes.c_void_p * len(chunks))(*chunks)
    return mc2.lib().mc2_alltoall_quant_mm(arr, rank_size, bs_local, h, x1_dtype, x1_scale, x2, x2_scale, bias,
                                           bias_dtype, mode, mode2, n, out, a2a_out, None, None, None, ws, ws_bytes,
                                           None)


@pytest.mark.parametrize("kw,status", [
    (dict(rank_size=3), mc2.MC2_ERR_SHAPE),
    (dict(rank_size=16), mc2.MC2_ERR_SHAPE),
    (dict(bs_local=0), mc2.MC2_ERR_SHAPE),
    (dict(h=0), mc2.MC2_ERR_SHAPE),
    (dict(n=0), mc2.MC2_ERR_SHAPE),
    (dict(bs_local=2 ** 30, rank_size=2), mc2.MC2_ERR_SHAPE),          # BS = 2^31 > INT32_MAX
    (dict(n=2 ** 31), mc2.MC2_ERR_SHAPE),
    (dict(rank_size=8, h=4376), mc2.MC2_ERR_SHAPE),                     # R*H = 35008 > 35000
    (dict(rank_size=2, h=12), mc2.MC2_ERR_SHAPE),                       # R*H = 24, not % 16
    (dict(mode=1), mc2.MC2_ERR_DTYPE),
    (dict(mode=0), mc2.MC2_ERR_DTYPE),
    (dict(mode2=1), mc2.MC2_ERR_DTYPE),
    (dict(mode=7, x1_dtype=mc2.MC2_I8), mc2.MC2_ERR_DTYPE),
    (dict(mode=3, x1_dtype=mc2.MC2_BF16, x1_scale=FAKE), mc2.MC2_ERR_DTYPE),
    (dict(bias_dtype=mc2.MC2_I8), mc2.MC2_ERR_DTYPE),
    (dict(mode=3, x1_dtype=mc2.MC2_I8, x1_scale=None), mc2.MC2_ERR_NULL),
    (dict(x2=None), mc2.MC2_ERR_NULL),
    (dict(x2_scale=None), mc2.MC2_ERR_NULL),
    (dict(bias=None), mc2.MC2_ERR_NULL),
    (dict(out=None), mc2.MC2_ERR_NULL),
    (dict(chunks=[FAKE, None]), mc2.MC2_ERR_NULL),
    (dict(ws=None), mc2.MC2_ERR_WORKSPACE),
    (dict(ws_bytes=16), mc2.MC2_ERR_WORKSPACE),
    (dict(n=40), mc2.MC2_ERR_UNSUPPORTED),
    (dict(out=FAKE + 4), mc2.MC2_ERR_UNSUPPORTED),
    (dict(a2a_out=FAKE + 8), mc2.MC2_ERR_UNSUPPORTED),
])
def test_alltoall_rejects(kw, status):
    assert a2a_call(**kw) == status, mc2.last_error()
    assert mc2.last_error() != ""


def test_alltoall_boundary_values_accepted_by_validation():
    if torch.cuda.is_available():
        pytest.skip("would launch on a real device with fake pointers")
    # R*H = 35000 is allowed by the page but is not a multiple of 16 -> shape error;
    # R*H = 34992 (largest multiple of 16 <= 35000) passes validation
    assert a2a_call(rank_size=8, h=4375) == mc2.MC2_ERR_SHAPE
    assert a2a_call(rank_size=8, h=4374) == mc2.MC2_ERR_CUDA, mc2.last_error()
    assert a2a_call(rank_size=2, h=8) == mc2.MC2_ERR_CUDA, mc2.last_error()  # R*H = 16


def test_workspace_query():
    nbytes = mc2.mc2_alltoall_quant_mm_workspace(8, 4096, 1024, 4096, 7, torch.bfloat16)
    assert nbytes >= 8192 * 4096 * 2 + 4096 * 8192 * 2 + 4096 * 4
    with pytest.raises(mc2.Mc2Error) as ei:
        mc2.mc2_alltoall_quant_mm_workspace(3, 4096, 1024, 4096, 7, torch.bfloat16)
    assert ei.value.status == mc2.MC2_ERR_SHAPE


def test_binding_refuses_cpu_tensors():
    x = [torch.zeros(16, 256, dtype=torch.bfloat16)] * 2
    with pytest.raises(ValueError):
        mc2.mc2_all_gather_mm(x, torch.zeros(256, 64, dtype=torch.bfloat16),
                              out=torch.zeros(32, 64, dtype=torch.bfloat16),
                              gathered=torch.zeros(32, 256, dtype=torch.bfloat16))


def qar_call(world_size=2, bs=4, h=1024, x_dtype=mc2.MC2_I8, scale_dtype=mc2.MC2_F32, out_dtype=mc2.MC2_BF16,
             xs=None, ss=None, out=FAKE):
    xs = [FAKE] * max(world_size, 1) if xs is None else xs
    ss = [FAKE] * max(world_size, 1) if ss is None else ss
    xa = (ctypes.c_void_p * len(xs))(*xs)
    sa = (ctypes.c_void_p * len(ss))(*ss)
    return mc2.lib().mc2_quant_all_reduce(xa, sa, world_size, bs, h, x_dtype, scale_dtype, out_dtype, out, None)


@pytest.mark.parametrize("kw,status", [
    (dict(world_size=3), mc2.MC2_ERR_SHAPE),
    (dict(world_size=1), mc2.MC2_ERR_SHAPE),
    (dict(world_size=16), mc2.MC2_ERR_SHAPE),
    (dict(bs=0), mc2.MC2_ERR_SHAPE),
    (dict(h=896), mc2.MC2_ERR_SHAPE),
    (dict(h=8320), mc2.MC2_ERR_SHAPE),
    (dict(h=1088), mc2.MC2_ERR_SHAPE),
    (dict(h=1023), mc2.MC2_ERR_SHAPE),
    (dict(x_dtype=mc2.MC2_BF16), mc2.MC2_ERR_DTYPE),
    (dict(x_dtype=mc2.MC2_E8M0), mc2.MC2_ERR_DTYPE),
    (dict(scale_dtype=mc2.MC2_BF16), mc2.MC2_ERR_DTYPE),
    (dict(x_dtype=mc2.MC2_I8, scale_dtype=mc2.MC2_E8M0), mc2.MC2_ERR_DTYPE),
    (dict(out_dtype=mc2.MC2_I8), mc2.MC2_ERR_DTYPE),
    (dict(out_dtype=mc2.MC2_F8E4M3), mc2.MC2_ERR_DTYPE),
    (dict(out=None), mc2.MC2_ERR_NULL),
    (dict(xs=[FAKE, None]), mc2.MC2_ERR_NULL),
    (dict(ss=[None, FAKE]), mc2.MC2_ERR_NULL),
    (dict(out=FAKE + 8), mc2.MC2_ERR_UNSUPPORTED),
    (dict(xs=[FAKE, FAKE + 4]), mc2.MC2_ERR_UNSUPPORTED),
    (dict(ss=[FAKE + 4, FAKE]), mc2.MC2_ERR_UNSUPPORTED),
])
def test_quant_all_reduce_rejects(kw, status):
    assert qar_call(**kw) == status, mc2.last_error()
    assert mc2.last_error() != ""


def test_quant_all_reduce_null_arrays():
    L = mc2.lib()
    assert L.mc2_quant_all_reduce(None, None, 2, 4, 1024, mc2.MC2_I8, mc2.MC2_F32, mc2.MC2_BF16, FAKE,
                                  None) == mc2.MC2_ERR_NULL


def test_quant_all_reduce_bounds_accepted_by_validation():
    if torch.cuda.is_available():
        pytest.skip("would launch on a real device with fake pointers")
    # H = 1024 and 8192 are the ends of the page's range; every type pairing
    # the page allows passes validation (and then fails only for want of a GPU)
    for h in (1024, 8192):
        assert qar_call(h=h) == mc2.MC2_ERR_CUDA, mc2.last_error()
    for xd in (mc2.MC2_F8E4M3, mc2.MC2_F8E5M2):
        for sd in (mc2.MC2_F32, mc2.MC2_E8M0):
            for od in (mc2.MC2_F32, mc2.MC2_F16, mc2.MC2_BF16):
                assert qar_call(world_size=8, x_dtype=xd, scale_dtype=sd, out_dtype=od) == mc2.MC2_ERR_CUDA


def _z(*shape, dtype=torch.bfloat16):
    return torch.zeros(*shape, dtype=dtype)


_AG = dict(x_chunks=[_z(16, 256)] * 2, x2=_z(256, 64))
_A2A = dict(chunks=[_z(8, 64)] * 4, x2=_z(256, 32, dtype=torch.int8), x2_scale=_z(32, dtype=torch.float32),
            bias=_z(32, dtype=torch.float32))


@pytest.mark.parametrize("call,kw,what", [
    # AllGatherMatmul: every tensor against the sizes of chunk 0 and x2
    ("ag", dict(x_chunks=[_z(16, 256), _z(8, 256)]), r"x_chunks\[1\] must have shape \(16, 256\)"),
    ("ag", dict(x_chunks=[_z(16, 256), _z(16, 256, dtype=torch.float16)]), r"x_chunks\[1\] must be of dtype"),
    ("ag", dict(x2=_z(128, 64)), r"x2 must have shape \(256, 64\)"),
    ("ag", dict(x2=_z(256, 64, dtype=torch.float16)), "x2 must be of dtype"),
    ("ag", dict(bias=_z(63)), r"bias must have shape \(64,\)"),
    ("ag", dict(out=_z(31, 64)), r"out must have shape \(32, 64\)"),
    ("ag", dict(gathered=_z(32, 128)), r"gathered must have shape \(32, 256\)"),
    # MatmulReduceScatter
    ("rs", dict(w_chunks=[_z(48, 64)]), "w_chunks must hold 2 shards"),
    ("rs", dict(w_chunks=[_z(48, 64), _z(48, 32)]), r"w_chunks\[1\] must have shape \(48, 64\)"),
    ("rs", dict(out_chunks=[_z(8, 48), _z(16, 48)]), r"out_chunks\[0\] must have shape \(16, 48\)"),
    # weight gradient
    ("wg", dict(x=_z(31, 128)), r"x must have shape \(32, 128\)"),
    ("wg", dict(dw=_z(128, 48)), r"dw must have shape \(48, 128\)"),
    ("wg", dict(db=_z(48, dtype=torch.float32)), "db must be of dtype"),
    # QuantAllReduce
    ("qar", dict(x_chunks=[_z(4, 1024, dtype=torch.int8), _z(4, 512, dtype=torch.int8)]),
     r"x_chunks\[1\] must have shape \(4, 1024\)"),
    ("qar", dict(scale_chunks=[_z(4, 8, dtype=torch.float32), _z(4, 4, dtype=torch.float32)]),
     r"scale_chunks\[1\] must hold 32 fp32 scales"),
    ("qar", dict(out=_z(4, 1024, dtype=torch.float16)), "out must be of dtype"),
    # AlltoAllQuantMatmul (the workspace entry point and the one without)
    ("a2a", dict(x2=_z(128, 32, dtype=torch.int8)), r"x2 must have shape \(256, 32\)"),
    ("a2a", dict(x2_scale=_z(31, dtype=torch.float32)), r"x2_scale must have shape \(32,\)"),
    ("a2a", dict(bias=_z(32, dtype=torch.float16)), "bias must be of dtype"),
    ("a2a", dict(x1_scale=_z(128)), r"x1_scale \(smooth scale\) must have shape \(256,\)"),
    ("a2a", dict(out=_z(8, 32, dtype=torch.float16)), "out must be of dtype"),
    ("a2a", dict(q_out=_z(8, 128, dtype=torch.int8)), r"q_out must have shape \(8, 256\)"),
    ("a2a", dict(acc_out=_z(8, 32, dtype=torch.float32)), "acc_out must be of dtype"),
    ("a2a", dict(alltoall_out=_z(4, 8, 32)), r"alltoall_out must have shape \(4, 8, 64\)"),
    ("a2a-full", dict(x1_scale=_z(4, dtype=torch.float32)), r"x1_scale \(per-token scale\) must have shape \(8,\)"),
    ("no-alloc", dict(out=None), "out must be given"),
])
def test_binding_checks_shapes_and_dtypes_before_any_launch(call, kw, what):
    """The kernels trust the sizes the binding passes them, so every tensor's
    shape and dtype is checked against those sizes first (these run on CPU
    tensors: the check comes before the device check and any library call)."""
    with pytest.raises(ValueError, match=what):
        if call == "ag":
            a = dict(_AG, **kw)
            mc2.mc2_all_gather_mm(a.pop("x_chunks"), a.pop("x2"), **a)
        elif call == "rs":
            a = dict(dict(x_chunks=[_z(32, 64)] * 2, w_chunks=[_z(48, 64)] * 2), **kw)
            mc2.mc2_matmul_reduce_scatter(a.pop("x_chunks"), a.pop("w_chunks"), **a)
        elif call == "wg":
            a = dict(dict(dy=_z(32, 48), x=_z(32, 128)), **kw)
            mc2.mc2_matmul_weight_grad(a.pop("dy"), a.pop("x"), **a)
        elif call == "qar":
            a = dict(dict(x_chunks=[_z(4, 1024, dtype=torch.int8)] * 2,
                          scale_chunks=[_z(4, 8, dtype=torch.float32)] * 2), **kw)
            mc2.mc2_quant_all_reduce(a.pop("x_chunks"), a.pop("scale_chunks"), **a)
        elif call in ("a2a", "a2a-full"):
            base = dict(_A2A) if call == "a2a" else dict(_A2A, chunks=[_z(8, 64, dtype=torch.int8)] * 4)
            a = dict(base, x1_quant_mode=7 if call == "a2a" else 3, **kw)
            mc2.mc2_alltoall_quant_mm(a.pop("chunks"), a.pop("x2"), a.pop("x2_scale"), a.pop("bias"), **a)
        else:
            a = dict(_A2A, x1_quant_mode=7, **kw)
            mc2.mc2_alltoall_quant_mm_no_alloc(a.pop("chunks"), a.pop("x2"), a.pop("x2_scale"), a.pop("bias"), **a)
