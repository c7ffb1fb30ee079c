"""CPU oracle for the MC2 fused-linear hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may import this package.  The product library never
loads it and shares no code with it.  The arithmetic lives in plain C
(``mc2_oracle.c``: fp64-accumulated bf16/fp16 matmul, exact int64-accumulated
int8 matmul, fp32 per-token quant and dequant, 16-bit conversions written from
the IEEE layouts); this module only marshals torch CPU tensors into it.

Pages followed (title -- section):
  * "torch_npu.npu_all_gather_base_mm" -- 功能说明, 接口原型, 输出说明, 约束说明
  * "aclnnAlltoAllQuantMatmul" -- 功能说明 / 计算公式 (dynamic- and full-quant)
  * "hyper_parallel .../tensor_parallel/mc2.py" -- module docstring (the
    all_gather_matmul / matmul_reduce_scatter duals and their dW), and
    AllGatherMatmulFunction / MatmulReduceScatterFunction
  * "QuantAllReduce" (mc2/quant_all_reduce) -- 功能说明 (formula), 参数说明,
    约束说明 (int8 / fp8 data, pertoken-pergroup fp32 or mx e8m0 scales)

Every function here is pinned by ``tests/test_oracle_*.py`` against closed
forms, brute force and independent library routines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mc2_oracle.c")
_LIB = os.path.join(_HERE, "libmc2_oracle.so")
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int


def compile_library(src: str, out: str) -> str:
    """gcc the oracle source `src` into the shared library `out` (OpenMP, no FMA contraction)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the C oracle (when its source is newer than the library)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_library(_SRC, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        # MC2_ORACLE_LIB names an oracle library built elsewhere from a copy of
        # mc2_oracle.c: the planted-mistake tests (tests/test_oracle_mutants.py)
        # run the pins against copies with one mistake each through it
        path = os.environ.get("MC2_ORACLE_LIB") or build()
        lib = ctypes.CDLL(path)
        lib.oracle_decode16.restype = ctypes.c_double
        lib.oracle_decode16.argtypes = [ctypes.c_uint16, _INT]
        lib.oracle_encode16_rne.restype = ctypes.c_uint16
        lib.oracle_encode16_rne.argtypes = [ctypes.c_double, _INT]
        lib.oracle_decode16_array.argtypes = [_P, _I64, _INT, _P]
        lib.oracle_encode16_array.argtypes = [_P, _I64, _INT, _P]
        lib.oracle_gather.argtypes = [_P, _INT, _I64, _I64, _P]
        lib.oracle_all_gather_mm.argtypes = [_P, _INT, _I64, _I64, _P, _I64, _INT, _P, _INT, _P, _I64, _P]
        lib.oracle_permute.argtypes = [_P, _INT, _I64, _I64, _INT, _P, _I64, _P]
        lib.oracle_comm_out.argtypes = [_P, _INT, _I64, _I64, _INT, _P]
        lib.oracle_matmul_weight_grad.argtypes = [_P, _P, _I64, _I64, _I64, _INT, _P, _I64, _P, _P]
        lib.oracle_decode_fp8.restype = ctypes.c_double
        lib.oracle_decode_fp8.argtypes = [ctypes.c_uint8, _INT]
        lib.oracle_decode_e8m0.restype = ctypes.c_double
        lib.oracle_decode_e8m0.argtypes = [ctypes.c_uint8]
        lib.oracle_quant_all_reduce.argtypes = [_P, _P, _INT, _I64, _I64, _INT, _INT, _INT, _P]
        lib.oracle_quant_pertoken_dynamic.argtypes = [_P, _I64, _I64, _P, _INT, _P, _P]
        lib.oracle_int8_mm.argtypes = [_P, _I64, _I64, _P, _I64, _P]
        lib.oracle_dequant.argtypes = [_P, _I64, _I64, _P, _P, _P, _P]
        lib.oracle_alltoall_quant_mm.argtypes = [_P, _INT, _I64, _I64, _INT, _INT, _P, _P, _P, _P,
                                                 _I64, _P, _I64, _P, _P, _P, _P]
        lib.oracle_matmul_reduce_scatter.argtypes = [_P, _P, _INT, _I64, _I64, _I64, _INT, _P, _INT, _P, _I64, _P]
        lib.oracle_num_threads.restype = _INT
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# --------------------------------------------------------------------------- helpers
def _is_bf16(dtype: torch.dtype) -> int:
    if dtype == torch.bfloat16:
        return 1
    if dtype == torch.float16:
        return 0
    raise TypeError(f"expected a bf16 or fp16 tensor, got {dtype}")


def _c(t: torch.Tensor) -> torch.Tensor:
    assert t.device.type == "cpu", "the oracle runs on CPU tensors only"
    return t.contiguous()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _ptr_array(ts: Sequence[torch.Tensor]):
    arr = (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])
    return arr


def _rows_arg(rows):
    if rows is None:
        return None, 0
    r = torch.as_tensor(rows, dtype=torch.int64).contiguous()
    return r, int(r.numel())


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


# --------------------------------------------------------------------------- conversions
def decode16(bits: torch.Tensor, is_bf16: bool) -> torch.Tensor:
    """int16/uint16 bit patterns -> exact float64 values."""
    b = _c(bits.view(torch.int16))
    out = torch.empty(b.shape, dtype=torch.float64)
    _load().oracle_decode16_array(b.data_ptr(), b.numel(), int(is_bf16), out.data_ptr())
    return out


def encode16(values: torch.Tensor, is_bf16: bool) -> torch.Tensor:
    """float64 values -> 16-bit tensor (bf16 or fp16), round to nearest even."""
    v = _c(values.to(torch.float64))
    out = torch.empty(v.shape, dtype=torch.int16)
    _load().oracle_encode16_array(v.data_ptr(), v.numel(), int(is_bf16), out.data_ptr())
    return out.view(torch.bfloat16 if is_bf16 else torch.float16)


# --------------------------------------------------------------------------- AllGatherMatmul
def gather(chunks: Sequence[torch.Tensor]) -> torch.Tensor:
    """AllGather along m of the per-rank shards, by explicit copy."""
    cs = [_c(c) for c in chunks]
    m_local, k = cs[0].shape
    out = torch.empty((len(cs) * m_local, k), dtype=cs[0].dtype)
    _check(_load().oracle_gather(_ptr_array(cs), len(cs), m_local, k, out.data_ptr()), "gather")
    return out


def all_gather_mm(chunks: Sequence[torch.Tensor], x2: torch.Tensor, *, x2_is_nk: bool = False,
                  bias: Optional[torch.Tensor] = None, rows=None, gather_output: bool = True):
    """out = AllGather_m(chunks) @ x2 (+ bias), rounded once; returns (out, gathered|None).

    With ``rows`` only those gathered rows of ``out`` are computed (in order).
    """
    cs = [_c(c) for c in chunks]
    dt = cs[0].dtype
    isb = _is_bf16(dt)
    m_local, k = cs[0].shape
    x2c = _c(x2)
    n = x2c.shape[0] if x2_is_nk else x2c.shape[1]
    b = None if bias is None else _c(bias.to(dt))
    r, nr = _rows_arg(rows)
    nrows = nr if r is not None else len(cs) * m_local
    out = torch.empty((nrows, n), dtype=dt)
    rc = _load().oracle_all_gather_mm(_ptr_array(cs), len(cs), m_local, k, x2c.data_ptr(), n,
                                      int(x2_is_nk), _ptr(b), isb, _ptr(r), nr, out.data_ptr())
    _check(rc, "all_gather_mm")
    return out, (gather(cs) if gather_output else None)


def matmul_reduce_scatter(x_chunks: Sequence[torch.Tensor], w_chunks: Sequence[torch.Tensor], *,
                          w_is_nk: bool = True, bias: Optional[torch.Tensor] = None, rows=None) -> torch.Tensor:
    """Y = ReduceScatter_m(sum_r X_r @ W_r^T): returns the (m, n) stack of the R
    ranks' outputs (rank j = rows [j*m/R, (j+1)*m/R)), or only ``rows`` of it."""
    xs = [_c(x) for x in x_chunks]
    ws = [_c(w) for w in w_chunks]
    dt = xs[0].dtype
    isb = _is_bf16(dt)
    m, k_local = xs[0].shape
    n = ws[0].shape[0] if w_is_nk else ws[0].shape[1]
    b = None if bias is None else _c(bias.to(dt))
    r, nr = _rows_arg(rows)
    out = torch.empty((nr if r is not None else m, n), dtype=dt)
    rc = _load().oracle_matmul_reduce_scatter(_ptr_array(xs), _ptr_array(ws), len(xs), m, k_local, n,
                                              int(w_is_nk), _ptr(b), isb, _ptr(r), nr, out.data_ptr())
    _check(rc, "matmul_reduce_scatter")
    return out


def matmul_weight_grad(dy: torch.Tensor, x: torch.Tensor, *, rows=None, with_bias: bool = True):
    """dW = dY^T @ X (n, k) (or only ``rows`` of it) and dB = sum_t dY[t, :] (n)
    or None; dY (m, n) and X (m, k) of one 16-bit type.  Returns (dw, db)."""
    d = _c(dy)
    xx = _c(x)
    m, n = d.shape
    k = xx.shape[1]
    isb = _is_bf16(d.dtype)
    r, nr = _rows_arg(rows)
    dw = torch.empty((nr if r is not None else n, k), dtype=d.dtype)
    db = torch.empty((n,), dtype=d.dtype) if with_bias else None
    rc = _load().oracle_matmul_weight_grad(d.data_ptr(), xx.data_ptr(), m, n, k, isb, _ptr(r), nr,
                                           dw.data_ptr(), _ptr(db))
    _check(rc, "matmul_weight_grad")
    return dw, db


# --------------------------------------------------------------------------- AlltoAllQuantMatmul
def comm_out(chunks: Sequence[torch.Tensor]) -> torch.Tensor:
    """commOut (R, BS/R, H): block r is the chunk received from rank r (the
    optional alltoAllOut output)."""
    cs = [_c(c) for c in chunks]
    bs_local, h = cs[0].shape
    out = torch.empty((len(cs), bs_local, h), dtype=cs[0].dtype)
    _check(_load().oracle_comm_out(_ptr_array(cs), len(cs), bs_local, h, cs[0].element_size(), out.data_ptr()),
           "comm_out")
    return out


def permute(chunks: Sequence[torch.Tensor], rows=None) -> torch.Tensor:
    """permutedOut[t, r*H + h] = chunk_r[t, h] for the requested rows t."""
    cs = [_c(c) for c in chunks]
    bs_local, h = cs[0].shape
    eb = cs[0].element_size()
    r, nr = _rows_arg(rows)
    nrows = nr if r is not None else bs_local
    out = torch.empty((nrows, len(cs) * h), dtype=cs[0].dtype)
    _check(_load().oracle_permute(_ptr_array(cs), len(cs), bs_local, h, eb, _ptr(r), nr,
                                  out.data_ptr()), "permute")
    return out


def quant_pertoken_dynamic(permuted: torch.Tensor, smooth: Optional[torch.Tensor] = None):
    """Per-token dynamic int8 quant: returns (q int8, x1_scale fp32)."""
    p = _c(permuted)
    isb = _is_bf16(p.dtype)
    rows, cols = p.shape
    s = None if smooth is None else _c(smooth.to(p.dtype))
    q = torch.empty((rows, cols), dtype=torch.int8)
    sc = torch.empty((rows,), dtype=torch.float32)
    _check(_load().oracle_quant_pertoken_dynamic(p.data_ptr(), rows, cols, _ptr(s), isb,
                                                 q.data_ptr(), sc.data_ptr()), "quant")
    return q, sc


def int8_mm(a: torch.Tensor, x2: torch.Tensor) -> torch.Tensor:
    """Exact int8 x int8 matmul, int32 result (error if a sum leaves int32)."""
    ac, bc = _c(a), _c(x2)
    rows, k = ac.shape
    n = bc.shape[1]
    acc = torch.empty((rows, n), dtype=torch.int32)
    _check(_load().oracle_int8_mm(ac.data_ptr(), rows, k, bc.data_ptr(), n, acc.data_ptr()), "int8_mm")
    return acc


def int8_mm_fp64(a: torch.Tensor, x2: torch.Tensor, col_block: int = 1024) -> torch.Tensor:
    """The same exact int8 matmul through an fp64 library matmul.

    Every product of two int8 values is an integer of magnitude <= 127*127 and
    every partial sum over k <= 35000 terms is an integer below 2^30, far inside
    the 2^53 range where fp64 represents integers exactly, so the result is
    exact whatever order the library sums in.  Used for large row sets.
    """
    ac = _c(a)
    bc = _c(x2)
    k = ac.shape[1]
    if k * 127 * 127 >= 2 ** 53:
        raise ValueError("k too large for an exact fp64 sum")
    ad = ac.double()
    out = torch.empty((ac.shape[0], bc.shape[1]), dtype=torch.int32)
    for j0 in range(0, bc.shape[1], col_block):
        blk = ad @ bc[:, j0:j0 + col_block].double()
        if blk.abs().max().item() > 2 ** 31 - 1:
            raise RuntimeError("oracle int8_mm: a result does not fit in int32")
        out[:, j0:j0 + col_block] = blk.to(torch.int32)
    return out


def dequant(acc: torch.Tensor, x1_scale: torch.Tensor, x2_scale: torch.Tensor,
            bias: Optional[torch.Tensor]) -> torch.Tensor:
    """bf16(((float(acc) * x1s[t]) * x2s[n]) + bias[n]) in fp32, one op at a time."""
    a = _c(acc)
    rows, n = a.shape
    s1, s2 = _c(x1_scale.float()), _c(x2_scale.float())
    b = None if bias is None else _c(bias.float())
    out = torch.empty((rows, n), dtype=torch.int16)
    _check(_load().oracle_dequant(a.data_ptr(), rows, n, s1.data_ptr(), s2.data_ptr(), _ptr(b),
                                  out.data_ptr()), "dequant")
    return out.view(torch.bfloat16)


def alltoall_quant_mm(chunks: Sequence[torch.Tensor], x2: torch.Tensor, x2_scale: torch.Tensor,
                      bias: Optional[torch.Tensor], *, quant_mode: int,
                      x1_scale: Optional[torch.Tensor] = None, rows=None) -> dict:
    """The whole AlltoAllQuantMatmul path for the requested permuted rows.

    quant_mode 7: chunks bf16/fp16, ``x1_scale`` = optional smooth scale (R*H).
    quant_mode 3: chunks int8, ``x1_scale`` = per-token fp32 scale (BS/R).
    Returns dict(out bf16, q int8, x1_scale fp32, acc int32) for those rows.
    """
    cs = [_c(c) for c in chunks]
    R = len(cs)
    bs_local, h = cs[0].shape
    x2c = _c(x2)
    n = x2c.shape[1]
    if quant_mode == 7:
        isb = _is_bf16(cs[0].dtype)
        s_in = None if x1_scale is None else _c(x1_scale.to(cs[0].dtype))
    elif quant_mode == 3:
        isb = 1
        s_in = _c(x1_scale.float())
    else:
        raise ValueError("quant_mode must be 3 or 7")
    r, nr = _rows_arg(rows)
    nrows = nr if r is not None else bs_local
    if nrows * R * h * n > (1 << 31):
        # large: the same steps, with the exact fp64 library matmul for the int8 product
        P = permute(cs, rows=r)
        if quant_mode == 7:
            q, sc = quant_pertoken_dynamic(P, s_in)
        else:
            q = P
            sc = s_in if r is None else s_in[r]
        acc = int8_mm_fp64(q, x2c)
        out = dequant(acc, sc, x2_scale, bias)
        return {"out": out, "q": q, "x1_scale": sc.clone(), "acc": acc}
    out = torch.empty((nrows, n), dtype=torch.int16)
    q = torch.empty((nrows, R * h), dtype=torch.int8)
    sc = torch.empty((nrows,), dtype=torch.float32)
    acc = torch.empty((nrows, n), dtype=torch.int32)
    b = None if bias is None else _c(bias.float())
    s2 = _c(x2_scale.float())
    rc = _load().oracle_alltoall_quant_mm(_ptr_array(cs), R, bs_local, h, quant_mode, isb, _ptr(s_in),
                                          x2c.data_ptr(), s2.data_ptr(), _ptr(b), n,
                                          _ptr(r), nr, out.data_ptr(), q.data_ptr(), sc.data_ptr(),
                                          acc.data_ptr())
    _check(rc, "alltoall_quant_mm")
    return {"out": out.view(torch.bfloat16), "q": q, "x1_scale": sc, "acc": acc}


# --------------------------------------------------------------------------- QuantAllReduce
X_KINDS = {"int8": 0, "e4m3": 1, "e5m2": 2}
SCALE_KINDS = {"fp32": 0, "e8m0": 1}
_OUT_KINDS = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}


def decode_fp8(code: int, fmt: str) -> float:
    """Value of one fp8 code ("e4m3" = E4M3FN, "e5m2")."""
    return _load().oracle_decode_fp8(code & 0xFF, 1 if fmt == "e5m2" else 0)


def decode_e8m0(code: int) -> float:
    return _load().oracle_decode_e8m0(code & 0xFF)


def quant_all_reduce(x_chunks: Sequence[torch.Tensor], scale_chunks: Sequence[torch.Tensor], *, x_kind: str,
                     scale_kind: str, out_dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """out = sum_r dequant(x_r, scales_r), (bs, h).  x_r: (bs, h) 1-byte codes
    (uint8/int8 tensors holding int8, e4m3fn or e5m2 bits); scales_r: fp32
    (bs, h/128) or e8m0 codes (bs, h/64, 2) as uint8."""
    xs = [_c(x).view(torch.uint8) for x in x_chunks]
    if scale_kind == "fp32":
        ss = [_c(s.float()) for s in scale_chunks]
    else:
        ss = [_c(s).view(torch.uint8) for s in scale_chunks]
    bs, h = xs[0].shape
    out = torch.empty((bs, h), dtype=out_dtype)
    rc = _load().oracle_quant_all_reduce(_ptr_array(xs), _ptr_array(ss), len(xs), bs, h, X_KINDS[x_kind],
                                         SCALE_KINDS[scale_kind], _OUT_KINDS[out_dtype], out.data_ptr())
    _check(rc, "quant_all_reduce")
    return out
