"""GB300 (sm_103a) MC2 fused linears: Python binding of the C ABI in
``include/mc2_gb300.h``.

Argument marshalling only: every step of both operations runs in the CUDA
library ``libmc2_gb300.so`` (built in-tree by :mod:`.build`).  PyTorch
provides device memory and streams.  There is no CPU fallback: if the library
cannot be built or loaded, importing the functions raises.

  mc2_all_gather_mm        out = concat_m(x_chunks) @ x2 (+ bias), plus gathered
  mc2_alltoall_quant_mm    out = (Quant(permute(chunks)) @ x2) * x1s * x2s + bias
  mc2_matmul_reduce_scatter  out_j = (sum_r X_r @ W_r^T)[rows of rank j] (+ bias)
  mc2_matmul_weight_grad   dw = dy^T @ x, db = dy.sum(0)
  mc2_quant_all_reduce     out = sum_r dequant(x_r, scales_r)  (int8/fp8 codes)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from . import build as _build

MC2_OK = 0
MC2_ERR_NULL = -1
MC2_ERR_SHAPE = -2
MC2_ERR_DTYPE = -3
MC2_ERR_UNSUPPORTED = -4
MC2_ERR_WORKSPACE = -5
MC2_ERR_CUDA = -6
MC2_ERR_TIMEOUT = -7

MC2_F16, MC2_BF16, MC2_F32, MC2_I8 = 1, 2, 3, 4
MC2_F8E4M3, MC2_F8E5M2, MC2_E8M0 = 5, 6, 7
QUANT_PERCHANNEL = 2
QUANT_PERTOKEN = 3
QUANT_PERTOKEN_DYNAMIC = 7

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_lib = None


class Mc2Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_str(status)}: {message}")
        self.status = status
        self.message = message


def lib() -> ctypes.CDLL:
    """Load (building first if the sources changed) the CUDA library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.mc2_all_gather_mm.argtypes = [_P, _INT, _I64, _I64, _P, _I64, _INT, _P, _INT, _INT, _P, _P, _P]
        L.mc2_all_gather_mm.restype = _INT
        L.mc2_matmul_reduce_scatter.argtypes = [_P, _P, _INT, _I64, _I64, _I64, _INT, _P, _INT, _P, _P]
        L.mc2_matmul_reduce_scatter.restype = _INT
        L.mc2_matmul_weight_grad.argtypes = [_P, _I64, _I64, _P, _I64, _INT, _P, _P, _P]
        L.mc2_matmul_weight_grad.restype = _INT
        L.mc2_quant_all_reduce.argtypes = [_P, _P, _INT, _I64, _I64, _INT, _INT, _INT, _P, _P]
        L.mc2_quant_all_reduce.restype = _INT
        L.mc2_alltoall_quant_mm_workspace.argtypes = [_INT, _I64, _I64, _I64, _INT, _INT,
                                                      ctypes.POINTER(ctypes.c_size_t)]
        L.mc2_alltoall_quant_mm_workspace.restype = _INT
        L.mc2_alltoall_quant_mm.argtypes = [_P, _INT, _I64, _I64, _INT, _P, _P, _P, _P, _INT, _INT, _INT, _I64,
                                            _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
        L.mc2_alltoall_quant_mm.restype = _INT
        L.mc2_alltoall_quant_mm_no_alloc.argtypes = [_P, _INT, _I64, _I64, _INT, _P, _P, _P, _P, _INT, _INT, _INT,
                                                     _I64, _P, _P, _P, _P, _P, _P]
        L.mc2_alltoall_quant_mm_no_alloc.restype = _INT
        L.mc2_status_str.argtypes = [_INT]
        L.mc2_status_str.restype = ctypes.c_char_p
        L.mc2_last_error.argtypes = []
        L.mc2_last_error.restype = ctypes.c_char_p
        L.mc2_device_status.argtypes = []
        L.mc2_device_status.restype = _INT
        L.mc2_set_launch_events.argtypes = [_P, _INT]
        L.mc2_set_launch_events.restype = _INT
        L.mc2_test_expire_next_flag_waits.argtypes = [ctypes.c_uint64]
        L.mc2_test_expire_next_flag_waits.restype = _INT
        _lib = L
    return _lib


def library_path() -> str:
    return _build.LIB


def status_str(status: int) -> str:
    return lib().mc2_status_str(status).decode()


def last_error() -> str:
    return lib().mc2_last_error().decode()


def _check(status: int):
    if status != MC2_OK:
        raise Mc2Error(status, last_error())


_DTYPE_CODES = {torch.float16: MC2_F16, torch.bfloat16: MC2_BF16, torch.float32: MC2_F32, torch.int8: MC2_I8}


def _dtype_code(dt: torch.dtype) -> int:
    if dt not in _DTYPE_CODES:
        raise ValueError(f"unsupported dtype {dt}")
    return _DTYPE_CODES[dt]


def _current_device() -> int:
    """The CUDA device the library launches on, or -1 without CUDA."""
    return torch.cuda.current_device() if torch.cuda.is_available() else -1


# Every tensor goes to the library as a bare pointer, and its kernels trust the
# sizes passed beside it, so each tensor is checked first against the shape
# and dtype those sizes imply (a smaller buffer would be read or written past
# its end), against the current device (the library launches there: a tensor
# elsewhere would reach its kernels as a foreign pointer) and for contiguity.
# Without CUDA the device is -1, which a CPU tensor also reports: shape and
# dtype mistakes are then still reported first, and _need_device refuses the
# call before the library is reached.

def _refuse(t: torch.Tensor, shape, dtype, what: str, cur: int):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{what} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{what} must be of dtype {dtype}, got {t.dtype}")
    if cur < 0 or t.get_device() != cur:
        where = "a CUDA device (none is available)" if cur < 0 else f"the current device (cuda:{cur})"
        raise ValueError(f"{what} must be a CUDA tensor on {where}")
    raise ValueError(f"{what} must be contiguous")


def _arg(t: torch.Tensor, shape, dtype, what: str, cur: int) -> int:
    """The tensor's device pointer, once its shape, dtype, device and layout are right."""
    if t.shape != shape or t.dtype != dtype or t.get_device() != cur or not t.is_contiguous():
        _refuse(t, shape, dtype, what, cur)
    return t.data_ptr()


def _opt(t: Optional[torch.Tensor], shape, dtype, what: str, cur: int) -> Optional[int]:
    return None if t is None else _arg(t, shape, dtype, what, cur)


def _args(ts: Sequence[torch.Tensor], shape, dtype, what: str, cur: int):
    """A C array of the tensors' pointers, each checked as by _arg."""
    if len(ts) == 0:
        raise ValueError(f"{what} is empty")
    ptrs = []
    for t in ts:
        if t.shape != shape or t.dtype != dtype or t.get_device() != cur or not t.is_contiguous():
            _refuse(t, shape, dtype, f"{what}[{len(ptrs)}]", cur)
        ptrs.append(t.data_ptr())
    return (ctypes.c_void_p * len(ptrs))(*ptrs)


def _need_device(cur: int) -> None:
    if cur < 0:
        raise ValueError("the tensors must be CUDA tensors on the current device, and no CUDA device is available")


_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, cur: int) -> Optional[int]:
    if stream is None:
        if _raw_current_stream is not None:
            # the current stream's handle without building a Stream object (a call's
            # largest single piece of Python-side work)
            return _raw_current_stream(cur)
        stream = torch.cuda.current_stream()
    elif stream.device_index != cur:
        raise ValueError(f"stream must belong to the current device (cuda:{cur})")
    return stream.cuda_stream


def mc2_all_gather_mm(x_chunks: Sequence[torch.Tensor], x2: torch.Tensor, *, x2_is_nk: bool = False,
                      bias: Optional[torch.Tensor] = None, gather_output: bool = True,
                      out: Optional[torch.Tensor] = None, gathered: Optional[torch.Tensor] = None,
                      stream=None):
    """AllGatherMatmul on the rank chunks already resident on this GPU.

    x_chunks: world_size tensors (m_local, k); x2 (k, n), or w (n, k) with
    ``x2_is_nk``.  Returns (out (m, n), gathered (m, k) or None).
    """
    cur = _current_device()
    R = len(x_chunks)
    m_local, k = x_chunks[0].shape
    n = x2.shape[0] if x2_is_nk else x2.shape[1]
    dt = x_chunks[0].dtype
    ptrs = _args(x_chunks, (m_local, k), dt, "x_chunks", cur)
    x2p = _arg(x2, (n, k) if x2_is_nk else (k, n), dt, "x2", cur)
    bp = _opt(bias, (n,), dt, "bias", cur)
    if out is None:
        out = torch.empty((R * m_local, n), dtype=dt, device=x_chunks[0].device)
    outp = _arg(out, (R * m_local, n), dt, "out", cur)
    gp = None
    if gather_output:
        if gathered is None:
            gathered = torch.empty((R * m_local, k), dtype=dt, device=x_chunks[0].device)
        gp = _arg(gathered, (R * m_local, k), dt, "gathered", cur)
    _need_device(cur)
    st = lib().mc2_all_gather_mm(ptrs, R, m_local, k, x2p, n, int(x2_is_nk), bp, _dtype_code(dt), int(gather_output),
                                 outp, gp, _stream(stream, cur))
    _check(st)
    return out, (gathered if gather_output else None)


def mc2_matmul_reduce_scatter(x_chunks: Sequence[torch.Tensor], w_chunks: Sequence[torch.Tensor], *,
                              w_is_nk: bool = True, bias: Optional[torch.Tensor] = None,
                              out_chunks: Optional[Sequence[torch.Tensor]] = None, stream=None):
    """MatmulReduceScatter on the ranks' shards already resident on this GPU.

    x_chunks: world_size tensors (m, k_local); w_chunks: world_size weight shards
    (n, k_local) (or (k_local, n) with ``w_is_nk=False``).  Returns the list of
    the ranks' outputs, each (m / world_size, n).
    """
    cur = _current_device()
    R = len(x_chunks)
    m, k_local = x_chunks[0].shape
    n = w_chunks[0].shape[0] if w_is_nk else w_chunks[0].shape[1]
    dt = x_chunks[0].dtype
    if len(w_chunks) != R:
        raise ValueError(f"w_chunks must hold {R} shards (one per rank), got {len(w_chunks)}")
    if out_chunks is not None and len(out_chunks) != R:
        raise ValueError(f"out_chunks must hold {R} outputs (one per rank), got {len(out_chunks)}")
    xp = _args(x_chunks, (m, k_local), dt, "x_chunks", cur)
    wp = _args(w_chunks, (n, k_local) if w_is_nk else (k_local, n), dt, "w_chunks", cur)
    bp = _opt(bias, (n,), dt, "bias", cur)
    if out_chunks is None:
        out_chunks = [torch.empty((m // R, n), dtype=dt, device=x_chunks[0].device) for _ in range(R)]
    op = _args(out_chunks, (m // R, n), dt, "out_chunks", cur)
    _need_device(cur)
    st = lib().mc2_matmul_reduce_scatter(xp, wp, R, m, k_local, n, int(w_is_nk), bp, _dtype_code(dt), op,
                                         _stream(stream, cur))
    _check(st)
    return list(out_chunks)


def mc2_matmul_weight_grad(dy: torch.Tensor, x: torch.Tensor, *, with_bias: bool = True,
                           dw: Optional[torch.Tensor] = None, db: Optional[torch.Tensor] = None, stream=None):
    """dW = dY^T @ X (n, k) and, with ``with_bias``, dB = dY.sum(0) (n).

    dy (m, n) and x (m, k) of one 16-bit type on this GPU (for the all-gather
    layer, x is the ``gathered`` output of its forward call).  Returns (dw, db).
    """
    cur = _current_device()
    m, n = dy.shape
    k = x.shape[1]
    dt = dy.dtype
    dyp = _arg(dy, (m, n), dt, "dy", cur)
    xp = _arg(x, (m, k), dt, "x", cur)
    if dw is None:
        dw = torch.empty((n, k), dtype=dt, device=dy.device)
    dwp = _arg(dw, (n, k), dt, "dw", cur)
    dbp = None
    if with_bias:
        if db is None:
            db = torch.empty((n,), dtype=dt, device=dy.device)
        dbp = _arg(db, (n,), dt, "db", cur)
    _need_device(cur)
    st = lib().mc2_matmul_weight_grad(dyp, m, n, xp, k, _dtype_code(dt), dwp, dbp, _stream(stream, cur))
    _check(st)
    return dw, (db if with_bias else None)


_QAR_X = {"int8": MC2_I8, "e4m3": MC2_F8E4M3, "e5m2": MC2_F8E5M2}
_QAR_X_BY_DTYPE = {torch.int8: "int8", torch.float8_e4m3fn: "e4m3", torch.float8_e5m2: "e5m2"}


def mc2_quant_all_reduce(x_chunks: Sequence[torch.Tensor], scale_chunks: Sequence[torch.Tensor], *,
                         x_kind: Optional[str] = None, out_dtype: torch.dtype = torch.bfloat16,
                         out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """QuantAllReduce of the ranks' quantised shards resident on this GPU.

    x_chunks: world_size tensors (bs, h) or (b, s, h) of one-byte codes: int8,
    float8_e4m3fn or float8_e5m2 (or uint8 with ``x_kind`` "int8" | "e4m3" |
    "e5m2").  scale_chunks: fp32 (bs, h/128) per-token-per-group scales, or e8m0
    codes (bs, h/64, 2) as uint8 (mx).  Returns out of the same leading shape
    as x in ``out_dtype`` (fp32, fp16 or bf16).
    """
    cur = _current_device()
    x0 = x_chunks[0]
    if x_kind is None:
        if x0.dtype not in _QAR_X_BY_DTYPE:
            raise ValueError("x_kind is required for x of dtype %s" % x0.dtype)
        x_kind = _QAR_X_BY_DTYPE[x0.dtype]
    h = x0.shape[-1]
    bs = x0.numel() // h
    if len(scale_chunks) != len(x_chunks):
        raise ValueError(f"scale_chunks must hold {len(x_chunks)} tensors (one per rank), got {len(scale_chunks)}")
    xp = _args(x_chunks, x0.shape, x0.dtype, "x_chunks", cur)
    s0 = scale_chunks[0]
    sdt = MC2_F32 if s0.dtype == torch.float32 else MC2_E8M0
    # fp32: one scale per token per 128 elements, any shape; e8m0: one uint8 code per 32
    sdtype = torch.float32 if sdt == MC2_F32 else torch.uint8
    if h % 128 == 0:
        count = bs * (h // 128 if sdt == MC2_F32 else h // 32)
        for i, sc in enumerate(scale_chunks):
            if sc.numel() != count or sc.dtype != sdtype:
                raise ValueError(f"scale_chunks[{i}] must hold {count} "
                                 f"{'fp32 scales' if sdt == MC2_F32 else 'e8m0 codes (uint8)'}, "
                                 f"got {sc.numel()} of {sc.dtype}")
    sp = _args(scale_chunks, s0.shape, sdtype, "scale_chunks", cur)
    if out is None:
        out = torch.empty(x0.shape, dtype=out_dtype, device=x0.device)
    outp = _arg(out, x0.shape, out_dtype, "out", cur)
    _need_device(cur)
    st = lib().mc2_quant_all_reduce(xp, sp, len(x_chunks), bs, h, _QAR_X[x_kind], sdt, _dtype_code(out.dtype),
                                    outp, _stream(stream, cur))
    _check(st)
    return out


def mc2_alltoall_quant_mm_workspace(rank_size: int, bs_local: int, h: int, n: int, x1_quant_mode: int,
                                    x1_dtype: torch.dtype) -> int:
    nbytes = ctypes.c_size_t(0)
    _check(lib().mc2_alltoall_quant_mm_workspace(rank_size, bs_local, h, n, x1_quant_mode, _dtype_code(x1_dtype),
                                                 ctypes.byref(nbytes)))
    return int(nbytes.value)


def _a2a_args(chunks, x2, x2_scale, bias, x1_quant_mode, x1_scale, out, q_out, x1_scale_out, acc_out,
              alltoall_out, cur: int) -> list:
    """The pointers of an AlltoAllQuantMatmul call, each tensor checked against
    the sizes of the first chunk and of x2 (the quant modes and the 16-bit /
    int8 choice are the library's to refuse)."""
    R = len(chunks)
    bs_local, h = chunks[0].shape
    K = R * h
    n = x2.shape[1]
    x1_dtype = chunks[0].dtype
    if bias.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"bias must be of dtype torch.float32 or torch.bfloat16, got {bias.dtype}")
    if x1_quant_mode == QUANT_PERTOKEN:
        x1p = _opt(x1_scale, (bs_local,), torch.float32, "x1_scale (per-token scale)", cur)
    else:
        x1p = _opt(x1_scale, (K,), x1_dtype, "x1_scale (smooth scale)", cur)
    return [_args(chunks, (bs_local, h), x1_dtype, "chunks", cur), x1p,
            _arg(x2, (K, n), torch.int8, "x2", cur),
            _arg(x2_scale, (n,), torch.float32, "x2_scale", cur),
            _arg(bias, (n,), bias.dtype, "bias", cur),
            _arg(out, (bs_local, n), torch.bfloat16, "out", cur),
            _opt(alltoall_out, (R, bs_local, h), x1_dtype, "alltoall_out", cur),
            _opt(q_out, (bs_local, K), torch.int8, "q_out", cur),
            _opt(x1_scale_out, (bs_local,), torch.float32, "x1_scale_out", cur),
            _opt(acc_out, (bs_local, n), torch.int32, "acc_out", cur)]


def mc2_alltoall_quant_mm(chunks: Sequence[torch.Tensor], x2: torch.Tensor, x2_scale: torch.Tensor,
                          bias: torch.Tensor, *, x1_quant_mode: int, x1_scale: Optional[torch.Tensor] = None,
                          x2_quant_mode: int = QUANT_PERCHANNEL, out: Optional[torch.Tensor] = None,
                          q_out: Optional[torch.Tensor] = None, x1_scale_out: Optional[torch.Tensor] = None,
                          acc_out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                          alltoall_out: Optional[torch.Tensor] = None, stream=None) -> dict:
    """AlltoAllQuantMatmul on the received chunks already resident on this GPU.

    chunks: rank_size tensors (bs_local, h) (bf16/fp16 for mode 7, int8 for
    mode 3); x2 int8 (rank_size*h, n); x2_scale fp32 (n); bias fp32/bf16 (n).
    alltoall_out: optional (rank_size, bs_local, h) tensor of the chunks' dtype
    that receives commOut (the chunks stacked, before the permute).
    Returns dict(out, q, x1_scale, acc, alltoall_out) with the optional outputs
    that were given.
    """
    cur = _current_device()
    R = len(chunks)
    bs_local, h = chunks[0].shape
    n = x2.shape[1]
    dev = chunks[0].device
    x1_dtype = chunks[0].dtype
    if out is None:
        out = torch.empty((bs_local, n), dtype=torch.bfloat16, device=dev)
    a = _a2a_args(chunks, x2, x2_scale, bias, x1_quant_mode, x1_scale, out, q_out, x1_scale_out, acc_out,
                  alltoall_out, cur)
    _need_device(cur)
    if workspace is None:
        need = mc2_alltoall_quant_mm_workspace(R, bs_local, h, n, x1_quant_mode, x1_dtype)
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wp = _arg(workspace, workspace.shape, workspace.dtype, "workspace", cur)
    st = lib().mc2_alltoall_quant_mm(a[0], R, bs_local, h, _dtype_code(x1_dtype), a[1], a[2], a[3], a[4],
                                     _dtype_code(bias.dtype), x1_quant_mode, x2_quant_mode, n, a[5], a[6], a[7],
                                     a[8], a[9], wp, workspace.numel() * workspace.element_size(),
                                     _stream(stream, cur))
    _check(st)
    return {"out": out, "q": q_out, "x1_scale": x1_scale_out, "acc": acc_out, "alltoall_out": alltoall_out}


NO_ALLOC_SCRATCH_BYTES = 32 << 20


def mc2_alltoall_quant_mm_no_alloc(chunks: Sequence[torch.Tensor], x2: torch.Tensor, x2_scale: torch.Tensor,
                                   bias: torch.Tensor, *, x1_quant_mode: int, out: torch.Tensor,
                                   x1_scale: Optional[torch.Tensor] = None, x2_quant_mode: int = QUANT_PERCHANNEL,
                                   q_out: Optional[torch.Tensor] = None, x1_scale_out: Optional[torch.Tensor] = None,
                                   acc_out: Optional[torch.Tensor] = None, alltoall_out: Optional[torch.Tensor] = None,
                                   stream=None) -> dict:
    """The same computation as mc2_alltoall_quant_mm without a workspace.

    For callers that cannot allocate device memory: the library's built-in
    scratch (NO_ALLOC_SCRATCH_BYTES per GPU) is used instead, so problems whose
    workspace would exceed it are refused.  ``out`` must be given (nothing is
    allocated here).  Calls that may overlap on the GPU share that scratch and
    must be serialised by the caller.
    """
    cur = _current_device()
    if out is None:
        raise ValueError("out must be given (this entry point allocates nothing)")
    R = len(chunks)
    bs_local, h = chunks[0].shape
    n = x2.shape[1]
    a = _a2a_args(chunks, x2, x2_scale, bias, x1_quant_mode, x1_scale, out, q_out, x1_scale_out, acc_out,
                  alltoall_out, cur)
    _need_device(cur)
    st = lib().mc2_alltoall_quant_mm_no_alloc(a[0], R, bs_local, h, _dtype_code(chunks[0].dtype), a[1], a[2], a[3],
                                              a[4], _dtype_code(bias.dtype), x1_quant_mode, x2_quant_mode, n, a[5],
                                              a[6], a[7], a[8], a[9], _stream(stream, cur))
    _check(st)
    return {"out": out, "q": q_out, "x1_scale": x1_scale_out, "acc": acc_out, "alltoall_out": alltoall_out}


def mc2_device_status() -> int:
    """Synchronise and return (and clear) the kernels' bounded-wait status."""
    return int(lib().mc2_device_status())


def mc2_set_launch_events(events: Optional[Sequence["torch.cuda.Event"]]) -> None:
    """Record the given CUDA events around the kernel launches of the next calls
    on this host thread: events[0] before a call's first launch, events[i]
    after its i-th (see the header for each call's launches).  None or [] turns
    it off.  The events must be created with timing enabled and stay alive
    while set."""
    evs = list(events or [])
    handles = [e.cuda_event for e in evs]
    if any(h == 0 for h in handles):
        raise ValueError("record each event once (or create it) before installing it")
    arr = (ctypes.c_void_p * max(1, len(handles)))(*handles) if handles else None
    _check(lib().mc2_set_launch_events(arr, len(handles)))


def mc2_test_expire_next_flag_waits(wait_limit_ns: int) -> None:
    """Test hook: the next AlltoAllQuantMatmul call on this host thread runs its
    GEMM with every stream-K finishing wait set to run out after
    ``wait_limit_ns`` (see the header)."""
    _check(lib().mc2_test_expire_next_flag_waits(int(wait_limit_ns)))


__all__ = [
    "Mc2Error", "lib", "library_path", "status_str", "last_error", "mc2_all_gather_mm",
    "mc2_matmul_reduce_scatter", "mc2_matmul_weight_grad", "mc2_quant_all_reduce",
    "mc2_alltoall_quant_mm_workspace", "mc2_alltoall_quant_mm",
    "mc2_alltoall_quant_mm_no_alloc",
    "NO_ALLOC_SCRATCH_BYTES", "mc2_device_status", "mc2_set_launch_events", "mc2_test_expire_next_flag_waits",
    "MC2_OK", "MC2_ERR_NULL", "MC2_ERR_SHAPE", "MC2_ERR_DTYPE", "MC2_ERR_UNSUPPORTED", "MC2_ERR_WORKSPACE",
    "MC2_ERR_CUDA", "MC2_ERR_TIMEOUT", "MC2_F16", "MC2_BF16", "MC2_F32", "MC2_I8",
    "MC2_F8E4M3", "MC2_F8E5M2", "MC2_E8M0",
    "QUANT_PERCHANNEL", "QUANT_PERTOKEN", "QUANT_PERTOKEN_DYNAMIC",
]
