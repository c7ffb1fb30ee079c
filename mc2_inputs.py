"""Seeded synthetic inputs for the MC2 fused-linear workloads.

This module is shared by the tests, the benchmark and the smoke check.  It
holds shapes, value distributions and a fixed draw order, and none of the
method's arithmetic (no gather, permute, quant or matmul).  Everything is
drawn on the CPU with ``torch.Generator().manual_seed(seed)`` in this order:
the per-rank chunks r = 0 .. R-1, then x2 (or w), then the scales, then the
bias.  Callers copy the tensors to the device themselves.

Workloads (names used throughout the repository):

  ag-tiny    AllGatherMatmul, 8 ranks x (16, 512) fp16 ~N(0,1), x2 (512, 64)
             fp16 ~N(0,1), gathered output on.  Shapes of the example on the
             page "torch_npu.npu_all_gather_base_mm" (调用示例).
  ag-8x1024  AllGatherMatmul bf16, 8 ranks x (1024, 4096) ~N(0,1),
             x2 (4096, 4096) ~N(0, std k^-1/2), gathered output on, no bias.
  ag-4x4096  AllGatherMatmul bf16, 4 ranks x (4096, 8192) ~N(0,1), nn.Linear
             weight w (7168, 8192) ~N(0, std k^-1/2) passed as x2 = w^T,
             bias (7168) bf16 ~N(0, 0.02), gathered output on.
  a2a-dyn    AlltoAllQuantMatmul, quant mode 7 (per-token dynamic), 8 ranks x
             (4096, 1024) bf16 ~N(0,1) with 0.1% of elements x20, smooth scale
             (8192) bf16 ~U(0.5, 1.5), x2 int8 (8192, 4096) uniform on
             [-127, 127], x2 scale (4096) fp32 ~U(1e-3, 1e-2), bias (4096) fp32
             ~N(0, 0.1).
  a2a-dyn-small  the same with chunks (512, 1024).
  mmrs-4x2048  MatmulReduceScatter bf16, 4 ranks x activations (16384, 2048)
             ~N(0,1) and nn.Linear weight shards w_r (8192, 2048)
             ~N(0, std K^-1/2) with K = 8192 the unsharded contraction, no
             bias: the row-parallel dual of ag-4x4096.
  wgrad-ag-4x4096  weight/bias gradient of the ag-4x4096 layer: dY (16384, 7168)
             bf16 ~N(0, std m^-1/2) (the gradient of a token-mean loss, so that
             dW ~ N(0, 1)), gathered X (16384, 8192) bf16 ~N(0,1) -> dW (7168, 8192),
             dB (7168).
  qar-8x4096x8192  QuantAllReduce, 8 ranks x int8 (4096, 8192) uniform on
             [-127, 127] with pertoken-pergroup fp32 scales (4096, 64)
             ~U(1e-3, 1e-2), bf16 output.
  qar-mx-8x4096x8192  QuantAllReduce, 8 ranks x fp8 e4m3fn (4096, 8192) (values
             N(0, 64^2) cast to e4m3fn, saturated at +-448) with mx e8m0 scales
             (4096, 128, 2), codes uniform on [118, 134], bf16 output.
  a2a-full   AlltoAllQuantMatmul, quant mode 3 (pre-quantised int8), 8 ranks x
             (16384, 4096) int8 uniform on [-127, 127], per-token x1 scale
             (16384) fp32 ~U(1e-3, 1e-2), x2 int8 (32768, 7168), x2 scale
             (7168) fp32 ~U(1e-3, 1e-2), bias (7168) fp32 ~N(0, 0.1).
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class AGShape:
    world_size: int
    m_local: int
    k: int
    n: int
    dtype: torch.dtype = torch.bfloat16
    x2_is_nk: bool = False          # x2 given as the nn.Linear weight w (n, k)
    bias: bool = False
    gather_output: bool = True
    x_std: float = 1.0
    w_std: Optional[float] = None   # None: k ** -0.5
    bias_std: float = 0.02

    @property
    def m(self) -> int:
        return self.world_size * self.m_local

    @property
    def flops(self) -> float:
        return 2.0 * self.m * self.n * self.k


@dataclass(frozen=True)
class A2AShape:
    rank_size: int
    bs_local: int                   # BS / rankSize: rows of the permuted matrix
    h: int                          # hidden size of one received chunk
    n: int
    quant_mode: int                 # 7 per-token dynamic, 3 per-token (pre-quantised)
    x1_dtype: torch.dtype = torch.bfloat16   # for mode 7; mode 3 chunks are int8
    smooth: bool = True             # mode 7: pass the smooth scale x1ScaleOptional
    outlier_p: float = 0.001
    outlier_mult: float = 20.0
    bias: bool = True

    @property
    def k(self) -> int:
        return self.rank_size * self.h

    @property
    def ops(self) -> float:
        return 2.0 * self.bs_local * self.n * self.k


@dataclass(frozen=True)
class MMRSShape:
    world_size: int
    m: int                          # rows of every rank's activations (the scatter splits them)
    k_local: int                    # every rank's slice of the contraction
    n: int
    dtype: torch.dtype = torch.bfloat16
    w_is_nk: bool = True            # weight shards as nn.Linear w (n, k_local); else x2 = w^T
    bias: bool = False
    x_std: float = 1.0
    w_std: Optional[float] = None   # None: (world_size * k_local) ** -0.5
    bias_std: float = 0.02

    @property
    def k(self) -> int:
        return self.world_size * self.k_local

    @property
    def flops(self) -> float:
        return 2.0 * self.m * self.n * self.k


@dataclass(frozen=True)
class WGradShape:
    m: int                          # rows of dY and X: the contraction (all gathered tokens)
    n: int                          # output features (rows of dW)
    k: int                          # input features (columns of dW)
    dtype: torch.dtype = torch.bfloat16
    dy_std: Optional[float] = None  # None: m ** -0.5 (a token-mean loss), so dW ~ N(0, 1)
    x_std: float = 1.0

    @property
    def flops(self) -> float:
        return 2.0 * self.m * self.n * self.k


@dataclass(frozen=True)
class QARShape:
    world_size: int
    bs: int                         # tokens (b * s)
    h: int                          # hidden size, 128-aligned, [1024, 8192]
    x_kind: str = "int8"            # "int8" | "e4m3" | "e5m2"
    scale_kind: str = "fp32"        # "fp32": (bs, h/128) | "e8m0": (bs, h/64, 2)
    out_dtype: torch.dtype = torch.bfloat16

    @property
    def bytes(self) -> float:
        """Bytes the op must move: every rank's data and scales read once, the output written once."""
        sb = self.h // 128 * 4 if self.scale_kind == "fp32" else self.h // 32
        ob = torch.empty((), dtype=self.out_dtype).element_size()
        return float(self.bs) * (self.world_size * (self.h + sb) + self.h * ob)


WORKLOADS = {
    "ag-tiny": AGShape(world_size=8, m_local=16, k=512, n=64, dtype=torch.float16, w_std=1.0),
    "ag-8x1024": AGShape(world_size=8, m_local=1024, k=4096, n=4096),
    "ag-4x4096": AGShape(world_size=4, m_local=4096, k=8192, n=7168, x2_is_nk=True, bias=True),
    "a2a-dyn": A2AShape(rank_size=8, bs_local=4096, h=1024, n=4096, quant_mode=7),
    "a2a-dyn-small": A2AShape(rank_size=8, bs_local=512, h=1024, n=4096, quant_mode=7),
    "a2a-full": A2AShape(rank_size=8, bs_local=16384, h=4096, n=7168, quant_mode=3),
    "mmrs-4x2048": MMRSShape(world_size=4, m=16384, k_local=2048, n=8192),
    "wgrad-ag-4x4096": WGradShape(m=16384, n=7168, k=8192),
    "qar-8x4096x8192": QARShape(world_size=8, bs=4096, h=8192),
    "qar-mx-8x4096x8192": QARShape(world_size=8, bs=4096, h=8192, x_kind="e4m3", scale_kind="e8m0"),
}


def scaled(shape, **kw):
    """A copy of a workload shape with some fields changed (smaller test cases)."""
    return replace(shape, **kw)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def _randint8(g, shape):
    return torch.randint(-127, 128, shape, generator=g, dtype=torch.int8)


def ag_inputs(s: AGShape, seed: int = 0) -> dict:
    """chunks (list of R (m_local, k)), x2 ((k, n) or w (n, k)), bias (n) or None."""
    g = _gen(seed)
    chunks = [(torch.randn(s.m_local, s.k, generator=g) * s.x_std).to(s.dtype)
              for _ in range(s.world_size)]
    w_std = s.k ** -0.5 if s.w_std is None else s.w_std
    wshape = (s.n, s.k) if s.x2_is_nk else (s.k, s.n)
    x2 = (torch.randn(*wshape, generator=g) * w_std).to(s.dtype)
    bias = (torch.randn(s.n, generator=g) * s.bias_std).to(s.dtype) if s.bias else None
    return {"chunks": chunks, "x2": x2, "bias": bias}


def mmrs_inputs(s: MMRSShape, seed: int = 0) -> dict:
    """x_chunks (R x (m, k_local)), w_chunks (R x (n, k_local), or (k_local, n)
    when not w_is_nk), bias (n) or None."""
    g = _gen(seed)
    xs = [(torch.randn(s.m, s.k_local, generator=g) * s.x_std).to(s.dtype) for _ in range(s.world_size)]
    w_std = s.k ** -0.5 if s.w_std is None else s.w_std
    wshape = (s.n, s.k_local) if s.w_is_nk else (s.k_local, s.n)
    ws = [(torch.randn(*wshape, generator=g) * w_std).to(s.dtype) for _ in range(s.world_size)]
    bias = (torch.randn(s.n, generator=g) * s.bias_std).to(s.dtype) if s.bias else None
    return {"x_chunks": xs, "w_chunks": ws, "bias": bias}


def wgrad_inputs(s: WGradShape, seed: int = 0) -> dict:
    """dy (m, n), x (m, k)."""
    g = _gen(seed)
    dy_std = s.m ** -0.5 if s.dy_std is None else s.dy_std
    dy = (torch.randn(s.m, s.n, generator=g) * dy_std).to(s.dtype)
    x = (torch.randn(s.m, s.k, generator=g) * s.x_std).to(s.dtype)
    return {"dy": dy, "x": x}


def qar_inputs(s: QARShape, seed: int = 0) -> dict:
    """x_chunks: R x (bs, h) uint8 codes; scale_chunks: R x fp32 (bs, h/128) or
    R x uint8 e8m0 codes (bs, h/64, 2)."""
    g = _gen(seed)
    xs, ss = [], []
    for _ in range(s.world_size):
        if s.x_kind == "int8":
            xs.append(_randint8(g, (s.bs, s.h)).view(torch.uint8))
        elif s.x_kind == "e4m3":
            v = (torch.randn(s.bs, s.h, generator=g) * 64.0).clamp(-448.0, 448.0)
            xs.append(v.to(torch.float8_e4m3fn).view(torch.uint8))
        else:
            v = (torch.randn(s.bs, s.h, generator=g) * 1024.0).clamp(-57344.0, 57344.0)
            xs.append(v.to(torch.float8_e5m2).view(torch.uint8))
        if s.scale_kind == "fp32":
            ss.append(torch.rand(s.bs, s.h // 128, generator=g) * 9e-3 + 1e-3)
        else:
            ss.append(torch.randint(118, 135, (s.bs, s.h // 64, 2), generator=g, dtype=torch.uint8))
    return {"x_chunks": xs, "scale_chunks": ss}


def a2a_inputs(s: A2AShape, seed: int = 0) -> dict:
    """chunks (R x (bs_local, h)), x1_scale (smooth (R*h) or per-token (bs_local)),
    x2 int8 (R*h, n), x2_scale fp32 (n), bias fp32 (n) or None."""
    g = _gen(seed)
    chunks = []
    for _ in range(s.rank_size):
        if s.quant_mode == 7:
            v = torch.randn(s.bs_local, s.h, generator=g)
            hit = torch.rand(s.bs_local, s.h, generator=g) < s.outlier_p
            v = torch.where(hit, v * s.outlier_mult, v)
            chunks.append(v.to(s.x1_dtype))
        else:
            chunks.append(_randint8(g, (s.bs_local, s.h)))
    x2 = _randint8(g, (s.k, s.n))
    if s.quant_mode == 7:
        x1_scale = (torch.rand(s.k, generator=g) + 0.5).to(s.x1_dtype) if s.smooth else None
    else:
        x1_scale = torch.rand(s.bs_local, generator=g) * 9e-3 + 1e-3
    x2_scale = torch.rand(s.n, generator=g) * 9e-3 + 1e-3
    bias = torch.randn(s.n, generator=g) * 0.1 if s.bias else None
    return {"chunks": chunks, "x1_scale": x1_scale, "x2": x2, "x2_scale": x2_scale, "bias": bias}


def sample_rows(total: int, count: int, seed: int = 1) -> torch.Tensor:
    """A seeded subset of row indices (sorted) for checking very large outputs."""
    g = _gen(seed)
    count = min(count, total)
    return torch.sort(torch.randperm(total, generator=g)[:count]).values
