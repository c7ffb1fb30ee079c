"""GPU parity of mc2_quant_all_reduce (C ABI) against the CPU oracle.

"QuantAllReduce" (功能说明: output = Reduce(AllGather(scales) *
AllGather(x)), reduceOp sum; 参数说明: x int8 / fp8 e4m3fn / fp8 e5m2, scales
fp32 per token per group of 128 or e8m0 (bs, H/64, 2), output fp32 / fp16 /
bf16).

Tolerance, from the arithmetic: the oracle sums the exact products in fp64 and
rounds once; the kernel adds them in rank order with fp32 fused multiply-adds
(each step rounds once, |error| <= R * 2^-24 * sum_r |x_r s_r|) and then rounds
to the output type.  So |got - ref| <= ulp_out(max(|got|, |ref|)) +
R * 2^-24 * sum_r |x_r s_r|, with sum_r |x_r s_r| taken from the oracle run on
the absolute codes.  Where every partial sum is exact in fp32 (small integers
times powers of two, fp8 times e8m0 within range) the output is compared bit
for bit, and so are special codes (zeros, subnormals, infinities, NaN).
"""
import pytest
import torch

import mc2_inputs
import oracle
import quantized_gemm_rank_gb300 as mc2
from parity import assert_bits_equal

pytestmark = pytest.mark.gpu

S = mc2_inputs.QARShape
_PREC = {torch.float32: (24, -149), torch.float16: (11, -24), torch.bfloat16: (8, -133)}


def ulp(x: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    """Spacing of `dtype` values at |x| (x in float64): 2^(e - p) for |x| in
    [2^(e-1), 2^e), never below the smallest subnormal."""
    p, emin = _PREC[dtype]
    _, e = torch.frexp(x.abs())
    return torch.pow(2.0, (e.double() - p).clamp_min(emin))


def abs_codes(x: torch.Tensor, x_kind: str) -> torch.Tensor:
    if x_kind == "int8":
        return x.view(torch.int8).abs().view(torch.uint8)
    return x & 0x7F                                   # fp8: clear the sign bit


def run_gpu(inp, s, out_dtype):
    dev = torch.device("cuda")
    xs = [x.to(dev) for x in inp["x_chunks"]]
    ss = [sc.to(dev) for sc in inp["scale_chunks"]]
    out = mc2.mc2_quant_all_reduce(xs, ss, x_kind=s.x_kind, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert out.shape == (s.bs, s.h) and out.dtype == out_dtype
    return out.cpu()


def check(got, xs, ss, s, out_dtype, what):
    ref = oracle.quant_all_reduce(xs, ss, x_kind=s.x_kind, scale_kind=s.scale_kind, out_dtype=out_dtype)
    mag = oracle.quant_all_reduce([abs_codes(x, s.x_kind) for x in xs], ss, x_kind=s.x_kind,
                                  scale_kind=s.scale_kind, out_dtype=torch.float32).double()
    g, r = got.double(), ref.double()
    assert torch.isfinite(g).all() and torch.isfinite(r).all(), what
    tol = ulp(torch.maximum(g.abs(), r.abs()), out_dtype) + len(xs) * 2.0 ** -24 * mag * 1.0001
    err = (g - r).abs()
    bad = err > tol
    if bad.any():
        i = tuple(int(v) for v in bad.nonzero()[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {g.numel()} outside the bound; first at {i}: "
                             f"got {g[i].item():.9e} ref {r[i].item():.9e} tol {tol[i].item():.3e}")
    return ref


CASES = {
    "int8-fp32-r2-bf16": (S(world_size=2, bs=37, h=1024), torch.bfloat16),
    "int8-fp32-r4-fp16": (S(world_size=4, bs=5, h=1152), torch.float16),
    "int8-fp32-r8-fp32": (S(world_size=8, bs=19, h=1280), torch.float32),
    "e4m3-fp32-r8-bf16": (S(world_size=8, bs=23, h=2048, x_kind="e4m3"), torch.bfloat16),
    "e5m2-fp32-r4-fp32": (S(world_size=4, bs=9, h=1024, x_kind="e5m2"), torch.float32),
    "e5m2-fp32-r2-fp16": (S(world_size=2, bs=11, h=3072, x_kind="e5m2"), torch.float16),
    "e4m3-e8m0-r8-bf16": (S(world_size=8, bs=17, h=1024, x_kind="e4m3", scale_kind="e8m0"), torch.bfloat16),
    "e4m3-e8m0-r2-fp32": (S(world_size=2, bs=3, h=8192, x_kind="e4m3", scale_kind="e8m0"), torch.float32),
    "e5m2-e8m0-r4-bf16": (S(world_size=4, bs=13, h=1408, x_kind="e5m2", scale_kind="e8m0"), torch.bfloat16),
    "e5m2-e8m0-r8-fp32": (S(world_size=8, bs=1, h=1024, x_kind="e5m2", scale_kind="e8m0"), torch.float32),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_quant_all_reduce_parity(name):
    s, out_dtype = CASES[name]
    inp = mc2_inputs.qar_inputs(s, seed=21)
    got = run_gpu(inp, s, out_dtype)
    check(got, inp["x_chunks"], inp["scale_chunks"], s, out_dtype, name)


@pytest.mark.parametrize("x_kind", ["e4m3", "e5m2"])
def test_mx_fp16_out_within_range(x_kind):
    # e8m0 codes <= 127 keep every sum below the fp16 maximum
    s = S(world_size=4, bs=7, h=2048, x_kind=x_kind, scale_kind="e8m0")
    inp = mc2_inputs.qar_inputs(s, seed=22)
    inp["scale_chunks"] = [sc.clamp(max=127) for sc in inp["scale_chunks"]]
    got = run_gpu(inp, s, torch.float16)
    check(got, inp["x_chunks"], inp["scale_chunks"], s, torch.float16, x_kind)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_integer_data_power_of_two_scales_bit_exact(out_dtype):
    # |x| <= 6, scales 2^-2..2^1: every partial sum is exact in fp32 and the
    # result is exact in every output type
    g = torch.Generator().manual_seed(5)
    R, bs, h = 8, 29, 1152
    xs = [torch.randint(-6, 7, (bs, h), generator=g, dtype=torch.int8).view(torch.uint8) for _ in range(R)]
    ss = [torch.pow(2.0, torch.randint(-2, 2, (bs, h // 128), generator=g).float()) for _ in range(R)]
    s = S(world_size=R, bs=bs, h=h)
    got = run_gpu({"x_chunks": xs, "scale_chunks": ss}, s, out_dtype)
    ref = oracle.quant_all_reduce(xs, ss, x_kind="int8", scale_kind="fp32", out_dtype=out_dtype)
    assert_bits_equal(got, ref, f"int8 exact {out_dtype}")


@pytest.mark.parametrize("x_kind", ["e4m3", "e5m2"])
def test_special_codes(x_kind):
    # every fp8 code (zeros, subnormals, the largest finite, infinities, NaN)
    # on rank 0 times e8m0 scales spanning 2^-127 .. 2^0, rank 1 all zero:
    # each output is one exact product, compared bit for bit, NaN by position
    R, bs, h = 2, 4, 1024
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).repeat(bs * h // 256).view(bs, h)
    x0 = codes
    x1 = torch.zeros(bs, h, dtype=torch.uint8)
    sc = torch.tensor([[(0, 1, 100, 127)[t] for _ in range(h // 32)] for t in range(bs)],
                      dtype=torch.uint8).view(bs, h // 64, 2)
    s = S(world_size=R, bs=bs, h=h, x_kind=x_kind, scale_kind="e8m0")
    got = run_gpu({"x_chunks": [x0, x1], "scale_chunks": [sc, sc]}, s, torch.float32)
    ref = oracle.quant_all_reduce([x0, x1], [sc, sc], x_kind=x_kind, scale_kind="e8m0", out_dtype=torch.float32)
    gn, rn = torch.isnan(got), torch.isnan(ref)
    assert torch.equal(gn, rn), "NaN positions differ"
    assert_bits_equal(torch.where(gn, 0.0, got), torch.where(rn, 0.0, ref), f"{x_kind} special codes")


def test_e8m0_nan_scale():
    R, bs, h = 2, 2, 1024
    x = torch.full((bs, h), 0x38, dtype=torch.uint8)                 # e4m3 1.0
    sc = torch.full((bs, h // 64, 2), 127, dtype=torch.uint8)
    sc[1, 3, 1] = 255                                                # NaN scale for columns 224..255 of row 1
    s = S(world_size=R, bs=bs, h=h, x_kind="e4m3", scale_kind="e8m0")
    got = run_gpu({"x_chunks": [x, x], "scale_chunks": [sc, sc]}, s, torch.bfloat16).float()
    nan = torch.isnan(got)
    assert nan[1, 224:256].all() and int(nan.sum()) == 32
    assert (got[~nan] == 2.0).all()


@pytest.mark.parametrize("name", ["qar-8x4096x8192", "qar-mx-8x4096x8192"])
def test_full_workload_sampled_rows(name):
    s = mc2_inputs.WORKLOADS[name]
    inp = mc2_inputs.qar_inputs(s, seed=0)
    got = run_gpu(inp, s, s.out_dtype)
    rows = mc2_inputs.sample_rows(s.bs, 96, seed=1)
    sub = S(world_size=s.world_size, bs=len(rows), h=s.h, x_kind=s.x_kind, scale_kind=s.scale_kind)
    check(got[rows], [x[rows] for x in inp["x_chunks"]], [sc[rows] for sc in inp["scale_chunks"]], sub,
          s.out_dtype, name)


def test_three_dim_input_and_stream():
    # a (b, s, h) tensor is the (b*s, h) problem; the call runs on the given stream
    s = S(world_size=4, bs=2 * 24, h=1024)
    inp = mc2_inputs.qar_inputs(s, seed=23)
    dev = torch.device("cuda")
    xs = [x.view(2, 24, 1024).view(torch.int8).to(dev) for x in inp["x_chunks"]]
    ss = [sc.view(2, 24, 8).to(dev) for sc in inp["scale_chunks"]]
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        out = mc2.mc2_quant_all_reduce(xs, ss, out_dtype=torch.float32, stream=st)
    st.synchronize()
    assert out.shape == (2, 24, 1024)
    check(out.cpu().view(48, 1024), inp["x_chunks"], inp["scale_chunks"], s, torch.float32, "3-d")
