"""Pins for the QuantAllReduce oracle ("QuantAllReduce", 功能说明:
output = Reduce(AllGather(scales) * AllGather(x)), reduceOp sum; 参数说明 /
约束说明: int8 or fp8 data, pertoken-pergroup fp32 scales (group 128) or mx
e8m0 scales (bs, H/64, 2)).

* fp8 decoding: every one of the 256 codes of e4m3fn and e5m2 against torch's
  float8 dtypes (an independent library routine), plus hand-checked values
* e8m0: 2^(e - 127) for every finite code, NaN for 0xFF
* the group index: a one-hot x picks out exactly the scale of its group, at
  every group boundary, for both scale layouts
* integer data with power-of-two scales: the exact sum over ranks (Python
  loops) bit for bit, for each output dtype
* one rank is a plain dequant (torch fp64 on the expanded scales)
"""
import math

import pytest
import torch

import mc2_inputs
import oracle


@pytest.mark.parametrize("fmt,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_fp8_decode_all_codes(fmt, tdt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(tdt).to(torch.float64)
    for c in range(256):
        got = oracle.decode_fp8(c, fmt)
        want = ref[c].item()
        if math.isnan(want):
            assert math.isnan(got), (fmt, c)
        else:
            assert got == want, (fmt, c, got, want)


def test_fp8_decode_hand_values():
    assert oracle.decode_fp8(0x7E, "e4m3") == 448.0                # largest finite e4m3fn
    assert oracle.decode_fp8(0x01, "e4m3") == 2.0 ** -9             # smallest subnormal
    assert oracle.decode_fp8(0x38, "e4m3") == 1.0
    assert math.isnan(oracle.decode_fp8(0x7F, "e4m3"))
    assert oracle.decode_fp8(0x7B, "e5m2") == 57344.0               # largest finite e5m2
    assert oracle.decode_fp8(0x7C, "e5m2") == math.inf
    assert oracle.decode_fp8(0x01, "e5m2") == 2.0 ** -16
    assert oracle.decode_fp8(0xBC, "e5m2") == -1.0


def test_e8m0_decode():
    for e in range(255):
        assert oracle.decode_e8m0(e) == 2.0 ** (e - 127)
    assert math.isnan(oracle.decode_e8m0(255))


@pytest.mark.parametrize("scale_kind,G", [("fp32", 128), ("e8m0", 32)])
def test_group_index_one_hot(scale_kind, G):
    bs, h = 2, 1024
    groups = h // G
    if scale_kind == "fp32":
        sc = torch.tensor([[float(2 ** (g % 20)) * (1 + t) for g in range(groups)] for t in range(bs)])
        sval = lambda t, g: sc[t, g].item()  # noqa: E731
        x_kind, one = "int8", 1
    else:
        codes = torch.tensor([[100 + g for g in range(groups)] for t in range(bs)], dtype=torch.uint8)
        sc = codes.view(bs, h // 64, 2)
        sval = lambda t, g: 2.0 ** (100 + g - 127)  # noqa: E731
        x_kind, one = "e4m3", 0x38                      # e4m3 code of 1.0
    for j in [0, G - 1, G, 2 * G - 1, h - G, h - 1, 5 * G + 7]:
        t = j % bs
        x = torch.zeros(bs, h, dtype=torch.uint8)
        x[t, j] = one
        out = oracle.quant_all_reduce([x, torch.zeros_like(x)], [sc, sc], x_kind=x_kind, scale_kind=scale_kind,
                                      out_dtype=torch.float32)
        want = torch.zeros(bs, h, dtype=torch.float32)
        want[t, j] = sval(t, j // G)
        assert torch.equal(out, want), j


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_integer_sum_over_ranks_exact(out_dtype):
    g = torch.Generator().manual_seed(3)
    R, bs, h = 4, 3, 256
    xs = [torch.randint(-6, 7, (bs, h), generator=g, dtype=torch.int8) for _ in range(R)]
    ss = [torch.tensor([[2.0 ** int(torch.randint(-2, 2, (1,), generator=g)) for _ in range(h // 128)]
                        for _ in range(bs)]) for _ in range(R)]
    out = oracle.quant_all_reduce(xs, ss, x_kind="int8", scale_kind="fp32", out_dtype=out_dtype)
    want = torch.tensor([[sum(xs[r][t, j].item() * ss[r][t, j // 128].item() for r in range(R))
                          for j in range(h)] for t in range(bs)], dtype=torch.float64)
    assert torch.equal(out.double(), want)          # |sum| <= 4*6*2 < 2^8: exact in every output type


def test_single_rank_is_plain_dequant():
    s = mc2_inputs.QARShape(world_size=1, bs=8, h=1024)
    inp = mc2_inputs.qar_inputs(s, seed=4)
    out = oracle.quant_all_reduce(inp["x_chunks"], inp["scale_chunks"], x_kind="int8", scale_kind="fp32",
                                  out_dtype=torch.float32)
    x = inp["x_chunks"][0].view(torch.int8).double()
    sc = inp["scale_chunks"][0].double().repeat_interleave(128, dim=1)
    assert torch.equal(out, (x * sc).float())
