"""Pins for the oracle's own 16-bit decode / round-to-nearest-even encode.

Checked against (a) hand-derived IEEE encodings (tests/golden/fp16_rounding.json)
and (b) torch's independent conversions on every 16-bit pattern and on values
that are exactly fp32 (so torch's single rounding is the reference).
"""
import json
import os

import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp16_rounding.json")


def test_decode_every_pattern_matches_torch():
    bits = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    for is_bf16, dt in ((True, torch.bfloat16), (False, torch.float16)):
        ours = oracle.decode16(bits, is_bf16)
        ref = bits.view(dt).to(torch.float64)
        nan = torch.isnan(ref)
        assert torch.equal(torch.isnan(ours), nan)
        assert torch.equal(ours[~nan], ref[~nan])


@pytest.mark.parametrize("is_bf16", [True, False])
def test_encode_golden(is_bf16):
    cases = json.load(open(GOLDEN))["bf16" if is_bf16 else "f16"]
    vals = torch.tensor([float(eval(c["value"])) for c in cases], dtype=torch.float64)
    got = oracle.encode16(vals, is_bf16).view(torch.int16).to(torch.int32) & 0xFFFF
    want = torch.tensor([int(c["bits"], 16) for c in cases], dtype=torch.int32)
    assert torch.equal(got, want), [(c["value"], hex(g)) for c, g in zip(cases, got.tolist())]


@pytest.mark.parametrize("is_bf16", [True, False])
def test_encode_matches_torch_on_fp32_values(is_bf16):
    g = torch.Generator().manual_seed(3)
    dt = torch.bfloat16 if is_bf16 else torch.float16
    parts = [
        torch.randn(20000, generator=g),
        torch.randn(20000, generator=g) * 1e4,
        torch.randn(20000, generator=g) * 1e-6,       # fp16 subnormals
        torch.randn(20000, generator=g) * 1e-39,      # bf16 subnormals
        torch.randn(2000, generator=g) * 3e38,        # bf16 overflow
        torch.randn(2000, generator=g) * 7e4,         # fp16 overflow
    ]
    x = torch.cat(parts)  # fp32 values: torch rounds them once
    ours = oracle.encode16(x.double(), is_bf16).view(torch.int16)
    ref = x.to(dt).view(torch.int16)
    assert torch.equal(ours, ref)


def test_roundtrip_is_identity():
    bits = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    for is_bf16, dt in ((True, torch.bfloat16), (False, torch.float16)):
        v = oracle.decode16(bits, is_bf16)
        keep = ~torch.isnan(v)
        back = oracle.encode16(v[keep], is_bf16).view(torch.int16)
        assert torch.equal(back, bits[keep])


@pytest.mark.parametrize("is_bf16", [True, False])
def test_encode_special_values(is_bf16):
    # NaN stays NaN, infinities keep their sign, every value past the largest
    # finite one (after rounding) is infinity: the IEEE layouts' special codes,
    # decoded back by torch's own conversion
    dt = torch.bfloat16 if is_bf16 else torch.float16
    big = 3.5e38 if is_bf16 else 7.0e4
    vals = torch.tensor([float("nan"), -float("nan"), float("inf"), -float("inf"), big, -big],
                        dtype=torch.float64)
    got = oracle.encode16(vals, is_bf16).to(torch.float64)
    assert torch.isnan(got[:2]).all()
    assert got[2:].tolist() == [float("inf"), -float("inf"), float("inf"), -float("inf")]
    assert oracle.encode16(vals[2:], is_bf16).dtype == dt
