"""Pins for the AlltoAllQuantMatmul oracle ("aclnnAlltoAllQuantMatmul", 计算公式).

* permute: brute-force index tracing of AlltoAll + permute(1,0,2) + view with torch
* commOut (alltoAllOut): the same tracing, element by element from each rank's x1
* quant: hand-derived rows (ties, smooth scale, zero row), and closed-form
  properties on random rows: max|q| = 127, |q*scale - y| <= scale/2
* int8 matmul: numpy's integer matmul, the all-127 accumulator bound, overflow
* dequant: scales 1 and bias 0 reduce to bf16(float(acc))
* the steps decided by fp32 rounding (the quant's division by the scale, the
  dequant's left-to-right products) against exact rational arithmetic with
  each IEEE rounding written out (fractions.Fraction), on inputs where the
  other plausible readings give another result
* the whole path on hand-derived tiny examples (tests/golden/a2a_tiny.json)
"""
import json
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import mc2_inputs
import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _simulate_alltoall_permute(x1_per_rank, j):
    """Rank j's permutedOut, traced with torch from the formula's own ops:
    commOut = AlltoAll(x1.view(R, BS/R, H)); permutedOut = commOut.permute(1,0,2).view(BS/R, R*H)."""
    R = len(x1_per_rank)
    BS, H = x1_per_rank[0].shape
    # AlltoAll: rank j receives block j of every rank r's view(R, BS/R, H)
    comm = torch.stack([x.view(R, BS // R, H)[j] for x in x1_per_rank], 0)  # (R, BS/R, H)
    return comm, comm.permute(1, 0, 2).reshape(BS // R, R * H)


@pytest.mark.parametrize("R", [2, 4, 8])
@pytest.mark.parametrize("elem", [torch.int16, torch.int8])
def test_permute_index_tracing(R, elem):
    BS, H = 4 * R, 3
    # entries encode (rank, row, col) uniquely
    if elem == torch.int16:
        x1 = [torch.tensor([[r * 1000 + i * 10 + h for h in range(H)] for i in range(BS)], dtype=torch.int16)
              for r in range(R)]
    else:
        x1 = [torch.tensor([[(r * 37 + i * 5 + h * 3) % 255 - 127 for h in range(H)] for i in range(BS)],
                           dtype=torch.int8) for r in range(R)]
    for j in range(R):
        comm, want = _simulate_alltoall_permute(x1, j)
        chunks = [comm[r].contiguous() for r in range(R)]
        if elem == torch.int16:
            got = oracle.permute([c.view(torch.bfloat16) for c in chunks]).view(torch.int16)
        else:
            got = oracle.permute(chunks)
        assert torch.equal(got, want)
        sub = oracle.permute(chunks if elem == torch.int8 else [c.view(torch.bfloat16) for c in chunks],
                             rows=[3, 0])
        assert torch.equal(sub.view(elem), want[[3, 0]])


@pytest.mark.parametrize("R", [2, 4, 8])
@pytest.mark.parametrize("elem", [torch.int16, torch.int8])
def test_comm_out_index_tracing(R, elem):
    """commOut on rank j, traced element by element with Python loops from
    every rank's x1 (BS, H): rank r sends rows [j*BS/R, (j+1)*BS/R) of its x1
    to rank j, which stores them as block r."""
    BS, H = 2 * R, 5
    x1 = [torch.tensor([[(r * 53 + i * 7 + h * 3) % 251 - 125 for h in range(H)] for i in range(BS)],
                       dtype=elem) for r in range(R)]
    for j in range(R):
        want = torch.empty((R, BS // R, H), dtype=elem)
        for r in range(R):
            for t in range(BS // R):
                for h in range(H):
                    want[r, t, h] = x1[r][j * (BS // R) + t, h]
        chunks = [x1[r][j * (BS // R):(j + 1) * (BS // R)].contiguous() for r in range(R)]
        if elem == torch.int16:
            got = oracle.comm_out([c.view(torch.bfloat16) for c in chunks]).view(torch.int16)
        else:
            got = oracle.comm_out(chunks)
        assert torch.equal(got, want)
        # and its permute(1, 0, 2).view is the permuted matrix
        P = oracle.permute(chunks if elem == torch.int8 else [c.view(torch.bfloat16) for c in chunks])
        assert torch.equal(got.permute(1, 0, 2).reshape(BS // R, R * H), P.view(elem))


def _round_binary(x: Fraction, p: int, emin: int = -126) -> Fraction:
    """x rounded to the nearest binary float with p significand bits (ties to
    even), exponent >= emin (subnormals below it): one IEEE rounding, done
    exactly.  p = 24 is fp32, p = 8 is bf16 (overflow is out of range here)."""
    if x == 0:
        return Fraction(0)
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()   # 2^e <= a < 2^(e+2)
    if Fraction(2) ** e > a:
        e -= 1
    if Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, emin) - p + 1)
    n = a / quantum
    r = n.numerator // n.denominator
    rest = n - r
    if rest > Fraction(1, 2) or (rest == Fraction(1, 2) and r % 2 == 1):
        r += 1
    return (r * quantum) if x > 0 else -(r * quantum)


def _rne_int(x: Fraction) -> int:
    """Nearest integer, ties to even."""
    r = x.numerator // x.denominator
    rest = x - r
    return r + 1 if rest > Fraction(1, 2) or (rest == Fraction(1, 2) and r % 2 == 1) else r


def _f32(bits: int) -> Fraction:
    return Fraction(struct.unpack("<f", struct.pack("<I", bits))[0])


@pytest.mark.parametrize("amax,y", [(Fraction(9, 8), Fraction(9, 16)), (Fraction(75, 64), Fraction(75, 128))])
def test_quant_divides_by_the_fp32_scale(amax, y):
    # A row [amax, y] with y = amax / 2: the real quotient y / (amax / 127) is the
    # tie 63.5, so the fp32 rounding of the scale decides q.  Exactly:
    # scale = fl32(amax / 127), q = rne(fl32(y / scale)).  Multiplying by
    # fl32(1 / scale) instead lands on the other side of the tie here.
    scale = _round_binary(amax / 127, 24)
    q_div = _rne_int(_round_binary(y / scale, 24))
    q_rcp = _rne_int(_round_binary(y * _round_binary(1 / scale, 24), 24))
    assert q_div != q_rcp, "the case no longer separates the two readings"
    x = torch.tensor([[float(amax), float(y)]], dtype=torch.bfloat16)
    assert x.double().tolist() == [[float(amax), float(y)]]
    q, sc = oracle.quant_pertoken_dynamic(x)
    assert Fraction(sc.item()) == scale
    assert q[0].tolist() == [127, q_div]


@pytest.mark.parametrize("acc,s1_bits,s2_bits", [(5951682, 0x3BF14CAA, 0x3B0336D7), (434371, 0x3C1A1E4B, 0x3B4F01C5)])
def test_dequant_products_left_to_right(acc, s1_bits, s2_bits):
    # out = bf16(((float(acc) * x1s) * x2s) + bias), each step one fp32 rounding,
    # in the order the formula prints.  On these inputs the fp32 result lands on
    # (or next to) a bf16 tie, and the product taken in the other order rounds
    # to another bf16 value.
    s1, s2 = _f32(s1_bits), _f32(s2_bits)
    a = _round_binary(Fraction(acc), 24)
    printed = _round_binary(_round_binary(_round_binary(a * s1, 24) * s2, 24), 8)
    swapped = _round_binary(_round_binary(_round_binary(a * s2, 24) * s1, 24), 8)
    assert printed != swapped, "the case no longer separates the two orders"
    out = oracle.dequant(torch.tensor([[acc]], dtype=torch.int32), torch.tensor([float(s1)]),
                         torch.tensor([float(s2)]), torch.zeros(1))
    assert Fraction(out.double().item()) == printed


def test_quant_golden_rows():
    cases = json.load(open(os.path.join(GOLD, "quant_rows.json")))["cases"]
    for c in cases:
        x = torch.tensor([c["x"]], dtype=torch.bfloat16)
        assert torch.equal(x.double(), torch.tensor([c["x"]], dtype=torch.float64)), "fixture not bf16-exact"
        s = None if c["smooth"] is None else torch.tensor(c["smooth"], dtype=torch.bfloat16)
        q, sc = oracle.quant_pertoken_dynamic(x, s)
        assert sc.tolist() == [c["scale"]], c["why"]
        assert q[0].tolist() == c["q"], c["why"]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_quant_properties_random(dtype):
    s = mc2_inputs.scaled(mc2_inputs.WORKLOADS["a2a-dyn"], bs_local=64, h=96, rank_size=4, x1_dtype=dtype)
    inp = mc2_inputs.a2a_inputs(s, seed=12)
    P = oracle.permute(inp["chunks"])
    P[5].zero_()  # a zero row
    q, sc = oracle.quant_pertoken_dynamic(P, inp["x1_scale"])
    # y computed independently: exact fp64 product of the two 16-bit values
    y = P.double() * inp["x1_scale"].double()[None, :]
    amax = y.abs().max(1).values
    nz = amax > 0
    assert torch.equal(q.abs().max(1).values[nz], torch.full((int(nz.sum()),), 127, dtype=torch.int8))
    assert torch.all(q[~nz] == 0) and torch.all(sc[~nz] == 0)
    # scale is the fp32 quotient amax/127 (within one fp32 rounding of the exact one)
    assert torch.allclose(sc[nz].double(), amax[nz] / 127.0, rtol=2 ** -23, atol=0)
    err = (q.double() * sc.double()[:, None] - y).abs()
    bound = sc.double()[:, None] * (0.5 + 1e-6)
    assert torch.all(err[nz] <= bound[nz])


def test_quant_smooth_uses_permuted_column():
    # distinct smooth per permuted column: applying it by chunk column would fail
    R, H = 4, 2
    chunks = [torch.full((1, H), 1.0, dtype=torch.bfloat16) for _ in range(R)]
    smooth = torch.tensor([1, 2, 4, 8, 16, 32, 64, 127], dtype=torch.bfloat16)
    q, sc = oracle.quant_pertoken_dynamic(oracle.permute(chunks), smooth)
    assert sc.item() == 1.0
    assert q[0].tolist() == [1, 2, 4, 8, 16, 32, 64, 127]


def test_int8_mm_matches_numpy_and_bounds():
    g = torch.Generator().manual_seed(1)
    a = torch.randint(-127, 128, (33, 700), generator=g, dtype=torch.int8)
    b = torch.randint(-127, 128, (700, 19), generator=g, dtype=torch.int8)
    got = oracle.int8_mm(a, b)
    ref = a.numpy().astype(np.int64) @ b.numpy().astype(np.int64)
    assert np.array_equal(got.numpy().astype(np.int64), ref)
    # all-127 K-block of 1024: 1024 * 127 * 127 = 16516096
    ones = torch.full((2, 1024), 127, dtype=torch.int8)
    acc = oracle.int8_mm(ones, torch.full((1024, 3), 127, dtype=torch.int8))
    assert torch.all(acc == 16516096)
    acc = oracle.int8_mm(-ones, torch.full((1024, 3), 127, dtype=torch.int8))
    assert torch.all(acc == -16516096)
    # a sum that leaves int32 is an error, not a silent wrap
    big = torch.full((1, 140000), 127, dtype=torch.int8)
    with pytest.raises(RuntimeError):
        oracle.int8_mm(big, torch.full((140000, 1), 127, dtype=torch.int8))


def test_dequant_unit_scales_is_rounding_of_acc():
    g = torch.Generator().manual_seed(8)
    acc = torch.randint(-2 ** 31, 2 ** 31 - 1, (16, 40), generator=g, dtype=torch.int64).to(torch.int32)
    out = oracle.dequant(acc, torch.ones(16), torch.ones(40), None)
    # torch: int32 -> fp32 (nearest) -> bf16 (nearest even), both single roundings
    assert torch.equal(out.view(torch.int16), acc.float().to(torch.bfloat16).view(torch.int16))
    out0 = oracle.dequant(acc, torch.ones(16), torch.ones(40), torch.zeros(40))
    assert torch.equal(out0.view(torch.int16), out.view(torch.int16))


def test_dequant_order_of_operations():
    # acc = 3, x1s = 1/3 (fp32), x2s = 3: (3 * fl(1/3)) * 3 rounds differently from 3 * (fl(1/3) * 3)?
    # Check only that the oracle equals the left-to-right fp32 evaluation done by numpy.
    g = torch.Generator().manual_seed(9)
    acc = torch.randint(-10 ** 6, 10 ** 6, (8, 12), generator=g, dtype=torch.int32)
    s1 = torch.rand(8, generator=g) * 1e-2
    s2 = torch.rand(12, generator=g) * 1e-2
    b = torch.randn(12, generator=g)
    got = oracle.dequant(acc, s1, s2, b)
    v = acc.numpy().astype(np.float32)
    v = (v * s1.numpy()[:, None]).astype(np.float32)
    v = (v * s2.numpy()[None, :]).astype(np.float32)
    v = (v + b.numpy()[None, :]).astype(np.float32)
    assert torch.equal(got.view(torch.int16), torch.from_numpy(v).to(torch.bfloat16).view(torch.int16))


def _golden_case(case):
    if case["quant_mode"] == 7:
        chunks = [torch.tensor(c, dtype=torch.bfloat16) for c in case["chunks"]]
        s = None if case["smooth"] is None else torch.tensor(case["smooth"], dtype=torch.bfloat16)
    else:
        chunks = [torch.tensor(c, dtype=torch.int8) for c in case["chunks"]]
        s = torch.tensor(case["x1_scale"], dtype=torch.float32)
    x2 = torch.tensor(case["x2"], dtype=torch.int8)
    res = oracle.alltoall_quant_mm(chunks, x2, torch.tensor(case["x2_scale"]), torch.tensor(case["bias"]),
                                   quant_mode=case["quant_mode"], x1_scale=s)
    return chunks, res


def test_whole_path_golden():
    gold = json.load(open(os.path.join(GOLD, "a2a_tiny.json")))
    for key in ("dynamic", "full"):
        case = gold[key]
        chunks, res = _golden_case(case)
        assert oracle.permute(chunks).double().tolist() == case["permuted"]
        assert res["acc"].tolist() == case["acc"]
        assert res["out"].double().tolist() == case["out"]
        if key == "dynamic":
            assert res["q"].tolist() == case["q"]
            assert res["x1_scale"].tolist() == case["x1_scale"]
        else:
            assert res["x1_scale"].tolist() == case["x1_scale"]


def test_whole_path_matches_steps_and_row_subsets():
    s = mc2_inputs.scaled(mc2_inputs.WORKLOADS["a2a-dyn"], bs_local=24, h=64, n=40)
    inp = mc2_inputs.a2a_inputs(s, seed=21)
    res = oracle.alltoall_quant_mm(inp["chunks"], inp["x2"], inp["x2_scale"], inp["bias"], quant_mode=7,
                                   x1_scale=inp["x1_scale"])
    P = oracle.permute(inp["chunks"])
    q, sc = oracle.quant_pertoken_dynamic(P, inp["x1_scale"])
    acc = oracle.int8_mm(q, inp["x2"])
    ref = acc.numpy().astype(np.int64)
    assert np.array_equal(ref, q.numpy().astype(np.int64) @ inp["x2"].numpy().astype(np.int64))
    assert torch.equal(res["q"], q) and torch.equal(res["x1_scale"], sc) and torch.equal(res["acc"], acc)
    rows = [23, 1, 7]
    sub = oracle.alltoall_quant_mm(inp["chunks"], inp["x2"], inp["x2_scale"], inp["bias"], quant_mode=7,
                                   x1_scale=inp["x1_scale"], rows=rows)
    for key in ("out", "q", "x1_scale", "acc"):
        a, b = sub[key], res[key][rows]
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b)


def test_full_quant_mode_uses_input_scale():
    s = mc2_inputs.scaled(mc2_inputs.WORKLOADS["a2a-full"], bs_local=16, h=32, n=24)
    inp = mc2_inputs.a2a_inputs(s, seed=2)
    res = oracle.alltoall_quant_mm(inp["chunks"], inp["x2"], inp["x2_scale"], inp["bias"], quant_mode=3,
                                   x1_scale=inp["x1_scale"])
    P = oracle.permute(inp["chunks"])
    assert torch.equal(res["q"], P)
    assert torch.equal(res["x1_scale"], inp["x1_scale"])
    ref = P.numpy().astype(np.int64) @ inp["x2"].numpy().astype(np.int64)
    assert np.array_equal(res["acc"].numpy().astype(np.int64), ref)
    # a row subset takes each token's own scale: the rows of the full result
    rows = [15, 0, 9, 4]
    sub = oracle.alltoall_quant_mm(inp["chunks"], inp["x2"], inp["x2_scale"], inp["bias"], quant_mode=3,
                                   x1_scale=inp["x1_scale"], rows=rows)
    assert torch.equal(sub["x1_scale"], inp["x1_scale"][rows])
    assert torch.equal(sub["out"].view(torch.int16), res["out"][rows].view(torch.int16))


def test_fp64_int8_mm_route_equals_integer_loop():
    g = torch.Generator().manual_seed(31)
    a = torch.randint(-127, 128, (20, 3000), generator=g, dtype=torch.int8)
    b = torch.randint(-127, 128, (3000, 70), generator=g, dtype=torch.int8)
    assert torch.equal(oracle.int8_mm_fp64(a, b, col_block=32), oracle.int8_mm(a, b))
    full = torch.full((3, 35000), 127, dtype=torch.int8)
    assert torch.all(oracle.int8_mm_fp64(full, torch.full((35000, 2), -127, dtype=torch.int8)) == -35000 * 16129)


def test_large_composite_uses_same_steps():
    # big enough to take the fp64 route; compare with the step-by-step C path
    s = mc2_inputs.scaled(mc2_inputs.WORKLOADS["a2a-full"], bs_local=40, h=2048, n=4096)
    inp = mc2_inputs.a2a_inputs(s, seed=3)
    assert 40 * 8 * 2048 * 4096 > (1 << 31)
    big = oracle.alltoall_quant_mm(inp["chunks"], inp["x2"], inp["x2_scale"], inp["bias"], quant_mode=3,
                                   x1_scale=inp["x1_scale"])
    P = oracle.permute(inp["chunks"])
    acc = oracle.int8_mm(P, inp["x2"])
    assert torch.equal(big["acc"], acc)
    assert torch.equal(big["out"].view(torch.int16),
                       oracle.dequant(acc, inp["x1_scale"], inp["x2_scale"], inp["bias"]).view(torch.int16))
    # the same route for a row subset (all 40 rows in reverse order: still large):
    # each output row is the full result's row, with its own token's scale
    rows = list(range(39, -1, -1))
    sub = oracle.alltoall_quant_mm(inp["chunks"], inp["x2"], inp["x2_scale"], inp["bias"], quant_mode=3,
                                   x1_scale=inp["x1_scale"], rows=rows)
    assert torch.equal(sub["x1_scale"], inp["x1_scale"][rows])
    assert torch.equal(sub["out"].view(torch.int16), big["out"][rows].view(torch.int16))
