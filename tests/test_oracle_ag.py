"""Pins for the AllGatherMatmul oracle ("torch_npu.npu_all_gather_base_mm").

* gathered == concat_m(chunks) (输出说明: the second output is the allgather result)
* integer-valued inputs: the exact product (Python integer loops) is representable
  in the output type, so the oracle must reproduce it bit for bit -- this catches a
  dropped term, a wrong chunk or row index and a transposed operand
* world_size 1 is a plain matmul: compare with torch's fp64 matmul
* row-block independence (the dual identity in the mc2.py module docstring:
  row block r of AllGather_m(X) @ W^T is X_r @ W^T)
* x2 passed transposed (w (n,k), 约束说明) equals x2 = w^T contiguous
"""
import itertools

import pytest
import torch

import mc2_inputs
import oracle


def _int_tensor(g, shape, lo, hi, dtype):
    return torch.randint(lo, hi + 1, shape, generator=g).to(dtype)


def _brute(chunks, x2, x2_is_nk, bias):
    A = [row for c in chunks for row in c.tolist()]  # concat along m, by rows
    B = x2.tolist()
    k = len(A[0])
    n = len(B) if x2_is_nk else len(B[0])
    out = []
    for i in range(len(A)):
        row = []
        for j in range(n):
            s = 0
            for kk in range(k):
                b = B[j][kk] if x2_is_nk else B[kk][j]
                s += A[i][kk] * b
            if bias is not None:
                s += bias[j]
            row.append(s)
        out.append(row)
    return out


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("x2_is_nk,with_bias", [(False, False), (True, False), (False, True), (True, True)])
def test_integer_inputs_exact(dtype, x2_is_nk, with_bias):
    g = torch.Generator().manual_seed(11)
    R, ml, k, n = 3, 2, 7, 5
    chunks = [_int_tensor(g, (ml, k), -3, 3, dtype) for _ in range(R)]
    x2 = _int_tensor(g, (n, k) if x2_is_nk else (k, n), -3, 3, dtype)
    bias = (_int_tensor(g, (n,), -4, 4, dtype) * 0.5).to(dtype) if with_bias else None
    out, gathered = oracle.all_gather_mm(chunks, x2, x2_is_nk=x2_is_nk, bias=bias)
    bias_l = None if bias is None else bias.float().tolist()
    want = torch.tensor(_brute([c.float() for c in chunks], x2.float(), x2_is_nk, bias_l), dtype=torch.float64)
    assert torch.equal(out.double(), want)  # |sums| <= 7*9+2: exact in both types
    assert torch.equal(gathered, torch.cat(chunks, 0))


def test_gathered_is_concat_bitwise():
    s = mc2_inputs.scaled(mc2_inputs.WORKLOADS["ag-tiny"], world_size=4, m_local=8, k=64, n=16)
    inp = mc2_inputs.ag_inputs(s, seed=5)
    _, gathered = oracle.all_gather_mm(inp["chunks"], inp["x2"])
    assert torch.equal(gathered.view(torch.int16), torch.cat(inp["chunks"]).view(torch.int16))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_world_size_one_is_plain_matmul(dtype):
    g = torch.Generator().manual_seed(2)
    A = torch.randn(37, 300, generator=g).to(dtype)
    B = (torch.randn(300, 29, generator=g) * 0.05).to(dtype)
    out, _ = oracle.all_gather_mm([A], B)
    ref = A.double() @ B.double()
    # fp64 sums differ from torch's only in the last bits; one output ulp at most
    got = out.double()
    ulp = torch.abs(ref.to(dtype).double()).clamp_min(1e-30) * (2.0 ** (-7 if dtype == torch.bfloat16 else -10))
    assert torch.all(torch.abs(got - ref) <= ulp)
    assert (out.view(torch.int16) == ref.to(dtype).view(torch.int16)).float().mean() > 0.999


def test_row_blocks_are_independent_per_rank():
    s = mc2_inputs.scaled(mc2_inputs.WORKLOADS["ag-8x1024"], world_size=4, m_local=6, k=256, n=24)
    inp = mc2_inputs.ag_inputs(s, seed=9)
    full, _ = oracle.all_gather_mm(inp["chunks"], inp["x2"])
    for r, c in enumerate(inp["chunks"]):
        part, _ = oracle.all_gather_mm([c], inp["x2"])
        assert torch.equal(full[r * 6:(r + 1) * 6].view(torch.int16), part.view(torch.int16))


def test_transposed_weight_equals_row_major():
    s = mc2_inputs.scaled(mc2_inputs.WORKLOADS["ag-4x4096"], world_size=2, m_local=5, k=256, n=40)
    inp = mc2_inputs.ag_inputs(s, seed=4)
    w = inp["x2"]  # (n, k)
    a, _ = oracle.all_gather_mm(inp["chunks"], w, x2_is_nk=True, bias=inp["bias"])
    b, _ = oracle.all_gather_mm(inp["chunks"], w.t().contiguous(), x2_is_nk=False, bias=inp["bias"])
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_row_subset_matches_full():
    s = mc2_inputs.scaled(mc2_inputs.WORKLOADS["ag-8x1024"], world_size=2, m_local=16, k=256, n=32)
    inp = mc2_inputs.ag_inputs(s, seed=6)
    full, _ = oracle.all_gather_mm(inp["chunks"], inp["x2"])
    rows = [31, 0, 17, 16, 15]
    sub, _ = oracle.all_gather_mm(inp["chunks"], inp["x2"], rows=rows)
    assert torch.equal(sub.view(torch.int16), full[rows].view(torch.int16))


def test_example_shapes_against_fp64_matmul():
    """The page's call example: 8 ranks x (16, 512) fp16 times (512, 64)."""
    s = mc2_inputs.WORKLOADS["ag-tiny"]
    inp = mc2_inputs.ag_inputs(s, seed=0)
    out, gathered = oracle.all_gather_mm(inp["chunks"], inp["x2"])
    assert out.shape == (128, 64) and gathered.shape == (128, 512)
    ref = torch.cat(inp["chunks"]).double() @ inp["x2"].double()
    rel = (out.double() - ref).abs() / ref.abs().clamp_min(1e-3)
    assert rel.max() < 2.0 ** -10


def test_bias_is_added_before_one_rounding():
    # acc = 1 (exact), bias = 2**-8: 1 + 2**-8 ties to 1.0 in bf16 only if added
    # before a single rounding; two roundings (bias rounded after) give the same
    # here, so use a value that distinguishes: acc = 1 + 2**-8 - tiny is impossible
    # with bf16 inputs, so check the sum rounds like the exact value.
    A = torch.tensor([[1.0, 2.0 ** -8]], dtype=torch.bfloat16)
    B = torch.tensor([[1.0], [1.0]], dtype=torch.bfloat16)
    bias = torch.tensor([2.0 ** -8], dtype=torch.bfloat16)
    out, _ = oracle.all_gather_mm([A], B, bias=bias)
    # exact value 1 + 2**-7 is representable: a single rounding gives it; rounding
    # the matmul first (1 + 2**-8 -> 1.0) and then adding gives 1 + 2**-8 -> 1.0.
    assert out.item() == 1.0 + 2.0 ** -7
