"""Pins for the MatmulReduceScatter oracle ("hyper_parallel .../mc2.py" module
docstring: matmul_reduce_scatter forward Y = ReduceScatter_m(X @ W^T)).

* small-integer inputs: the exact sum over ranks (Python loops) is representable,
  so the oracle must reproduce it bit for bit (wrong rank, index or transpose fails)
* world_size 1 is a plain matmul (torch fp64)
* the reduction is over ranks: zeroing one rank's X removes exactly its term, and
  the result equals the single matmul of the k-concatenated shards (torch fp64)
* the scatter: rank j's block is rows [j*m/R, (j+1)*m/R) of the sum
* w (n, k) and x2 = w^T layouts agree
"""
import pytest
import torch

import oracle


def _ints(g, shape, dtype, lo=-3, hi=3):
    return torch.randint(lo, hi + 1, shape, generator=g).to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("w_is_nk", [True, False])
def test_integer_inputs_exact(dtype, w_is_nk):
    g = torch.Generator().manual_seed(4)
    R, m, kl, n = 3, 6, 5, 4
    xs = [_ints(g, (m, kl), dtype) for _ in range(R)]
    ws = [_ints(g, (n, kl) if w_is_nk else (kl, n), dtype) for _ in range(R)]
    bias = (_ints(g, (n,), dtype, -4, 4) * 0.5).to(dtype)
    got = oracle.matmul_reduce_scatter(xs, ws, w_is_nk=w_is_nk, bias=bias)
    want = [[sum(xs[r][i, kk].item() * (ws[r][j, kk].item() if w_is_nk else ws[r][kk, j].item())
                 for r in range(R) for kk in range(kl)) + bias[j].item() for j in range(n)] for i in range(m)]
    assert torch.equal(got.double(), torch.tensor(want, dtype=torch.float64))


def test_world_size_one_is_plain_matmul():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(21, 300, generator=g).to(torch.bfloat16)
    w = (torch.randn(17, 300, generator=g) * 0.05).to(torch.bfloat16)
    got = oracle.matmul_reduce_scatter([x], [w])
    ref = x.double() @ w.double().t()
    ulp = ref.to(torch.bfloat16).double().abs().clamp_min(1e-30) * 2.0 ** -7
    assert torch.all((got.double() - ref).abs() <= ulp)


def test_reduction_over_ranks_and_scatter_blocks():
    g = torch.Generator().manual_seed(6)
    R, m, kl, n = 4, 16, 64, 24
    xs = [torch.randn(m, kl, generator=g).to(torch.bfloat16) for _ in range(R)]
    ws = [(torch.randn(n, kl, generator=g) * 0.1).to(torch.bfloat16) for _ in range(R)]
    full = oracle.matmul_reduce_scatter(xs, ws)
    # one matmul of the k-concatenated shards, exact in fp64, rounded by torch
    cat = torch.cat(xs, 1).double() @ torch.cat(ws, 1).double().t()
    ulp = cat.to(torch.bfloat16).double().abs().clamp_min(1e-30) * 2.0 ** -7
    assert torch.all((full.double() - cat).abs() <= ulp)
    # zeroing rank 2's activations removes exactly its partial product
    xs0 = [x.clone() for x in xs]
    xs0[2].zero_()
    part = oracle.matmul_reduce_scatter(xs0, ws)
    cat0 = sum(xs0[r].double() @ ws[r].double().t() for r in range(R))
    assert torch.all((part.double() - cat0).abs() <= cat0.to(torch.bfloat16).double().abs().clamp_min(1e-30) * 2 ** -7)
    # rank j's output = rows [j*m/R, (j+1)*m/R) of the sum (the scatter)
    for j in range(R):
        rows = list(range(j * m // R, (j + 1) * m // R))
        blk = oracle.matmul_reduce_scatter(xs, ws, rows=rows)
        assert torch.equal(blk.view(torch.int16), full[rows].view(torch.int16))


def test_layouts_agree():
    g = torch.Generator().manual_seed(7)
    xs = [torch.randn(8, 256, generator=g).to(torch.bfloat16) for _ in range(2)]
    ws = [torch.randn(40, 256, generator=g).to(torch.bfloat16) for _ in range(2)]
    a = oracle.matmul_reduce_scatter(xs, ws, w_is_nk=True)
    b = oracle.matmul_reduce_scatter(xs, [w.t().contiguous() for w in ws], w_is_nk=False)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
