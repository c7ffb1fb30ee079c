"""Pins for the weight/bias-gradient oracle ("hyper_parallel .../mc2.py":
module docstring dW = dY^T @ AllGather_m(X); AllGatherMatmulFunction.backward
grad_w = grad_out.t().matmul(gathered), grad_bias = grad_out.sum(dim=0)).

* small-integer inputs: the exact sums (Python loops) are representable, so the
  oracle must reproduce them bit for bit (a transposed operand, a wrong index or
  a dropped row fails)
* random inputs: within one rounding of the fp64 library matmul / sum
* the all-gather split: dW from the gathered X equals the sum over the ranks'
  chunks of dY_r^T @ X_r (the contraction split along m)
* a row subset of dW is bit-identical to the same rows of the full result
"""
import pytest
import torch

import oracle


def _ulp_bound(ref64, dtype):
    mant = 7 if dtype == torch.bfloat16 else 10
    return ref64.to(dtype).double().abs().clamp_min(1e-30) * 2.0 ** -mant


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_integer_inputs_exact(dtype):
    g = torch.Generator().manual_seed(8)
    m, n, k = 7, 5, 6
    dy = torch.randint(-4, 5, (m, n), generator=g).to(dtype)
    x = torch.randint(-4, 5, (m, k), generator=g).to(dtype)
    dw, db = oracle.matmul_weight_grad(dy, x)
    want_w = [[sum(dy[t, i].item() * x[t, j].item() for t in range(m)) for j in range(k)] for i in range(n)]
    want_b = [sum(dy[t, i].item() for t in range(m)) for i in range(n)]
    assert dw.shape == (n, k) and db.shape == (n,)
    assert torch.equal(dw.double(), torch.tensor(want_w, dtype=torch.float64))
    assert torch.equal(db.double(), torch.tensor(want_b, dtype=torch.float64))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_random_within_one_rounding(dtype):
    g = torch.Generator().manual_seed(9)
    m, n, k = 300, 40, 72
    dy = torch.randn(m, n, generator=g).to(dtype)
    x = torch.randn(m, k, generator=g).to(dtype)
    dw, db = oracle.matmul_weight_grad(dy, x)
    ref_w = dy.double().t() @ x.double()
    ref_b = dy.double().sum(0)
    assert torch.all((dw.double() - ref_w).abs() <= _ulp_bound(ref_w, dtype))
    assert torch.all((db.double() - ref_b).abs() <= _ulp_bound(ref_b, dtype))


def test_all_gather_split_of_the_contraction():
    g = torch.Generator().manual_seed(10)
    R, m_local, n, k = 4, 24, 16, 40
    xs = [torch.randn(m_local, k, generator=g).to(torch.bfloat16) for _ in range(R)]
    dy = torch.randn(R * m_local, n, generator=g).to(torch.bfloat16)
    dw, _ = oracle.matmul_weight_grad(dy, oracle.gather(xs), with_bias=False)
    parts = sum(dy[r * m_local:(r + 1) * m_local].double().t() @ xs[r].double() for r in range(R))
    assert torch.all((dw.double() - parts).abs() <= _ulp_bound(parts, torch.bfloat16))


def test_row_subset_matches_full():
    g = torch.Generator().manual_seed(11)
    dy = torch.randn(64, 30, generator=g).to(torch.bfloat16)
    x = torch.randn(64, 48, generator=g).to(torch.bfloat16)
    full, db = oracle.matmul_weight_grad(dy, x)
    rows = [29, 0, 13]
    sub, db2 = oracle.matmul_weight_grad(dy, x, rows=rows)
    assert torch.equal(sub.view(torch.int16), full[rows].view(torch.int16))
    assert torch.equal(db.view(torch.int16), db2.view(torch.int16))
