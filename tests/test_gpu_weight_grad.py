"""GPU parity of mc2_matmul_weight_grad (C ABI) against the CPU oracle.

"hyper_parallel .../mc2.py" (AllGatherMatmulFunction.backward): grad_w =
grad_out.t().matmul(gathered) and grad_bias = grad_out.sum(dim=0).  dY^T is
read M-major straight from dY.  Cases span several tiles with ragged tails in
all three dimensions (a contraction tail inside a 64-row k-tile), both dtypes,
one-CTA and CTA-pair tiles, integer-exact data, and the full-size workload on
sampled rows.
"""
import pytest
import torch

import mc2_inputs
import oracle
import quantized_gemm_rank_gb300 as mc2
from parity import assert_bits_equal, assert_close_16, rows_per_block

pytestmark = pytest.mark.gpu

S = mc2_inputs.WGradShape


def run_gpu(inp, with_bias=True):
    dev = torch.device("cuda")
    dw, db = mc2.mc2_matmul_weight_grad(inp["dy"].to(dev), inp["x"].to(dev), with_bias=with_bias)
    torch.cuda.synchronize()
    assert mc2.mc2_device_status() == mc2.MC2_OK
    return dw.cpu(), (None if db is None else db.cpu())


CASES = {
    "bf16-ragged-pair": S(m=300, n=328, k=520),
    "fp16-ragged-pair": S(m=1100, n=264, k=264, dtype=torch.float16),
    "bf16-one-cta-tile": S(m=2100, n=96, k=776),
    "bf16-2kblocks": S(m=2048, n=512, k=512),
    "fp16-short-contraction": S(m=40, n=136, k=256, dtype=torch.float16),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_weight_grad_parity(name):
    inp = mc2_inputs.wgrad_inputs(CASES[name], seed=5)
    dw, db = run_gpu(inp)
    ref_w, ref_b = oracle.matmul_weight_grad(inp["dy"], inp["x"])
    assert_close_16(dw, ref_w, f"{name}: dw")
    assert_close_16(db, ref_b, f"{name}: db")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_integer_valued_inputs_bit_exact(dtype):
    """Small integers: every sum is an exact fp32 integer, so dW and dB must
    equal the oracle bit for bit (a transposed or shifted operand shows up)."""
    s = S(m=1090, n=272, k=328, dtype=dtype)
    g = torch.Generator().manual_seed(6)
    inp = {"dy": torch.randint(-3, 4, (s.m, s.n), generator=g).to(dtype),
           "x": torch.randint(-3, 4, (s.m, s.k), generator=g).to(dtype)}
    dw, db = run_gpu(inp)
    ref_w, ref_b = oracle.matmul_weight_grad(inp["dy"], inp["x"])
    assert_bits_equal(dw, ref_w, "integer dw")
    assert_bits_equal(db, ref_b, "integer db")


def test_without_bias_gradient():
    inp = mc2_inputs.wgrad_inputs(CASES["bf16-ragged-pair"], seed=7)
    a, _ = run_gpu(inp, with_bias=True)
    b, nb = run_gpu(inp, with_bias=False)
    assert nb is None
    assert_bits_equal(a, b, "dw with/without db")


def test_all_gather_layer_backward_end_to_end():
    """The all-gather layer's dW from the gathered output of the forward call
    equals the oracle on the chunks' concatenation."""
    dev = torch.device("cuda")
    shape = mc2_inputs.AGShape(world_size=4, m_local=256, k=512, n=384, x2_is_nk=True)
    inp = mc2_inputs.ag_inputs(shape, seed=9)
    _, gathered = mc2.mc2_all_gather_mm([c.to(dev) for c in inp["chunks"]], inp["x2"].to(dev), x2_is_nk=True)
    g = torch.Generator().manual_seed(10)
    dy = (torch.randn(shape.m, shape.n, generator=g) * shape.m ** -0.5).to(torch.bfloat16)
    dw, db = mc2.mc2_matmul_weight_grad(dy.to(dev), gathered)
    torch.cuda.synchronize()
    ref_w, ref_b = oracle.matmul_weight_grad(dy, oracle.gather(inp["chunks"]))
    assert_close_16(dw.cpu(), ref_w, "AG backward dw")
    assert_close_16(db.cpu(), ref_b, "AG backward db")


def test_full_size_row_of_every_warp_block():
    """wgrad-ag-4x4096 at full size (dW is 7168 x 8192: 28 x 32 tiles): one
    seeded row of dW from every 32-row block plus the first and last, every
    element of dB, and all outputs finite."""
    shape = mc2_inputs.WORKLOADS["wgrad-ag-4x4096"]
    inp = mc2_inputs.wgrad_inputs(shape, seed=0)
    dw, db = run_gpu(inp)
    rows = rows_per_block(shape.n, 32, seed=1, extra=(0, shape.n - 1))
    ref_w, ref_b = oracle.matmul_weight_grad(inp["dy"], inp["x"], rows=rows)
    assert_close_16(dw[rows], ref_w, "wgrad-ag-4x4096 rows")
    assert_close_16(db, ref_b, "wgrad-ag-4x4096 db")
    assert torch.isfinite(dw.float()).all()


def _sweep(count, seed):
    import random
    rng = random.Random(seed)
    return [S(m=rng.choice([1, 64, 100, 513, 1090, 2048]), n=rng.choice([8, 64, 128, 136, 272, 520, 1024]),
              k=rng.choice([8, 64, 264, 512, 1000]), dtype=rng.choice([torch.bfloat16, torch.float16]))
            for _ in range(count)]


@pytest.mark.parametrize("case,shape", list(enumerate(_sweep(16, 88))))
def test_seeded_shape_sweep(case, shape):
    """Seeded random shapes (one CTA and CTA pairs over dW's rows; contraction
    lengths from 1 to 2048 rows, ragged): dW and the bias gradient summed inside
    the GEMM, within the stated tolerance of the oracle."""
    inp = mc2_inputs.wgrad_inputs(shape, seed=500 + case)
    dw, db = run_gpu(inp)
    ref_w, ref_b = oracle.matmul_weight_grad(inp["dy"], inp["x"])
    assert_close_16(dw, ref_w, f"sweep {case}: dw")
    assert_close_16(db, ref_b, f"sweep {case}: db")
