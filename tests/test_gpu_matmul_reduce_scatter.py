"""GPU parity of mc2_matmul_reduce_scatter (C ABI) against the CPU oracle.

"hyper_parallel .../mc2.py" (module docstring, MatmulReduceScatterFunction):
every rank's partial product X_r @ W_r^T is summed over the ranks and the sum's
row blocks are scattered, rank j receiving rows [j*m/R, (j+1)*m/R).  Cases span
several tiles with ragged m / n tails, rank boundaries inside a 1024-long K
block, both weight layouts, bias, both dtypes, and the full-size workload on
sampled rows.
"""
import pytest
import torch

import mc2_inputs
import oracle
import quantized_gemm_rank_gb300 as mc2
from parity import assert_bits_equal, assert_close_16, rows_per_block

pytestmark = pytest.mark.gpu

S = mc2_inputs.MMRSShape


def run_gpu(inp, shape):
    dev = torch.device("cuda")
    xs = [x.to(dev) for x in inp["x_chunks"]]
    ws = [w.to(dev) for w in inp["w_chunks"]]
    bias = None if inp["bias"] is None else inp["bias"].to(dev)
    outs = mc2.mc2_matmul_reduce_scatter(xs, ws, w_is_nk=shape.w_is_nk, bias=bias)
    torch.cuda.synchronize()
    assert mc2.mc2_device_status() == mc2.MC2_OK
    assert len(outs) == shape.world_size
    for o in outs:
        assert o.shape == (shape.m // shape.world_size, shape.n)
    return torch.cat([o.cpu() for o in outs], 0)


def run_oracle(inp, shape, rows=None):
    return oracle.matmul_reduce_scatter(inp["x_chunks"], inp["w_chunks"], w_is_nk=shape.w_is_nk,
                                        bias=inp["bias"], rows=rows)


CASES = {
    "bf16-nk-ragged": S(world_size=4, m=200, k_local=320, n=520),
    "fp16-kn-bias": S(world_size=2, m=272, k_local=576, n=264, dtype=torch.float16, w_is_nk=False, bias=True),
    "bf16-nk-bias-8ranks": S(world_size=8, m=136, k_local=256, n=776, bias=True),
    "bf16-kn-one-tile-row": S(world_size=8, m=64, k_local=512, n=256, w_is_nk=False),
    "bf16-nk-2kblocks-pair": S(world_size=2, m=512, k_local=1536, n=512, bias=True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_matmul_reduce_scatter_parity(name):
    shape = CASES[name]
    inp = mc2_inputs.mmrs_inputs(shape, seed=11)
    assert_close_16(run_gpu(inp, shape), run_oracle(inp, shape), name)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("w_is_nk", [False, True])
def test_integer_valued_inputs_bit_exact(dtype, w_is_nk):
    """Small-integer operands: every partial sum is an exact fp32 integer, so the
    GPU must equal the oracle bit for bit (a wrong rank's weight, a transposed
    shard or a misplaced scatter block shows up here)."""
    shape = S(world_size=4, m=264, k_local=384, n=328, dtype=dtype, w_is_nk=w_is_nk, bias=True)
    g = torch.Generator().manual_seed(21)
    inp = mc2_inputs.mmrs_inputs(shape, seed=3)
    inp["x_chunks"] = [torch.randint(-3, 4, x.shape, generator=g).to(dtype) for x in inp["x_chunks"]]
    inp["w_chunks"] = [torch.randint(-3, 4, w.shape, generator=g).to(dtype) for w in inp["w_chunks"]]
    inp["bias"] = torch.randint(-8, 9, (shape.n,), generator=g).to(dtype)
    assert_bits_equal(run_gpu(inp, shape), run_oracle(inp, shape), "integer-valued")


def test_each_rank_contributes_its_own_term():
    """One rank's activations set to zero: the result must equal the oracle with
    that rank removed, bit for bit on integer data."""
    shape = S(world_size=4, m=256, k_local=256, n=256)
    g = torch.Generator().manual_seed(5)
    inp = mc2_inputs.mmrs_inputs(shape, seed=5)
    inp["x_chunks"] = [torch.randint(-2, 3, x.shape, generator=g).to(torch.bfloat16) for x in inp["x_chunks"]]
    inp["w_chunks"] = [torch.randint(-2, 3, w.shape, generator=g).to(torch.bfloat16) for w in inp["w_chunks"]]
    for dead in range(shape.world_size):
        cur = dict(inp)
        cur["x_chunks"] = [torch.zeros_like(x) if r == dead else x for r, x in enumerate(inp["x_chunks"])]
        assert_bits_equal(run_gpu(cur, shape), run_oracle(cur, shape), f"rank {dead} zeroed")


def test_full_size_row_of_every_warp_block():
    """mmrs-4x2048 at full size (64 x 32 tiles over the co-resident CTA pairs):
    one seeded row from every 32-row block, the first and last row of each
    rank's output, and all outputs finite."""
    shape = mc2_inputs.WORKLOADS["mmrs-4x2048"]
    inp = mc2_inputs.mmrs_inputs(shape, seed=0)
    got = run_gpu(inp, shape)
    per = shape.m // shape.world_size
    edges = [e for r in range(shape.world_size) for e in (r * per, (r + 1) * per - 1)]
    rows = rows_per_block(shape.m, 32, seed=1, extra=edges)
    assert_close_16(got[rows], run_oracle(inp, shape, rows=rows), "mmrs-4x2048 rows")
    assert torch.isfinite(got.float()).all()


def _sweep(count, seed):
    import random
    rng = random.Random(seed)
    shapes = []
    for _ in range(count):
        R = rng.choice([2, 4, 8])
        m = R * rng.choice([8, 17, 32, 64, 100, 128, 256])
        k_local = rng.choice([256, 320, 512, 1024])
        n = rng.choice([8, 64, 264, 520, 1024])
        shapes.append(S(world_size=R, m=m, k_local=k_local, n=n, dtype=rng.choice([torch.bfloat16, torch.float16]),
                        w_is_nk=rng.choice([True, False]), bias=rng.choice([True, False])))
    return shapes


@pytest.mark.parametrize("case,shape", list(enumerate(_sweep(16, 77))))
def test_seeded_shape_sweep(case, shape):
    """Seeded random shapes (one CTA and CTA pairs, ranks whose row blocks do and
    do not fill a warp's 32 rows, both weight layouts, with and without bias):
    every row of every rank's output within the stated tolerance of the oracle."""
    inp = mc2_inputs.mmrs_inputs(shape, seed=400 + case)
    assert_close_16(run_gpu(inp, shape), run_oracle(inp, shape), f"sweep {case}")
