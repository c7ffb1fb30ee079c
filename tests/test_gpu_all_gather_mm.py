"""GPU parity of mc2_all_gather_mm (C ABI) against the CPU oracle.

"torch_npu.npu_all_gather_base_mm": out = AllGather_m(input) @ x2 and the
gathered input as the second output.  Cases span several 128 x 256 x 64 tiles
with ragged m / n / k tails, chunk boundaries inside an m-tile, both x2 layouts,
bias, both dtypes, ag-8x1024 at full size on every row, and ag-4x4096 at
full size on one row of every 32-row block.
"""
import pytest
import torch

import mc2_inputs
import oracle
import quantized_gemm_rank_gb300 as mc2
from parity import assert_bits_equal, assert_close_16, rows_per_block

pytestmark = pytest.mark.gpu


def run_gpu(inp, shape):
    dev = torch.device("cuda")
    chunks = [c.to(dev) for c in inp["chunks"]]
    x2 = inp["x2"].to(dev)
    bias = None if inp["bias"] is None else inp["bias"].to(dev)
    out, gathered = mc2.mc2_all_gather_mm(chunks, x2, x2_is_nk=shape.x2_is_nk, bias=bias,
                                          gather_output=shape.gather_output)
    torch.cuda.synchronize()
    assert mc2.mc2_device_status() == mc2.MC2_OK
    return out.cpu(), (None if gathered is None else gathered.cpu())


CASES = {
    # name: (AGShape, note)
    "ragged-bf16-kn": mc2_inputs.AGShape(world_size=4, m_local=72, k=328, n=520),
    "ragged-fp16-nk-bias": mc2_inputs.AGShape(world_size=2, m_local=136, k=392, n=264, dtype=torch.float16,
                                              x2_is_nk=True, bias=True),
    "bf16-nk-bias-8ranks": mc2_inputs.AGShape(world_size=8, m_local=40, k=512, n=776, x2_is_nk=True, bias=True),
    "fp16-kn-nogather": mc2_inputs.AGShape(world_size=2, m_local=256, k=256, n=512, dtype=torch.float16,
                                           gather_output=False),
    "bf16-kn-bias-tile-aligned": mc2_inputs.AGShape(world_size=2, m_local=256, k=1024, n=512, bias=True),
    "ag-tiny": mc2_inputs.WORKLOADS["ag-tiny"],
    # one CTA with an output at most 64 wide: the N = 64 tile, its B as one 3-D box
    # (n = 64), as a 2-D box with the columns past n zero-filled (n = 40), or K-major
    # (x2 = w^T); ragged rows; K spanning several 1024-deep blocks
    "narrow-bf16-kn-n40-ragged": mc2_inputs.AGShape(world_size=2, m_local=56, k=600, n=40),
    "narrow-fp16-nk-bias-n8": mc2_inputs.AGShape(world_size=8, m_local=8, k=2056, n=8, dtype=torch.float16,
                                                 x2_is_nk=True, bias=True),
    "narrow-bf16-kn-n64-k3000": mc2_inputs.AGShape(world_size=4, m_local=32, k=3000, n=64, bias=True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_all_gather_mm_parity(name):
    shape = CASES[name]
    inp = mc2_inputs.ag_inputs(shape, seed=7)
    out, gathered = run_gpu(inp, shape)
    ref, ref_g = oracle.all_gather_mm(inp["chunks"], inp["x2"], x2_is_nk=shape.x2_is_nk, bias=inp["bias"],
                                      gather_output=shape.gather_output)
    assert_close_16(out, ref, f"{name}: out")
    if shape.gather_output:
        assert_bits_equal(gathered, ref_g, f"{name}: gathered")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("x2_is_nk", [False, True])
def test_integer_valued_inputs_bit_exact(dtype, x2_is_nk):
    """Small-integer operands: fp32 accumulation is exact, so the GPU must equal
    the oracle bit for bit (any layout or indexing slip shows up here)."""
    g = torch.Generator().manual_seed(5)
    R, ml, k, n = 4, 40, 520, 264
    chunks = [torch.randint(-4, 5, (ml, k), generator=g).to(dtype) for _ in range(R)]
    x2 = torch.randint(-4, 5, (n, k) if x2_is_nk else (k, n), generator=g).to(dtype)
    bias = torch.randint(-8, 9, (n,), generator=g).to(dtype)
    dev = torch.device("cuda")
    out, gathered = mc2.mc2_all_gather_mm([c.to(dev) for c in chunks], x2.to(dev), x2_is_nk=x2_is_nk,
                                          bias=bias.to(dev))
    ref, ref_g = oracle.all_gather_mm(chunks, x2, x2_is_nk=x2_is_nk, bias=bias)
    assert_bits_equal(out, ref, "out")
    assert_bits_equal(gathered, ref_g, "gathered")


def test_full_size_every_row_ag_8x1024():
    """ag-8x1024 at full size, in the launch configuration the benchmark times
    (32 x 16 tiles over the co-resident CTA pairs: several persistent waves and
    raster groups): every output row against the oracle
    ("torch_npu.npu_all_gather_base_mm", 输出说明)."""
    shape = mc2_inputs.WORKLOADS["ag-8x1024"]
    inp = mc2_inputs.ag_inputs(shape, seed=0)
    out, gathered = run_gpu(inp, shape)
    ref, _ = oracle.all_gather_mm(inp["chunks"], inp["x2"], x2_is_nk=shape.x2_is_nk, bias=inp["bias"],
                                  gather_output=False)
    assert_close_16(out, ref, "ag-8x1024: every row")
    assert_bits_equal(gathered, torch.cat(inp["chunks"], 0), "ag-8x1024: gathered")


def test_full_size_row_of_every_warp_block_ag_4x4096():
    """ag-4x4096 (64 x 28 tiles, 24 persistent waves) at full size: one seeded
    row from every 32-row block (each epilogue warp's rows in every CTA of
    every tile row), the first and last row of each rank's chunk, and all
    outputs finite."""
    shape = mc2_inputs.WORKLOADS["ag-4x4096"]
    inp = mc2_inputs.ag_inputs(shape, seed=0)
    out, gathered = run_gpu(inp, shape)
    edges = [e for r in range(shape.world_size) for e in (r * shape.m_local, (r + 1) * shape.m_local - 1)]
    rows = rows_per_block(shape.m, 32, seed=1, extra=edges)
    assert rows.numel() >= shape.m // 32
    ref, _ = oracle.all_gather_mm(inp["chunks"], inp["x2"], x2_is_nk=shape.x2_is_nk, bias=inp["bias"],
                                  rows=rows, gather_output=False)
    assert_close_16(out[rows], ref, "ag-4x4096: rows")
    assert torch.isfinite(out.float()).all()
    assert_bits_equal(gathered, torch.cat(inp["chunks"], 0), "ag-4x4096: gathered")


def test_repeat_calls_are_deterministic():
    shape = CASES["ragged-bf16-kn"]
    inp = mc2_inputs.ag_inputs(shape, seed=3)
    a, _ = run_gpu(inp, shape)
    b, _ = run_gpu(inp, shape)
    assert_bits_equal(a, b, "repeat")


# The largest contraction the page allows (k < 65535, here 65528 = 1024 K blocks
# of 64), on one-CTA tiles (m = 16) and on CTA-pair tiles (m = 272), with the
# x2 (k, n) layout read as one 3-D box per stage (n % 64 == 0) and as 64-column
# boxes (n % 64 != 0).
MAX_K_CASES = {
    "maxk-one-cta-3d": mc2_inputs.AGShape(world_size=2, m_local=8, k=65528, n=64),
    "maxk-pair-2d-bias": mc2_inputs.AGShape(world_size=2, m_local=136, k=65528, n=72, bias=True),
    "maxk-pair-nk": mc2_inputs.AGShape(world_size=2, m_local=136, k=65528, n=128, x2_is_nk=True),
}


@pytest.mark.parametrize("name", sorted(MAX_K_CASES))
def test_largest_k(name):
    shape = MAX_K_CASES[name]
    inp = mc2_inputs.ag_inputs(shape, seed=9)
    out, gathered = run_gpu(inp, shape)
    ref, ref_g = oracle.all_gather_mm(inp["chunks"], inp["x2"], x2_is_nk=shape.x2_is_nk, bias=inp["bias"])
    assert_close_16(out, ref, f"{name}: out")
    assert_bits_equal(gathered, ref_g, f"{name}: gathered")


# Several K blocks of 1024 per tile (the fp32 block sums added in order),
# fewer pair tiles than co-resident CTA pairs, a ragged last K block and
# n-tile: every output row against the oracle.
KBLOCK_CASES = {
    "kblocks-bf16-kn-bias": mc2_inputs.AGShape(world_size=2, m_local=1280, k=3072, n=1024, bias=True),
    "kblocks-fp16-nk-ragged": mc2_inputs.AGShape(world_size=4, m_local=520, k=2112, n=1000, dtype=torch.float16,
                                                 x2_is_nk=True),
}


@pytest.mark.parametrize("name", sorted(KBLOCK_CASES))
def test_several_k_blocks_every_row(name):
    shape = KBLOCK_CASES[name]
    inp = mc2_inputs.ag_inputs(shape, seed=21)
    out, gathered = run_gpu(inp, shape)
    ref, ref_g = oracle.all_gather_mm(inp["chunks"], inp["x2"], x2_is_nk=shape.x2_is_nk, bias=inp["bias"])
    assert_close_16(out, ref, f"{name}: out")
    assert_bits_equal(gathered, ref_g, f"{name}: gathered")


@pytest.mark.parametrize("x2_is_nk", [False, True])
def test_several_k_blocks_integer_valued_bit_exact(x2_is_nk):
    """Small-integer operands over four K blocks (the last one ragged): every
    block sum is exact, so a block added twice or missed changes the bits."""
    g = torch.Generator().manual_seed(9)
    R, ml, k, n = 2, 1280, 3136, 776
    chunks = [torch.randint(-3, 4, (ml, k), generator=g).to(torch.bfloat16) for _ in range(R)]
    x2 = torch.randint(-3, 4, (n, k) if x2_is_nk else (k, n), generator=g).to(torch.bfloat16)
    dev = torch.device("cuda")
    out, gathered = mc2.mc2_all_gather_mm([c.to(dev) for c in chunks], x2.to(dev), x2_is_nk=x2_is_nk)
    ref, ref_g = oracle.all_gather_mm(chunks, x2, x2_is_nk=x2_is_nk)
    assert_bits_equal(out, ref, "out")
    assert_bits_equal(gathered, ref_g, "gathered")


def test_binding_refuses_a_host_tensor_among_device_ones():
    """The library launches on the current device; the binding refuses any
    operand that lives elsewhere (here x2 on the host) before calling it."""
    dev = torch.device("cuda")
    x = [torch.zeros(16, 256, dtype=torch.bfloat16, device=dev)] * 2
    with pytest.raises(ValueError, match="x2 must be a CUDA tensor on the current device"):
        mc2.mc2_all_gather_mm(x, torch.zeros(256, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="out must be a CUDA tensor"):
        mc2.mc2_all_gather_mm(x, torch.zeros(256, 64, dtype=torch.bfloat16, device=dev),
                              out=torch.zeros(32, 64, dtype=torch.bfloat16))


@pytest.mark.parametrize("name", ["ag-tiny", "ragged-bf16-kn", "narrow-fp16-nk-bias-n8", "bf16-kn-bias-tile-aligned"])
def test_chunks_of_one_buffer_match_separate_chunks(name):
    """Chunks that lie back to back (the slices of one receive buffer) are read
    through one map of the whole A when a chunk is shorter than a tile; chunks
    in separate allocations box by box.  Both layouts give the same bits, and
    the oracle's result."""
    shape = CASES[name]
    inp = mc2_inputs.ag_inputs(shape, seed=11)
    dev = torch.device("cuda")
    x2 = inp["x2"].to(dev)
    bias = None if inp["bias"] is None else inp["bias"].to(dev)
    whole = torch.cat(inp["chunks"]).to(dev)
    sliced = list(whole.split(shape.m_local))
    separate, gaps = [], []
    for c in inp["chunks"]:
        separate.append(c.to(dev))
        gaps.append(torch.empty(1 << 16, dtype=torch.uint8, device=dev))   # keep them apart
    outs = []
    for chunks in (sliced, separate):
        out, g = mc2.mc2_all_gather_mm(chunks, x2, x2_is_nk=shape.x2_is_nk, bias=bias,
                                       gather_output=shape.gather_output)
        torch.cuda.synchronize()
        assert mc2.mc2_device_status() == mc2.MC2_OK
        outs.append((out.cpu(), None if g is None else g.cpu()))
    assert_bits_equal(outs[0][0], outs[1][0], f"{name}: out, one buffer vs separate")
    ref, ref_g = oracle.all_gather_mm(inp["chunks"], inp["x2"], x2_is_nk=shape.x2_is_nk, bias=inp["bias"],
                                      gather_output=shape.gather_output)
    assert_close_16(outs[0][0], ref, f"{name}: out")
    if shape.gather_output:
        assert_bits_equal(outs[0][1], ref_g, f"{name}: gathered")



def test_run_time_tiles_on_a_large_grid():
    """8192 tiles of 256 x 256 (one CTA pair launched per tile; the running pairs
    take over the tiles of pairs not yet launched): one seeded row of every
    256-row tile block checked against the oracle, the gathered output bit for
    bit, and every output finite."""
    shape = mc2_inputs.AGShape(world_size=8, m_local=8192, k=256, n=8192, bias=True)
    inp = mc2_inputs.ag_inputs(shape, seed=21)
    dev = torch.device("cuda")
    out, gathered = mc2.mc2_all_gather_mm([c.to(dev) for c in inp["chunks"]], inp["x2"].to(dev),
                                          bias=inp["bias"].to(dev))
    torch.cuda.synchronize()
    assert mc2.mc2_device_status() == mc2.MC2_OK
    rows = rows_per_block(shape.m, 256, seed=22)
    ref, _ = oracle.all_gather_mm(inp["chunks"], inp["x2"], bias=inp["bias"], rows=rows, gather_output=False)
    o = out.cpu()
    assert_close_16(o[rows], ref, "8192 tiles: sampled rows")
    assert torch.isfinite(o).all()
    assert_bits_equal(gathered.cpu(), torch.cat(inp["chunks"]), "8192 tiles: gathered")


def _ag_sweep(count, seed):
    import random
    rng = random.Random(seed)
    shapes = []
    for _ in range(count):
        R = rng.choice([2, 4, 8])
        m_local = rng.choice([8, 16, 40, 64, 72, 128, 136, 256, 512, 1000])
        k = rng.choice([256, 264, 512, 1032, 2048])
        n = rng.choice([8, 64, 136, 256, 264, 520, 1000, 2048])
        shapes.append(mc2_inputs.AGShape(world_size=R, m_local=m_local, k=k, n=n,
                                         dtype=rng.choice([torch.bfloat16, torch.float16]),
                                         x2_is_nk=rng.choice([True, False]), bias=rng.choice([True, False]),
                                         gather_output=rng.choice([True, False])))
    return shapes


@pytest.mark.parametrize("case,shape", list(enumerate(_ag_sweep(24, 2026))))
def test_seeded_shape_sweep(case, shape):
    """Seeded random shapes over both tile forms (one CTA, narrow or wide; CTA
    pairs with run-time tiles), both x2 layouts, with and without bias and the
    gathered output: every output within the stated tolerance of the oracle,
    the gathered output bit for bit."""
    inp = mc2_inputs.ag_inputs(shape, seed=300 + case)
    out, gathered = run_gpu(inp, shape)
    ref, ref_g = oracle.all_gather_mm(inp["chunks"], inp["x2"], x2_is_nk=shape.x2_is_nk, bias=inp["bias"],
                                      gather_output=shape.gather_output)
    assert_close_16(out, ref, f"sweep {case}: out")
    if shape.gather_output:
        assert_bits_equal(gathered, ref_g, f"sweep {case}: gathered")
