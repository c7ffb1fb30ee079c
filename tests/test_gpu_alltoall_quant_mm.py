"""GPU parity of mc2_alltoall_quant_mm (C ABI) against the CPU oracle.

"aclnnAlltoAllQuantMatmul" (计算公式): permute the received chunks, quantise per
token (mode 7) or take the int8 chunks as they are (mode 3), int8 matmul with
exact int32 accumulation, dequant by x1 scale x x2 scale, add bias, bf16 out.
Every output is compared bit for bit: q, x1_scale, the int32 accumulators and
out (the same fp32 operations in the same order on both sides).
"""
import pytest
import torch

import mc2_inputs
import oracle
import quantized_gemm_rank_gb300 as mc2
from parity import assert_bits_equal

pytestmark = pytest.mark.gpu


def run_gpu(inp, shape, want_debug=True, bias_bf16=False):
    dev = torch.device("cuda")
    chunks = [c.to(dev) for c in inp["chunks"]]
    x1s = None if inp["x1_scale"] is None else inp["x1_scale"].to(dev)
    bias = inp["bias"].to(torch.bfloat16 if bias_bf16 else torch.float32).to(dev)
    K = shape.rank_size * shape.h
    q = torch.empty((shape.bs_local, K), dtype=torch.int8, device=dev) if want_debug else None
    s = torch.empty((shape.bs_local,), dtype=torch.float32, device=dev) if want_debug else None
    acc = torch.empty((shape.bs_local, shape.n), dtype=torch.int32, device=dev) if want_debug else None
    res = mc2.mc2_alltoall_quant_mm(chunks, inp["x2"].to(dev), inp["x2_scale"].to(dev), bias,
                                    x1_quant_mode=shape.quant_mode, x1_scale=x1s, q_out=q, x1_scale_out=s,
                                    acc_out=acc)
    torch.cuda.synchronize()
    assert mc2.mc2_device_status() == mc2.MC2_OK
    return {k: (None if v is None else v.cpu()) for k, v in res.items()}


def run_oracle(inp, shape, rows=None, bias_bf16=False):
    bias = inp["bias"]
    if bias_bf16:
        bias = bias.to(torch.bfloat16).float()
    return oracle.alltoall_quant_mm(inp["chunks"], inp["x2"], inp["x2_scale"], bias,
                                    quant_mode=shape.quant_mode, x1_scale=inp["x1_scale"], rows=rows)


def compare(got, ref, name, rows=None):
    sel = (lambda t: t) if rows is None else (lambda t: t[rows])
    assert_bits_equal(sel(got["acc"]), ref["acc"], f"{name}: acc")
    assert_bits_equal(sel(got["q"]), ref["q"], f"{name}: q")
    assert_bits_equal(sel(got["x1_scale"]), ref["x1_scale"], f"{name}: x1_scale")
    assert_bits_equal(sel(got["out"]), ref["out"], f"{name}: out")


A2A = mc2_inputs.A2AShape
CASES = {
    "dyn-bf16-ragged": A2A(rank_size=4, bs_local=200, h=96, n=272, quant_mode=7),
    "dyn-fp16-scalar-h": A2A(rank_size=8, bs_local=72, h=6, n=48, quant_mode=7, x1_dtype=torch.float16),
    "dyn-bf16-nosmooth": A2A(rank_size=2, bs_local=130, h=256, n=528, quant_mode=7, smooth=False),
    "dyn-bf16-2kblocks": A2A(rank_size=8, bs_local=136, h=320, n=256, quant_mode=7),
    "full-int8-ragged": A2A(rank_size=8, bs_local=136, h=48, n=320, quant_mode=3),
    "full-int8-scalar-h": A2A(rank_size=2, bs_local=40, h=24, n=32, quant_mode=3),
    "full-int8-3kblocks": A2A(rank_size=4, bs_local=256, h=640, n=512, quant_mode=3),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_alltoall_quant_mm_parity(name):
    shape = CASES[name]
    inp = mc2_inputs.a2a_inputs(shape, seed=13)
    got = run_gpu(inp, shape)
    ref = run_oracle(inp, shape)
    compare(got, ref, name)


def test_bias_bf16_accepted():
    shape = CASES["dyn-bf16-ragged"]
    inp = mc2_inputs.a2a_inputs(shape, seed=4)
    got = run_gpu(inp, shape, bias_bf16=True)
    ref = run_oracle(inp, shape, bias_bf16=True)
    compare(got, ref, "bias-bf16")


def test_zero_and_outlier_rows():
    shape = A2A(rank_size=4, bs_local=64, h=128, n=256, quant_mode=7)
    inp = mc2_inputs.a2a_inputs(shape, seed=8)
    for c in inp["chunks"]:
        c[3].zero_()            # zero row: scale 0, q 0, out = bias
        c[9, 5] = 3.0e4         # a single huge outlier in row 9 of every chunk
    got = run_gpu(inp, shape)
    ref = run_oracle(inp, shape)
    compare(got, ref, "zero/outlier rows")
    assert torch.all(got["q"][3] == 0) and got["x1_scale"][3].item() == 0.0


@pytest.mark.parametrize("sign", [1, -1])
def test_accumulator_bound_all_127(sign):
    """All-127 operands: every 1024-long block reaches 1024*127*127 = 16516096
    (just under 2^24) and the total 4096*16129 = 66064384 is far above it, so
    the int32 result is exact only if each block is flushed exactly."""
    shape = A2A(rank_size=8, bs_local=128, h=512, n=256, quant_mode=3)
    inp = mc2_inputs.a2a_inputs(shape, seed=1)
    inp["chunks"] = [torch.full_like(c, 127 * sign) for c in inp["chunks"]]
    inp["x2"] = torch.full_like(inp["x2"], 127)
    got = run_gpu(inp, shape)
    ref = run_oracle(inp, shape)
    assert torch.all(ref["acc"] == sign * 4096 * 16129)
    compare(got, ref, "all-127")


def test_full_size_dynamic_sampled_rows():
    shape = mc2_inputs.WORKLOADS["a2a-dyn"]
    inp = mc2_inputs.a2a_inputs(shape, seed=0)
    got = run_gpu(inp, shape)
    rows = mc2_inputs.sample_rows(shape.bs_local, 96, seed=1)
    ref = run_oracle(inp, shape, rows=rows)
    compare(got, ref, "a2a-dyn", rows=rows)
    # the quantised activations and scales of every row (cheap on the CPU)
    P = oracle.permute(inp["chunks"])
    q, s = oracle.quant_pertoken_dynamic(P, inp["x1_scale"])
    assert_bits_equal(got["q"], q, "a2a-dyn: all q")
    assert_bits_equal(got["x1_scale"], s, "a2a-dyn: all scales")


def test_literal_small_config_every_row():
    """The dynamic-quant config read literally (8 chunks of (512, 1024) -> a
    (512, 8192) permuted matrix), small enough for the oracle to check every
    output: one wave of tiles, each over all eight K blocks."""
    shape = mc2_inputs.WORKLOADS["a2a-dyn-small"]
    inp = mc2_inputs.a2a_inputs(shape, seed=0)
    got = run_gpu(inp, shape)
    ref = run_oracle(inp, shape)
    compare(got, ref, "a2a-dyn-small")


def test_full_size_full_quant_subset():
    """The full-quant workload; the oracle checks a seeded 1024-row subset."""
    shape = mc2_inputs.WORKLOADS["a2a-full"]
    inp = mc2_inputs.a2a_inputs(shape, seed=0)
    got = run_gpu(inp, shape)
    rows = mc2_inputs.sample_rows(shape.bs_local, 1024, seed=1)
    ref = run_oracle(inp, shape, rows=rows)
    compare(got, ref, "a2a-full", rows=rows)


def test_without_debug_outputs_matches():
    shape = CASES["dyn-bf16-2kblocks"]
    inp = mc2_inputs.a2a_inputs(shape, seed=2)
    a = run_gpu(inp, shape, want_debug=True)
    b = run_gpu(inp, shape, want_debug=False)
    assert_bits_equal(a["out"], b["out"], "out with/without debug outputs")


@pytest.mark.parametrize("name", ["dyn-bf16-ragged", "dyn-fp16-scalar-h", "full-int8-ragged", "full-int8-scalar-h",
                                  "full-int8-3kblocks"])
def test_alltoall_out_is_comm_out(name):
    """alltoAllOut (commOut): every received chunk as block r, bit for bit, and
    the main outputs unchanged by asking for it."""
    shape = CASES[name]
    inp = mc2_inputs.a2a_inputs(shape, seed=17)
    dev = torch.device("cuda")
    chunks = [c.to(dev) for c in inp["chunks"]]
    x1s = None if inp["x1_scale"] is None else inp["x1_scale"].to(dev)
    args = (chunks, inp["x2"].to(dev), inp["x2_scale"].to(dev), inp["bias"].to(dev))
    co = torch.full((shape.rank_size, shape.bs_local, shape.h), 7, dtype=chunks[0].dtype, device=dev)
    a = mc2.mc2_alltoall_quant_mm(*args, x1_quant_mode=shape.quant_mode, x1_scale=x1s, alltoall_out=co)
    b = mc2.mc2_alltoall_quant_mm(*args, x1_quant_mode=shape.quant_mode, x1_scale=x1s)
    torch.cuda.synchronize()
    assert mc2.mc2_device_status() == mc2.MC2_OK
    assert_bits_equal(co.cpu(), oracle.comm_out(inp["chunks"]), f"{name}: alltoall_out")
    assert_bits_equal(a["out"].cpu(), b["out"].cpu(), f"{name}: out with/without alltoall_out")
    ref = run_oracle(inp, shape)
    assert_bits_equal(a["out"].cpu(), ref["out"], f"{name}: out")


def test_alltoall_out_full_size_dynamic():
    shape = mc2_inputs.WORKLOADS["a2a-dyn"]
    inp = mc2_inputs.a2a_inputs(shape, seed=0)
    dev = torch.device("cuda")
    chunks = [c.to(dev) for c in inp["chunks"]]
    co = torch.empty((shape.rank_size, shape.bs_local, shape.h), dtype=chunks[0].dtype, device=dev)
    mc2.mc2_alltoall_quant_mm(chunks, inp["x2"].to(dev), inp["x2_scale"].to(dev), inp["bias"].to(dev),
                              x1_quant_mode=7, x1_scale=inp["x1_scale"].to(dev), alltoall_out=co)
    torch.cuda.synchronize()
    assert mc2.mc2_device_status() == mc2.MC2_OK
    assert_bits_equal(co.cpu(), oracle.comm_out(inp["chunks"]), "a2a-dyn: alltoall_out")


def test_quant_ties_and_near_ties_on_gpu():
    """Exact half-integer quotients (scale 1: every k + 0.5 for k in [-126, 125]),
    values a few bf16 ulps around them, and the hand-derived golden rows: the GPU
    must round each to the same integer as the oracle's IEEE division."""
    import json
    import os
    R, h = 2, 256
    K = R * h
    rows = []
    ties = [127.0] + [k + 0.5 for k in range(-126, 126)]
    rows.append(ties + [0.0] * (K - len(ties)))
    near = [127.0]
    for k in range(-120, 120, 3):
        for d in (-2 ** -6, 2 ** -6, -2 ** -5, 2 ** -5):
            near.append(k + 0.5 + d)
    rows.append(near[:K] + [0.0] * (K - len(near[:K])))
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "quant_rows.json")))["cases"]
    for c in gold:
        if c["smooth"] is None:
            rows.append(c["x"] + [0.0] * (K - len(c["x"])))
    P = torch.tensor(rows, dtype=torch.bfloat16)
    chunks = [P[:, r * h:(r + 1) * h].contiguous() for r in range(R)]
    shape = A2A(rank_size=R, bs_local=P.shape[0], h=h, n=64, quant_mode=7, smooth=False)
    g = torch.Generator().manual_seed(3)
    inp = {"chunks": chunks, "x1_scale": None,
           "x2": torch.randint(-127, 128, (K, 64), generator=g, dtype=torch.int8),
           "x2_scale": torch.rand(64, generator=g) * 1e-2, "bias": torch.randn(64, generator=g)}
    got = run_gpu(inp, shape)
    ref = run_oracle(inp, shape)
    compare(got, ref, "ties")
    # the tie row: q = round-half-even of k + 0.5
    want = [127] + [k if k % 2 == 0 else k + 1 for k in range(-126, 126)]
    assert got["q"][0, :len(want)].tolist() == want


def _tiny_rows(dtype, K):
    """Rows whose smooth products reach the bottom of fp32 (the smooth scale is
    per column, so each row puts its non-zero values in one band of columns):
    products that underflow to zero or to fp32 subnormals, a row whose absmax
    is subnormal (scale subnormal, 1 / scale infinite: the IEEE-division
    fallback), a row whose scale itself underflows to zero, a row of tiny
    normal products, and a mixed row."""
    g = torch.Generator().manual_seed(17)
    band = K // 4
    if dtype == torch.bfloat16:
        # smooth bands: 1, 2^-100, 2^-120, the smallest bf16 subnormal 2^-133
        smooth = torch.cat([torch.ones(band), torch.full((band,), 2.0 ** -100), torch.full((band,), 2.0 ** -120),
                            torch.full((K - 3 * band,), 2.0 ** -133)])
        sub = 2.0 ** -133 * torch.randint(1, 128, (band,), generator=g).double()   # bf16 subnormals
    else:
        # fp16: 1, 2^-14, 2^-20, the smallest fp16 subnormal 2^-24 (no product leaves fp32's normal range)
        smooth = torch.cat([torch.ones(band), torch.full((band,), 2.0 ** -14), torch.full((band,), 2.0 ** -20),
                            torch.full((K - 3 * band,), 2.0 ** -24)])
        sub = 2.0 ** -24 * torch.randint(1, 1024, (band,), generator=g).double()   # fp16 subnormals
    signs = torch.where(torch.rand(K, generator=g) < 0.5, -1.0, 1.0).double()
    rnd = torch.randn(K, generator=g).double() * signs.abs()
    rows = []
    for b in range(4):                                  # one band at a time: normal values
        r = torch.zeros(K, dtype=torch.float64)
        r[b * band:(b + 1) * band] = rnd[b * band:(b + 1) * band] * 1e-3
        rows.append(r)
    r = torch.zeros(K, dtype=torch.float64)             # subnormal inputs in the smooth-1 band
    r[:band] = sub * signs[:band]
    rows.append(r)
    r = torch.zeros(K, dtype=torch.float64)             # subnormal inputs in the smallest band
    r[3 * band:3 * band + band] = sub * signs[:band]
    rows.append(r)
    rows.append(rnd * 4.0)                              # everything at once
    P = torch.stack(rows).to(dtype)
    return P, smooth.to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_tiny_products_and_subnormal_scales(dtype):
    """The fused prologue at the bottom of fp32: smooth products that underflow
    (where its mixed-precision multiply-add and the oracle's fp32 multiply must
    round alike), subnormal absmax and scales (the IEEE-division fallback), a
    scale that underflows to zero; q, the scales and the output bit for bit."""
    R, h = 2, 256
    K = R * h
    P, smooth = _tiny_rows(dtype, K)
    chunks = [P[:, r * h:(r + 1) * h].contiguous() for r in range(R)]
    shape = A2A(rank_size=R, bs_local=P.shape[0], h=h, n=64, quant_mode=7, x1_dtype=dtype)
    g = torch.Generator().manual_seed(5)
    inp = {"chunks": chunks, "x1_scale": smooth,
           "x2": torch.randint(-127, 128, (K, 64), generator=g, dtype=torch.int8),
           "x2_scale": torch.rand(64, generator=g) * 1e-2, "bias": torch.randn(64, generator=g)}
    got = run_gpu(inp, shape)
    ref = run_oracle(inp, shape)
    compare(got, ref, f"tiny {dtype}")
    if dtype == torch.bfloat16:
        sc = ref["x1_scale"]
        assert (sc[(sc > 0)] < 2.0 ** -126).any(), "no row with a subnormal scale"
        assert (sc == 0).any() and (P.double().abs().sum(1)[sc == 0] > 0).any(), "no non-zero row with a zero scale"


@pytest.mark.parametrize("n,mode", [(2560, 3), (4352, 7), (4352, 3)])
def test_partial_last_wave_exact(n, mode):
    """Shapes whose tile count is not a multiple of the co-resident CTA pairs:
    the last partial wave's tiles are split by K blocks across all pairs
    (stream-K) and their int32 partial sums combined; every output element bit
    for bit."""
    shape = A2A(rank_size=8, bs_local=2048, h=512, n=n, quant_mode=mode)   # 8 x (n/256) tiles, 4 K blocks each
    inp = mc2_inputs.a2a_inputs(shape, seed=31)
    got = run_gpu(inp, shape)
    ref = run_oracle(inp, shape)
    compare(got, ref, f"partial wave n={n} mode={mode}")


def test_all_127_bound_over_k_blocks():
    """All-127 operands over eight K blocks, through the stream-K tail: the
    exact int32 partials reach the accumulator bound (8192 * 16129 =
    132128768)."""
    shape = A2A(rank_size=8, bs_local=2048, h=1024, n=2560, quant_mode=3)
    inp = mc2_inputs.a2a_inputs(shape, seed=2)
    inp["chunks"] = [torch.full_like(c, -127) for c in inp["chunks"]]
    inp["x2"] = torch.full_like(inp["x2"], 127)
    got = run_gpu(inp, shape)
    assert torch.all(got["acc"] == -8192 * 16129)
    ref = run_oracle(inp, shape, rows=[0, 1, 1023, 2047])
    compare(got, ref, "all-127", rows=[0, 1, 1023, 2047])


# rank_size * H at the top of the page's range (<= 35000, a multiple of 16):
# 8 x 4368 = 34944 (the per-token quant kernel and the permuted int8 widening,
# the rows being too long for the fused prologue) and 8 x 4096 = 32768 (the
# fused prologue at its largest row, 64 KiB in shared memory).
MAX_K_CASES = {
    "dyn-maxk-34944": A2A(rank_size=8, bs_local=136, h=4368, n=64, quant_mode=7),
    "dyn-maxk-32768-prologue": A2A(rank_size=8, bs_local=136, h=4096, n=64, quant_mode=7),
    "full-maxk-34944": A2A(rank_size=8, bs_local=136, h=4368, n=64, quant_mode=3),
}


@pytest.mark.parametrize("name", sorted(MAX_K_CASES))
def test_largest_rank_h(name):
    shape = MAX_K_CASES[name]
    inp = mc2_inputs.a2a_inputs(shape, seed=14)
    got = run_gpu(inp, shape)
    ref = run_oracle(inp, shape)
    compare(got, ref, name)


def test_stream_k_workspace_needs_no_zeroing():
    """The stream-K flags in the workspace carry a per-launch epoch: a workspace
    full of arbitrary bytes, or holding the flags an earlier launch left, gives
    the same exact result (136 tiles: the 60 after one whole wave are split by
    K blocks over the 76 pairs)."""
    shape = A2A(rank_size=8, bs_local=2048, h=512, n=4352, quant_mode=7)
    inp = mc2_inputs.a2a_inputs(shape, seed=33)
    dev = torch.device("cuda")
    chunks = [c.to(dev) for c in inp["chunks"]]
    args = (chunks, inp["x2"].to(dev), inp["x2_scale"].to(dev), inp["bias"].to(dev))
    nbytes = mc2.mc2_alltoall_quant_mm_workspace(shape.rank_size, shape.bs_local, shape.h, shape.n, 7,
                                                 chunks[0].dtype)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    rows = mc2_inputs.sample_rows(shape.bs_local, 64, seed=5)
    ref = run_oracle(inp, shape, rows=rows)
    outs = []
    for fill in (0x00, 0xA5, 0xFF, None, None):   # None: the previous launch's flags stay
        if fill is not None:
            ws.fill_(fill)
        acc = torch.empty((shape.bs_local, shape.n), dtype=torch.int32, device=dev)
        res = mc2.mc2_alltoall_quant_mm(*args, x1_quant_mode=7, x1_scale=inp["x1_scale"].to(dev), acc_out=acc,
                                        workspace=ws)
        torch.cuda.synchronize()
        assert mc2.mc2_device_status() == mc2.MC2_OK
        assert_bits_equal(acc.cpu()[rows], ref["acc"], f"fill {fill}: acc")
        assert_bits_equal(res["out"].cpu()[rows], ref["out"], f"fill {fill}: out")
        outs.append(res["out"].cpu())
    for o in outs[1:]:
        assert_bits_equal(o, outs[0], "every launch identical")


def _sweep_shapes(count, seed):
    import random
    rng = random.Random(seed)
    shapes = []
    for _ in range(count):
        R = rng.choice([2, 4, 8])
        mode = rng.choice([3, 7])
        h = rng.choice([8, 16, 24, 40, 64, 96, 128, 136, 256, 320, 512])
        if (R * h) % 16:
            h += 8
        bs = rng.choice([1, 7, 64, 100, 128, 129, 200, 256, 300, 513, 1100])
        n = rng.choice([16, 48, 256, 272, 512, 784, 1024, 2048])
        extra = {"x1_dtype": rng.choice([torch.bfloat16, torch.float16])} if mode == 7 else {}
        shapes.append(A2A(rank_size=R, bs_local=bs, h=h, n=n, quant_mode=mode, **extra))
    return shapes


@pytest.mark.parametrize("case,shape", list(enumerate(_sweep_shapes(30, 7))))
def test_seeded_shape_sweep(case, shape):
    """Seeded random shapes: ranks 2/4/8, both quant modes, rows on both sides of
    the one-CTA / CTA-pair boundary (and with stream-K tails), ragged h and n;
    every output bit for bit against the oracle."""
    inp = mc2_inputs.a2a_inputs(shape, seed=100 + case)
    got = run_gpu(inp, shape)
    ref = run_oracle(inp, shape)
    compare(got, ref, f"sweep {case} {shape}")
