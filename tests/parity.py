"""Comparison rules shared by the GPU parity tests.

Floating-point outputs of the bf16/fp16 matmul: max relative error 1e-2 where
|ref| > 1e-3, absolute error 1e-3 elsewhere (the GPU accumulates in fp32, the
oracle in fp64; both round once to the output type).  Integer and byte outputs
(gathered, q, accumulators) and the dequant output (an exact integer
accumulator followed by the same fp32 operations on both sides) are compared
bit for bit.
"""
import torch

REL_TOL = 1e-2
ABS_TOL = 1e-3


def assert_close_16(got: torch.Tensor, ref: torch.Tensor, what: str = "out"):
    g = got.detach().cpu().double()
    r = ref.detach().cpu().double()
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert torch.isfinite(g).all(), f"{what}: non-finite values"
    err = (g - r).abs()
    big = r.abs() > ABS_TOL
    rel = torch.where(big, err / r.abs().clamp_min(1e-30), torch.zeros_like(err))
    small_err = torch.where(big, torch.zeros_like(err), err)
    worst_rel = rel.max().item() if rel.numel() else 0.0
    worst_abs = small_err.max().item() if small_err.numel() else 0.0
    if not (worst_rel <= REL_TOL and worst_abs <= ABS_TOL):
        idx = tuple(int(i) for i in (rel == rel.max()).nonzero()[0])
        nbad = int(((rel > REL_TOL) | (small_err > ABS_TOL)).sum())
        raise AssertionError(
            f"{what}: max rel err {worst_rel:.3e} (tol {REL_TOL}), max abs err on small values {worst_abs:.3e}; "
            f"{nbad} of {g.numel()} elements outside; worst at {idx}: got {g[idx].item():.6e} ref {r[idx].item():.6e}")


def assert_bits_equal(got: torch.Tensor, ref: torch.Tensor, what: str):
    g = got.detach().cpu()
    r = ref.detach().cpu()
    assert g.shape == r.shape, (what, g.shape, r.shape)
    if g.dtype in (torch.bfloat16, torch.float16):
        g, r = g.view(torch.int16), r.view(torch.int16)
    elif g.dtype == torch.float32:
        g, r = g.view(torch.int32), r.view(torch.int32)
    if not torch.equal(g, r):
        bad = (g != r).nonzero()
        raise AssertionError(f"{what}: {bad.shape[0]} of {g.numel()} elements differ; first at {bad[0].tolist()}: "
                             f"got {g[tuple(bad[0])].item()} want {r[tuple(bad[0])].item()}")


def rows_per_block(total: int, block: int, seed: int, extra=()) -> torch.Tensor:
    """Sorted row indices: one seeded row inside every `block`-row block of
    [0, total) (block 32 = the rows one epilogue warp of a CTA writes), plus the
    rows in `extra` (chunk edges).  Used where the oracle cannot afford every
    output row of a full-size workload."""
    g = torch.Generator().manual_seed(seed)
    starts = torch.arange(0, total, block)
    span = torch.clamp(total - starts, max=block)
    offs = (torch.rand(starts.numel(), generator=g) * span).long()
    rows = torch.cat([starts + offs, torch.tensor(list(extra), dtype=torch.long)])
    return torch.unique(rows[(rows >= 0) & (rows < total)])
