"""The comparison rules of the GPU parity tests (tests/parity.py), checked on
the CPU: each must pass what it should and catch a planted difference."""
import pytest
import torch

from parity import ABS_TOL, REL_TOL, assert_bits_equal, assert_close_16, rows_per_block


def _ref16(dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(0)
    return (torch.randn(64, 48, generator=g) * 4).to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_bits_equal_catches_one_flipped_bit(dtype):
    r = _ref16(dtype)
    assert_bits_equal(r.clone(), r, "same")
    g = r.clone().view(torch.int16)
    g[17, 5] ^= 1                       # the lowest mantissa bit of one element
    with pytest.raises(AssertionError, match="1 of 3072 elements differ; first at \\[17, 5\\]"):
        assert_bits_equal(g.view(dtype), r, "flipped")


def test_bits_equal_is_bitwise():
    z = torch.zeros(4, dtype=torch.float32)
    with pytest.raises(AssertionError):
        assert_bits_equal(-z, z, "signed zero")           # -0.0 == 0.0 as numbers, not as bits
    n = torch.full((3,), float("nan"), dtype=torch.bfloat16)
    assert_bits_equal(n.clone(), n, "same NaN bits")
    q = torch.tensor([[1, -2, 127]], dtype=torch.int8)
    q2 = q.clone()
    q2[0, 2] = 126
    with pytest.raises(AssertionError):
        assert_bits_equal(q2, q, "int8")
    with pytest.raises(AssertionError):
        assert_bits_equal(q[:, :2], q, "shape")


def test_close_16_bounds():
    r = _ref16()
    assert_close_16(r.clone(), r)
    # just inside the relative bound on one element passes, just outside fails
    i = (r.double().abs() > 1).nonzero()[0]
    v = r[tuple(i)].double().item()
    inside = r.double().clone()
    inside[tuple(i)] = v * (1 + 0.9 * REL_TOL)
    assert_close_16(inside, r.double())
    outside = r.double().clone()
    outside[tuple(i)] = v * (1 + 1.1 * REL_TOL)
    with pytest.raises(AssertionError, match="1 of 3072 elements outside"):
        assert_close_16(outside, r.double())


def test_close_16_small_values_use_the_absolute_bound():
    r = torch.zeros(8, 8, dtype=torch.float64)
    r[0, 0] = 0.5 * ABS_TOL
    g = r.clone()
    g[0, 0] = 1.4 * ABS_TOL           # relative error 180%, absolute 0.9e-3: passes
    assert_close_16(g, r)
    g[0, 0] = 2.6 * ABS_TOL           # absolute 2.1e-3: fails
    with pytest.raises(AssertionError):
        assert_close_16(g, r)


@pytest.mark.parametrize("bad", [float("nan"), float("inf"), -float("inf")])
def test_close_16_refuses_non_finite(bad):
    r = _ref16().double()
    g = r.clone()
    g[3, 3] = bad
    with pytest.raises(AssertionError, match="non-finite"):
        assert_close_16(g, r)


def test_close_16_refuses_another_shape():
    r = _ref16()
    with pytest.raises(AssertionError):
        assert_close_16(r[:, :47], r)


@pytest.mark.parametrize("total,block", [(16384, 32), (8192, 128), (1000, 32), (31, 32)])
def test_rows_per_block_covers_every_block(total, block):
    extra = (0, total - 1, total // 2)
    rows = rows_per_block(total, block, seed=3, extra=extra)
    assert torch.equal(rows, torch.unique(rows))                       # sorted, no repeats
    assert int(rows.min()) >= 0 and int(rows.max()) < total
    hit = torch.zeros((total + block - 1) // block, dtype=torch.bool)
    hit[rows // block] = True
    assert bool(hit.all()), "a block without a sampled row"
    assert set(extra) <= set(rows.tolist())
    assert torch.equal(rows, rows_per_block(total, block, seed=3, extra=extra))   # seeded
