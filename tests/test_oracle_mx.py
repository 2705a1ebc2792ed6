"""MXFP8 quantise-dequantise of the oracle against independent facts.

The element grid and its rounding are pinned to torch's float8_e4m3fn
conversion (a library routine); the block scale to the OCP MX v1.0 rule on
worked values; plus exactness on representable blocks, the zero block,
saturation, the error bound and token-axis partial blocks.
"""
import numpy as np
import pytest
import torch

from oracle import mx


def e4m3_grid():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    vals = vals[np.isfinite(vals)]
    return np.unique(vals)


def test_grid_matches_library():
    grid = e4m3_grid()
    assert grid.max() == 448.0 and grid.min() == -448.0
    pos = grid[grid > 0]
    assert pos.min() == 2.0 ** -9                     # smallest subnormal
    assert np.array_equal(mx.e4m3_round(grid), grid)  # every grid value is a fixed point


def test_rounding_matches_library_random_and_ties():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(20000) * 40,
                        rng.standard_normal(20000) * 0.01,
                        rng.uniform(-448, 448, 20000)])
    grid = e4m3_grid()
    mids = (grid[1:] + grid[:-1]) / 2.0               # exact ties in fp64
    v = np.concatenate([v, mids])
    lib = torch.from_numpy(v).to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    # fp32 is exact for these values (the midpoints need at most 5 significant bits)
    assert np.array_equal(torch.from_numpy(v).to(torch.float32).double().numpy()[-mids.size:], mids)
    ours = mx.e4m3_round(v)
    assert np.array_equal(ours, lib)


def test_saturation():
    v = np.array([448.0, 449.0, 463.99, 464.0, 500.0, 1e6, -1e6, -470.0])
    assert np.array_equal(mx.e4m3_round(v), [448, 448, 448, 448, 448, 448, -448, -448])


def test_scale_rule_worked_values():
    amax = np.array([448.0, 256.0, 511.9, 1.0, 0.75, 2.0 ** -120, 0.0, 3e38])
    # floor(log2 amax) - 8, clipped to the E8M0 range, -127 for a zero block
    assert mx.e8m0_scale_exponent(amax).tolist() == [0, 0, 0, -8, -9, -127, -127, 119]


def test_exact_on_representable_blocks():
    rng = np.random.default_rng(1)
    grid = e4m3_grid()
    for s_exp in (-20, -8, 0, 5):
        blk = rng.choice(grid, size=(16, 32))
        blk[:, 0] = 256.0 * rng.choice([1.0, 1.25, 1.5, 1.75], size=16)   # amax in [256, 448]
        blk *= 2.0 ** s_exp
        assert np.array_equal(mx.mx_qdq(blk, axis=1), blk)


def test_zero_block_and_mixed():
    v = np.zeros((3, 64))
    v[1, 40] = 3.0
    q = mx.mx_qdq(v, axis=1)
    assert np.array_equal(q[0], np.zeros(64)) and q[1, 40] == 3.0
    assert np.count_nonzero(q) == 1


def test_error_bound_and_monotone():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((64, 256)) * np.exp(rng.uniform(-5, 5, (64, 1)))
    q = mx.mx_qdq(v, axis=1)
    blocks = v.reshape(64, 8, 32)
    s = np.exp2(mx.e8m0_scale_exponent(np.abs(blocks).max(axis=2)))[..., None]
    s = np.broadcast_to(s, blocks.shape).reshape(64, 256)
    bound = np.maximum.reduce([np.abs(v) * 2.0 ** -4,      # half an ulp, 3 mantissa bits
                               s * 2.0 ** -10,             # half the subnormal step
                               np.abs(v) - 448.0 * s])     # saturation
    assert np.all(np.abs(q - v) <= bound * (1 + 1e-12))
    x = np.sort(rng.standard_normal(4096) * 100)
    assert np.all(np.diff(mx.e4m3_round(x)) >= 0)


def test_partial_token_blocks_are_zero_padded():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((40, 5))
    q = mx.mx_qdq(v, axis=0)
    assert np.array_equal(q[:32], mx.mx_qdq(v[:32], axis=0))
    assert np.array_equal(q[32:], mx.mx_qdq(v[32:], axis=0))


@pytest.mark.parametrize("axis", [0, 1])
def test_axis(axis):
    rng = np.random.default_rng(4)
    v = rng.standard_normal((64, 96))
    q = mx.mx_qdq(v, axis=axis)
    qt = mx.mx_qdq(v.T, axis=1 - axis).T
    assert np.array_equal(q, qt)


def test_planted_rounding_mistake_is_caught(monkeypatch):
    """Round-half-away-from-zero instead of ties-to-even is caught by the library pin."""
    def bad(q):
        q = np.asarray(q, dtype=np.float64)
        a = np.abs(q)
        e = np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), mx.E4M3_EMIN)
        step = np.exp2(e - mx.E4M3_MBITS)
        return np.copysign(np.minimum(np.floor(a / step + 0.5) * step, 448.0), q)
    monkeypatch.setattr(mx, "e4m3_round", bad)
    with pytest.raises(AssertionError):
        test_rounding_matches_library_random_and_ties()
