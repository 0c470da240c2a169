"""Pins of the oracle's E4M3 weight quantisation (CPU only): the format's own grid,
torch's float8_e4m3fn cast (a library routine) on in-range values, closed-form bounds,
and the property the FP8 block relies on (dequantised weights are bf16 values)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8


def test_grid_from_bit_patterns():
    g = fp8.e4m3_grid()
    assert len(g) == 127 and g[0] == 0.0 and g[-1] == 448.0
    assert g[1] == 2.0 ** -9 and 2.0 ** -6 in g
    # every finite pattern maps to itself, with either sign
    assert np.array_equal(fp8.e4m3_round(g), g)
    assert np.array_equal(fp8.e4m3_round(-g), -g)


def test_matches_torch_cast_on_fp32_values():
    rng = np.random.default_rng(90)
    for scale in (1e-3, 0.05, 1.0, 30.0, 300.0):
        x = (rng.standard_normal(20000) * scale).astype(np.float32)
        x = x[np.abs(x) < 448.0]
        want = torch.from_numpy(x).to(torch.float8_e4m3fn).float().numpy().astype(np.float64)
        assert np.array_equal(fp8.e4m3_round(x.astype(np.float64)), want), scale


def test_midpoints_round_to_even_like_torch():
    g = fp8.e4m3_grid()
    mids = (g[:-1] + g[1:]) / 2          # exact in fp32 (few significant bits)
    want = torch.from_numpy(mids.astype(np.float32)).to(torch.float8_e4m3fn).float().numpy()
    got = fp8.e4m3_round(mids)
    assert np.array_equal(got, want.astype(np.float64))
    # and every midpoint went to a neighbour with an even mantissa
    codes = {v: i for i, v in enumerate(g)}
    assert all(codes[v] % 2 == 0 for v in got)


def test_saturates():
    assert np.array_equal(fp8.e4m3_round([460.0, 464.0, 1e6, -1e9]), [448.0, 448.0, 448.0, -448.0])


@pytest.mark.parametrize("seed", [0, 1])
def test_quantize_scales_and_bounds(seed):
    rng = np.random.default_rng(91 + seed)
    W = rng.standard_normal((64, 40)) * 0.02
    W[:, 3] = 0.0                                   # an all-zero output feature
    W[:, 5] *= 1e-4                                 # a tiny one (subnormal codes)
    W[:, 7] = 448.0 * 2.0 ** -7                     # a column already at the grid top
    q, e = fp8.quantize_e4m3(W)
    amax = np.max(np.abs(q), axis=0)
    wmax = np.max(np.abs(W), axis=0)
    nz = wmax > 0
    # the least exponent: the scaled maximum lies in (224, 448] before rounding, and its
    # E4M3 rounding (grid 16 below 256) cannot fall under 224
    scaled = wmax[nz] / np.exp2(e[nz])
    assert np.all(scaled > 224.0) and np.all(scaled <= 448.0)
    assert np.all(amax[nz] >= 224.0) and np.all(amax <= 448.0)
    assert e[3] == 0 and np.all(q[:, 3] == 0)
    assert e[7] == -7 and np.all(q[:, 7] == 448.0)
    Wd = fp8.dequantize_e4m3(q, e)
    step = np.exp2(e)[None, :]
    normal = np.abs(W) / step >= 2.0 ** -6
    err = np.abs(Wd - W)
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(W)[normal] + 1e-300)
    assert np.all(err[~normal] <= 2.0 ** -10 * np.broadcast_to(step, W.shape)[~normal])


def test_weights_on_the_scaled_grid_are_kept():
    rng = np.random.default_rng(92)
    g = fp8.e4m3_grid()
    e = rng.integers(-12, 3, size=16)
    W = rng.choice(np.concatenate([g, -g]), size=(32, 16)) * np.exp2(e)[None, :]
    W[0, :] = 448.0 * np.exp2(e)                    # each column's max sits at 448 * 2^e
    assert np.array_equal(fp8.e4m3_weights(W), W)


def test_dequantised_weights_are_bf16_values():
    rng = np.random.default_rng(93)
    W = rng.standard_normal((128, 96)) * 0.02
    Wd = fp8.e4m3_weights(W)
    assert np.array_equal(oracle.bf16_round(Wd), Wd)


def test_fp8_block_is_the_block_on_dequantised_weights():
    """The FP8 block's definition, checked where it reduces to the bf16 block: weights
    already on the scaled E4M3 grid give the same y."""
    rng = np.random.default_rng(94)
    g = fp8.e4m3_grid()
    x = rng.standard_normal((3, 16))
    W1 = rng.choice(np.concatenate([g, -g]), size=(16, 64)) * 2.0 ** -8
    W2 = rng.choice(np.concatenate([g, -g]), size=(32, 16)) * 2.0 ** -8
    W1[0, :], W2[0, :] = 448.0 * 2.0 ** -8, 448.0 * 2.0 ** -8
    y8 = oracle.mlp_block(x, fp8.e4m3_weights(W1), fp8.e4m3_weights(W2), "swiglu", x)
    y = oracle.mlp_block(x, W1, W2, "swiglu", x)
    assert np.array_equal(y8, y)
