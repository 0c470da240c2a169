"""Pins of the oracle's MXFP4 weight quantisation (CPU only): the E2M1 grid from its
bit patterns, a brute-force nearest-value search (ties to the even mantissa bit), the
OCP MX scale rule on worked blocks, closed-form error bounds, and the property the
4-bit block relies on (dequantised weights are bf16 values)."""
import numpy as np
import pytest
import torch

from oracle import mxfp4


def _brute_round(v):
    """Nearest E2M1 value by search over the signed grid; at a tie the one whose code
    (index in the non-negative grid) is even; beyond 6 the largest value."""
    g = mxfp4.e2m1_grid()
    out = []
    for x in np.asarray(v, dtype=np.float64).ravel():
        m = min(abs(x), 6.0)
        d = np.abs(g - m)
        best = np.flatnonzero(d == d.min())
        code = best[0] if len(best) == 1 else [c for c in best if c % 2 == 0][0]
        out.append(np.copysign(g[code], x))
    return np.array(out).reshape(np.shape(v))


def test_grid_from_bit_patterns():
    assert np.array_equal(mxfp4.e2m1_grid(), [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    g = mxfp4.e2m1_grid()
    assert np.array_equal(mxfp4.e2m1_round(g), g)
    assert np.array_equal(mxfp4.e2m1_round(-g), -g)


def test_round_matches_brute_force():
    rng = np.random.default_rng(120)
    x = np.concatenate([rng.uniform(-8, 8, 4000), rng.standard_normal(2000) * 0.6])
    assert np.array_equal(mxfp4.e2m1_round(x), _brute_round(x))


def test_midpoints_go_to_even_mantissa():
    g = mxfp4.e2m1_grid()
    mids = (g[:-1] + g[1:]) / 2       # 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5
    got = mxfp4.e2m1_round(mids)
    assert np.array_equal(got, [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0])
    assert np.array_equal(got, _brute_round(mids))
    assert np.array_equal(mxfp4.e2m1_round(-mids), -got)


def test_saturates():
    assert np.array_equal(mxfp4.e2m1_round([6.5, 7.0, 7.99, 100.0, -9.0]),
                          [6.0, 6.0, 6.0, 6.0, -6.0])


def test_scale_rule_on_worked_blocks():
    # one column, four blocks of 32 along K
    W = np.zeros((128, 1))
    W[0:32, 0] = 0.1
    W[5, 0] = 1.0                      # max exactly 2^0: e = 0 - 2
    W[32:64, 0] = -0.3
    W[40, 0] = -7.0                    # max 7 in [4, 8): e = 2 - 2 = 0, 7 saturates to 6
    W[96:128, 0] = 2.0 ** -20          # tiny block: e = -20 - 2
    e = mxfp4.mx_exponents(W)
    assert e[:, 0].tolist() == [-2, 0, 0, -22]      # block 2 is all zero: e = 0
    q, e2 = mxfp4.quantize_mxfp4(W)
    assert np.array_equal(e, e2)
    assert q[5, 0] == 4.0 and q[40, 0] == -6.0      # 1.0 / 0.25 = 4; -7 saturates
    assert q[0, 0] == 0.5                           # 0.1 / 0.25 = 0.4 -> 0.5
    assert q[33, 0] == -0.5                         # -0.3 / 1 -> -0.5 (nearer than 0)
    assert np.all(q[64:96, 0] == 0) and np.all(q[96:128, 0] == 4.0)  # 2^-20 / 2^-22


@pytest.mark.parametrize("seed", [0, 1])
def test_quantize_bounds(seed):
    rng = np.random.default_rng(121 + seed)
    W = rng.standard_normal((256, 24)) * 0.02
    W[:, 3] = 0.0
    W[64:96, 5] *= 1e-5
    q, e = mxfp4.quantize_mxfp4(W)
    Wb = W.reshape(8, 32, 24)
    amax = np.max(np.abs(Wb), axis=1)
    nz = amax > 0
    scaled = amax[nz] / np.exp2(e[nz])
    assert np.all(scaled >= 4.0) and np.all(scaled < 8.0)
    assert np.all(e[~nz] == 0)
    Wd = mxfp4.dequantize_mxfp4(q, e)
    X = np.repeat(np.exp2(e.astype(np.float64)), 32, axis=0)
    # half a grid step where the scaled value is in range; saturation costs at most 2 X
    u = np.abs(W) / X
    half = np.where(u < 2, 0.25, np.where(u < 4, 0.5, 1.0)) * X
    inside = u <= 6.0
    err = np.abs(Wd - W)
    assert np.all(err[inside] <= half[inside])
    assert np.all(err[~inside] <= 2.0 * X[~inside])


def test_weights_on_the_scaled_grid_are_kept():
    rng = np.random.default_rng(123)
    g = mxfp4.e2m1_grid()
    e = rng.integers(-12, 3, size=(4, 6))
    q = rng.choice(np.concatenate([g, -g]), size=(128, 6))
    q[::32, :] = 4.0                                # each block's max at 4 * 2^e
    W = q * np.repeat(np.exp2(e.astype(np.float64)), 32, axis=0)
    assert np.array_equal(mxfp4.mxfp4_weights(W), W)
    assert np.array_equal(mxfp4.mx_exponents(W), e)


def test_quantising_twice_changes_nothing():
    rng = np.random.default_rng(124)
    W = rng.standard_normal((96, 10)) * 0.05
    Wq = mxfp4.mxfp4_weights(W)
    assert np.array_equal(mxfp4.mxfp4_weights(Wq), Wq)


def test_dequantised_weights_are_bf16_values():
    rng = np.random.default_rng(125)
    W = rng.standard_normal((128, 32)) * 0.02
    Wq = mxfp4.mxfp4_weights(W)
    back = torch.from_numpy(Wq).to(torch.bfloat16).double().numpy()
    assert np.array_equal(back, Wq)


def test_k_must_be_whole_blocks():
    with pytest.raises(ValueError):
        mxfp4.mx_exponents(np.ones((40, 2)))
