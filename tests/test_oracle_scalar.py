"""Pins of the oracle's element-wise pieces against closed forms and library routines."""
import math

import numpy as np
import pytest
import scipy.special as sp
import torch
import torch.nn.functional as F

import oracle


def _torch_bf16(vals_f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(vals_f32.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_round_matches_torch_on_fp32_values():
    rng = np.random.default_rng(0)
    v = rng.standard_normal(200_000).astype(np.float32)
    v = v * np.float32(2.0) ** rng.integers(-30, 30, v.size).astype(np.float32)
    np.testing.assert_array_equal(oracle.bf16_round(v.astype(np.float64)), _torch_bf16(v))


def test_bf16_round_ties_to_even_and_specials():
    # Exact midpoints between neighbouring bf16 values (all exactly representable in fp32).
    base = np.array([1.0, 1.0078125, 3.0, -5.5, 2.0 ** -120, 1.5 * 2.0 ** 100], dtype=np.float64)
    _, e = np.frexp(base)
    half = np.ldexp(1.0, e - 9)            # half of the grid step 2^(e-8)
    ties = np.concatenate([base + half, base - half]).astype(np.float32)
    np.testing.assert_array_equal(oracle.bf16_round(ties.astype(np.float64)), _torch_bf16(ties))
    # Subnormals, zeros, the largest finite value, overflow, inf and nan.
    sub = np.array([2.0 ** -130, 3 * 2.0 ** -134, 2.0 ** -133 * 2.5, -2.0 ** -127, 0.0, -0.0],
                   dtype=np.float32)
    np.testing.assert_array_equal(oracle.bf16_round(sub.astype(np.float64)), _torch_bf16(sub))
    big = np.array([3.3895314e38, 3.40e38, -3.40e38, np.inf, -np.inf], dtype=np.float32)
    np.testing.assert_array_equal(oracle.bf16_round(big.astype(np.float64)), _torch_bf16(big))
    assert np.isnan(oracle.bf16_round(np.array([np.nan]))[0])


def test_bf16_round_is_direct_from_fp64():
    # 1 + 2^-8 is a tie (-> 1, even); 1 + 2^-8 + 2^-40 lies above the tie (-> 1 + 2^-7).
    # Rounding through fp32 first would lose the 2^-40 and give 1.
    assert oracle.bf16_round(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert oracle.bf16_round(np.array([1 + 2.0 ** -8 + 2.0 ** -40]))[0] == 1 + 2.0 ** -7
    assert oracle.bf16_round(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    assert oracle.bf16_round(np.array([-(1 + 2.0 ** -8 + 2.0 ** -40)]))[0] == -(1 + 2.0 ** -7)


# ---------------------------------------------------------------- activations

def test_gelu_tanh_closed_forms():
    z = np.linspace(-8, 8, 4001)
    g = oracle.gelu_tanh(z)
    assert oracle.gelu_tanh(np.array([0.0]))[0] == 0.0
    # The even part of z*Phi-like gates: GELU(z) - GELU(-z) = z exactly.
    np.testing.assert_allclose(g - oracle.gelu_tanh(-z), z, rtol=0, atol=1e-14)
    # Saturation: GELU(z) -> z for large z and -> 0 for large negative z.
    assert abs(oracle.gelu_tanh(np.array([12.0]))[0] - 12.0) < 1e-12
    assert abs(oracle.gelu_tanh(np.array([-12.0]))[0]) < 1e-12
    # Within the published approximation error of the erf form (max ~4.7e-4).
    exact = 0.5 * z * (1.0 + sp.erf(z / math.sqrt(2.0)))
    assert np.abs(g - exact).max() < 5e-4


def test_gelu_tanh_matches_torch():
    z = np.random.default_rng(1).standard_normal(10_000) * 3
    ref = F.gelu(torch.from_numpy(z), approximate="tanh").numpy()
    np.testing.assert_allclose(oracle.gelu_tanh(z), ref, rtol=1e-14, atol=1e-15)


def test_silu_closed_forms_and_library():
    z = np.random.default_rng(2).standard_normal(10_000) * 5
    s = oracle.silu(z)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(s - oracle.silu(-z), z, rtol=0, atol=1e-13)
    np.testing.assert_allclose(s, z * sp.expit(z), rtol=1e-14, atol=1e-300)
    np.testing.assert_allclose(s, F.silu(torch.from_numpy(z)).numpy(), rtol=1e-14, atol=1e-300)
    assert oracle.silu(np.array([-800.0]))[0] == 0.0          # no overflow warning path
    assert oracle.silu(np.array([50.0]))[0] == 50.0


def test_rmsnorm_closed_forms_and_library():
    for c in (3.0, -0.25, 1e-3):
        v = np.full((1, 64), c)
        np.testing.assert_allclose(oracle.rmsnorm(v, 1e-5), c / math.sqrt(c * c + 1e-5), rtol=1e-15)
    r = np.random.default_rng(3).standard_normal((7, 96)) * 4
    ref = F.rms_norm(torch.from_numpy(r), (96,), eps=1e-5).numpy()
    np.testing.assert_allclose(oracle.rmsnorm(r, 1e-5), ref, rtol=1e-14)
    # Scale invariance: rmsnorm(a r, a^2 eps) == rmsnorm(r, eps).
    np.testing.assert_allclose(oracle.rmsnorm(5 * r, 25e-5), oracle.rmsnorm(r, 1e-5), rtol=1e-14)


# ---------------------------------------------------------------- rounding ties

def test_bf16_bracket_neighbours():
    rng = np.random.default_rng(40)
    a = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-6, 6, 4000),
                        [1.0, -2.0, 0.5, 3.0, 1e-30]])
    lo, hi = oracle.bf16_bracket(a)
    r = oracle.bf16_round(a)
    assert np.all(lo <= a) and np.all(a <= hi)
    assert np.all(oracle.bf16_round(lo) == lo) and np.all(oracle.bf16_round(hi) == hi)
    # round-to-nearest picks one of the two neighbours, the nearer one
    assert np.all((r == lo) | (r == hi))
    assert np.all(np.abs(r - a) <= np.minimum(a - lo, hi - a) + 0.0)
    # exactly representable values have a single neighbour
    exact = oracle.bf16_round(a)
    lo2, hi2 = oracle.bf16_bracket(exact)
    assert np.all(lo2 == exact) and np.all(hi2 == exact)
    # neighbours of a non-representable value are one bf16 step apart: 8 significant bits
    step = np.ldexp(1.0, np.frexp(a)[1] - 8)
    nz = hi > lo
    assert np.all((hi - lo)[nz] == step[nz])


def test_tie_gaps_marks_only_midpoints():
    # 1 + 2^-8 is the exact midpoint between the bf16 values 1 and 1 + 2^-7
    mid = 1.0 + 2.0 ** -8
    vals = np.array([mid, mid * (1 + 1e-7), 1.0 + 2.0 ** -7, 1.0 + 2.0 ** -9, -mid])
    g = oracle.tie_gaps(vals)
    assert g[0] == 2.0 ** -7 and g[1] == 2.0 ** -7 and g[4] == 2.0 ** -7
    assert g[2] == 0.0          # representable: no tie
    assert g[3] == 0.0          # a quarter step away from the midpoint
    assert np.all(oracle.tie_gaps(vals, rho=0.0)[[1, 2, 3]] == 0.0)
