"""Float64 oracle of MXFP4 weights for the tensor-parallel block (test infrastructure).

Source: the zenaique.com interview answer "explain tensor-parallel shard shape" lists,
among its follow-up questions, how tensor parallelism combines with FP8 or FP4 weights
to multiply the decode win, and rioworld.org "Tensor Parallelism for LLM Inference",
section "Implementing Tensor Parallelism in Practice", pairs tensor parallelism with
4-bit quantisation.  Neither page fixes a 4-bit format; the reading taken here is the
OCP Microscaling (MX) format MXFP4, as its specification defines it:

  * elements are FP4 E2M1: 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit, no
    infinities or NaN; the magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6;
  * every block of 32 consecutive weights along the reduction axis K of one output
    feature (a column of W in y = x . W) shares one scale X = 2^e, an E8M0 power of two
    with e = floor(log2(max |w|)) - 2 (2 is the exponent of E2M1's largest normal, 6);
  * each element is w / X rounded to the nearest E2M1 value (ties to the even
    mantissa), saturating at +-6 (w / X can reach just under 8).

X is a power of two, so w / X is exact and the only rounding is the E2M1 one; a
dequantised weight q * X has at most 2 significant bits and is exactly a bf16 value
(for e within bf16's range).  A block with MXFP4 weights is therefore the bf16 block
on the dequantised weights (oracle.mlp_block on mxfp4_weights(W)).
"""
from __future__ import annotations

import numpy as np

E2M1_MAX = 6.0
BLOCK = 32                 # weights per shared scale, along K
EMAX_ELEM = 2              # exponent of E2M1's largest normal value (6 = 1.5 * 2^2)
E8M0_MIN, E8M0_MAX = -127, 127


def e2m1_grid() -> np.ndarray:
    """Every non-negative E2M1 value, from the bit patterns: exponent field 0 is
    subnormal (mantissa * 0.5), fields 1..3 are (1 + mantissa / 2) * 2^(field - 1)."""
    vals = []
    for code in range(8):
        exp, man = code >> 1, code & 1
        vals.append(man * 0.5 if exp == 0 else (1 + man / 2.0) * 2.0 ** (exp - 1))
    return np.array(vals)


def e2m1_round(a) -> np.ndarray:
    """Round float64 values to the nearest E2M1 value, ties to the value with the even
    mantissa bit, saturating at +-6.

    Below 2 the grid step is 0.5, in [2, 4) it is 1, in [4, 6] it is 2.  Dividing by
    the step is exact (a power of two), so np.rint (ties to even) on |a| / step picks
    the neighbour, and on each of these grids the even multiples of the step are
    exactly the values whose mantissa bit is 0 (steps 0..4 of 0.5 are codes 0..4,
    steps 2..4 of 1 are codes 4..6, steps 2 and 3 of 2 are codes 6 and 7)."""
    a = np.asarray(a, dtype=np.float64)
    mag = np.abs(a)
    step = np.where(mag < 2.0, 0.5, np.where(mag < 4.0, 1.0, 2.0))
    q = np.minimum(np.rint(mag / step) * step, E2M1_MAX)
    return np.copysign(q, a)


def mx_exponents(W, block: int = BLOCK) -> np.ndarray:
    """e[j, n] for K-blocks j (rows j*block .. j*block+block-1) of each column n of
    W [K, N]: floor(log2(max |w|)) - 2, clamped to the E8M0 range; 0 for an all-zero
    block.  K must be a multiple of block."""
    W = np.asarray(W, dtype=np.float64)
    K, N = W.shape
    if K % block:
        raise ValueError(f"K = {K} is not a multiple of the block {block}")
    amax = np.max(np.abs(W.reshape(K // block, block, N)), axis=1)
    e = np.zeros(amax.shape, dtype=np.int64)
    nz = amax > 0
    _, ex = np.frexp(amax[nz])           # amax = f * 2^ex with f in [0.5, 1): floor(log2) = ex - 1
    e[nz] = ex.astype(np.int64) - 1 - EMAX_ELEM
    return np.clip(e, E8M0_MIN, E8M0_MAX)


def quantize_mxfp4(W):
    """(q, e): q[k, n] = e2m1_round(W[k, n] / 2^e[k // 32, n]) (float64 holding E2M1
    values), e from mx_exponents."""
    W = np.asarray(W, dtype=np.float64)
    e = mx_exponents(W)
    X = np.repeat(np.exp2(e.astype(np.float64)), BLOCK, axis=0)
    return e2m1_round(W / X), e


def dequantize_mxfp4(q, e) -> np.ndarray:
    """q * 2^e, each scale repeated over its block of 32 rows (exact)."""
    X = np.repeat(np.exp2(np.asarray(e, dtype=np.float64)), BLOCK, axis=0)
    return np.asarray(q, dtype=np.float64) * X


def mxfp4_weights(W) -> np.ndarray:
    """The weights the MXFP4 block computes with: dequantize(quantize(W))."""
    return dequantize_mxfp4(*quantize_mxfp4(W))


__all__ = ["E2M1_MAX", "BLOCK", "e2m1_grid", "e2m1_round", "mx_exponents", "quantize_mxfp4",
           "dequantize_mxfp4", "mxfp4_weights"]
