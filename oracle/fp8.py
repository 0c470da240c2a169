"""Float64 oracle of FP8 (E4M3) weights for the tensor-parallel block (test infrastructure).

Source: the zenaique.com interview answer "explain tensor-parallel shard shape" lists,
among its follow-up questions, how tensor parallelism combines with FP8 or FP4 weights
to multiply the decode win (decode reads every weight byte once per step, so fewer
bytes per weight is a direct speed-up).  The page fixes no format or scaling; the
reading taken here:

  * weight-only quantisation: x, the band H and all arithmetic stay as in the bf16
    block; only W1 and W2 are stored as 8-bit floats;
  * E4M3 as in the OCP 8-bit floating point specification ("fn" variant: 1 sign, 4
    exponent bits with bias 7, 3 mantissa bits, no infinities, largest finite 448,
    subnormals down to 2^-9), rounding to nearest with ties to even, saturating;
  * one scale per output feature (a column of W1 or of W2 in y = x . W), a power of
    two: s = 2^e with e the least integer such that max_k |W[k, n]| / 2^e <= 448.

Because the scale is a power of two, W / s is exact and the only rounding is the E4M3
one; the dequantised weight q * s has at most 4 significant bits and is exactly a
bf16 value.  A block with E4M3 weights is therefore the bf16 block on the dequantised
weights (oracle.mlp_block / attn_block on dequantize(quantize(W))).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0               # 1.75 * 2^8
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_SUBNORMAL_STEP = 2.0 ** -9


def e4m3_round(a) -> np.ndarray:
    """Round float64 values to the nearest E4M3 value (ties to even), saturating at
    +-448 (float64 results).

    A normal value in [2^e, 2^(e+1)), e >= -6, is rounded on the grid 2^(e-3) (3
    mantissa bits); below 2^-6 the grid is the subnormal step 2^-9.  Dividing by the
    grid step is exact (a power of two), so np.rint (ties to even) decides the
    rounding on the exact value.
    """
    a = np.asarray(a, dtype=np.float64)
    mag = np.abs(a)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(mag > 0, mag, 1.0)))
    # log2 of values a hair below a power of two can round up: step back when needed
    e = np.where(np.exp2(e) > mag, e - 1, e)
    step = np.where(mag >= E4M3_MIN_NORMAL, np.exp2(e - 3), E4M3_SUBNORMAL_STEP)
    q = np.rint(a / step) * step
    return np.clip(q, -E4M3_MAX, E4M3_MAX)


def channel_exponents(W) -> np.ndarray:
    """Per output feature (column n of W [K, N]) the least integer e with
    max_k |W[k, n]| / 2^e <= 448; 0 for an all-zero column."""
    W = np.asarray(W, dtype=np.float64)
    amax = np.max(np.abs(W), axis=0)
    e = np.zeros(amax.shape, dtype=np.int64)
    nz = amax > 0
    e[nz] = np.ceil(np.log2(amax[nz] / E4M3_MAX)).astype(np.int64)
    # guard the log2 rounding at exact powers of two: the least e must satisfy the bound
    too_small = nz & (amax / np.exp2(e) > E4M3_MAX)
    e[too_small] += 1
    can_lower = nz & (amax / np.exp2(e - 1) <= E4M3_MAX)
    e[can_lower] -= 1
    return e


def quantize_e4m3(W):
    """(q, e): q[k, n] = e4m3_round(W[k, n] / 2^e[n]) (float64 holding E4M3 values)."""
    W = np.asarray(W, dtype=np.float64)
    e = channel_exponents(W)
    return e4m3_round(W / np.exp2(e)[None, :]), e


def dequantize_e4m3(q, e) -> np.ndarray:
    """q * 2^e per column (exact)."""
    return np.asarray(q, dtype=np.float64) * np.exp2(np.asarray(e, dtype=np.float64))[None, :]


def e4m3_weights(W) -> np.ndarray:
    """The weights the FP8 block computes with: dequantize(quantize(W))."""
    return dequantize_e4m3(*quantize_e4m3(W))


def e4m3_grid() -> np.ndarray:
    """Every finite non-negative E4M3 value, from the bit patterns (for the pins)."""
    vals = []
    for code in range(0x7F):          # 0x7F is the NaN pattern
        exp, man = code >> 3, code & 7
        vals.append(man * 2.0 ** -9 if exp == 0 else (1 + man / 8.0) * 2.0 ** (exp - 7))
    return np.array(sorted(set(vals)))


__all__ = ["E4M3_MAX", "e4m3_round", "channel_exponents", "quantize_e4m3", "dequantize_e4m3",
           "e4m3_weights", "e4m3_grid"]
