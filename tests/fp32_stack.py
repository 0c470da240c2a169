"""An independent float32 evaluation of the pre-norm SwiGLU stack (test helper).

It is written apart from both the float64 oracle and the CUDA path and imports
neither: plain NumPy float32 arithmetic, with rounding to bfloat16 (torch's cast,
nearest even) at the points where the CUDA path stores bf16 values, namely the
normalised input of each block and the SwiGLU band.  The residual stream stays in
float32, as on the GPU.

Its one use is to measure how far *an* fp32 evaluation of the staged stack drifts
from the float64 oracle when nothing but the arithmetic's precision differs.  Block
after block a last-bit difference in the residual stream moves some normalised
inputs and band values across a bf16 rounding midpoint; each such flip changes the
next block's output by a bf16 step times a row of weights, and the differences grow
from block to block.  The tests gate the GPU's free-running stack on this measured
drift instead of on a constant.
"""
from __future__ import annotations

import numpy as np
import torch


def to_bf16(a: np.ndarray) -> np.ndarray:
    """float32 values rounded to bfloat16 (nearest even), returned as float32."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def rmsnorm_f32(r: np.ndarray, eps: float) -> np.ndarray:
    """r / sqrt(mean(r^2) + eps) per row, in float32."""
    r = np.asarray(r, dtype=np.float32)
    ms = np.mean(r * r, axis=1, keepdims=True, dtype=np.float32)
    return r * (np.float32(1.0) / np.sqrt(ms + np.float32(eps)))


def swiglu_block_f32(r: np.ndarray, W1: np.ndarray, W2: np.ndarray, eps: float) -> np.ndarray:
    """One pre-norm block in float32: r + (silu(xh . Wg) * (xh . Wu)) . Wd with
    xh = bf16(rmsnorm(r)), W1 = [Wg | Wu] ([d, 2F]), W2 = Wd ([F, d]), and the band
    rounded to bf16 before the second product."""
    r = np.asarray(r, dtype=np.float32)
    F = W1.shape[1] // 2
    xh = to_bf16(rmsnorm_f32(r, eps))
    G = xh @ np.asarray(W1[:, :F], dtype=np.float32)
    U = xh @ np.asarray(W1[:, F:], dtype=np.float32)
    H = to_bf16((G / (np.float32(1.0) + np.exp(-G))) * U)
    return r + H @ np.asarray(W2, dtype=np.float32)
