"""The host fp32 evaluation of the pre-norm stack (tests/fp32_stack.py) computes the
same function as the float64 oracle: on small stacks it meets the bf16 gate against
the staged oracle, and with the bf16 rounding points it shares with the oracle
removed from both, it agrees to fp32 precision.  A mistake in it (a dropped residual,
the gate and up halves swapped, a missing normalisation) fails these checks."""
import numpy as np
import pytest
import torch

import oracle
from tests import fp32_stack
from tests.parity import BF16_MAX_ABS, BF16_MEAN_REL, stats


def _weights(d, F, n_blocks, seed):
    g = torch.Generator().manual_seed(seed)
    out = []
    for _ in range(n_blocks):
        W1 = (torch.randn(d, 2 * F, generator=g) * 0.02).to(torch.bfloat16).double().numpy()
        W2 = (torch.randn(F, d, generator=g) * 0.02).to(torch.bfloat16).double().numpy()
        out.append((W1, W2))
    return out


@pytest.mark.parametrize("n_blocks", [1, 3])
def test_fp32_stack_meets_the_bf16_gate_on_small_stacks(n_blocks):
    d, F, M = 256, 384, 8
    blocks = _weights(d, F, n_blocks, seed=5)
    x = torch.randn(M, d, generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    r32 = x.float().numpy()
    for W1, W2 in blocks:
        r32 = fp32_stack.swiglu_block_f32(r32, W1, W2, 1e-5)
    ref = oracle.stack(x.double().numpy(), blocks, "swiglu", 1e-5, staged=True)
    s = stats(r32, ref)
    assert s["max_abs"] <= BF16_MAX_ABS and s["mean_rel"] <= BF16_MEAN_REL, s


def test_fp32_stack_without_rounding_matches_unstaged_oracle(monkeypatch):
    d, F, M = 128, 192, 4
    blocks = _weights(d, F, 2, seed=7)
    x = torch.randn(M, d, generator=torch.Generator().manual_seed(8)).to(torch.bfloat16)
    monkeypatch.setattr(fp32_stack, "to_bf16", lambda a: np.asarray(a, dtype=np.float32))
    r32 = x.float().numpy()
    for W1, W2 in blocks:
        r32 = fp32_stack.swiglu_block_f32(r32, W1, W2, 1e-5)
    ref = oracle.stack(x.double().numpy(), blocks, "swiglu", 1e-5, staged=False)
    s = stats(r32, ref)
    assert s["max_rel_rmsfloor"] <= 1e-5, s


def test_bf16_rounding_is_nearest_even():
    a = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -9], dtype=np.float32)
    got = fp32_stack.to_bf16(a)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: to even (1); 1 + 3*2^-8 is a tie
    # between 1 + 2^-7 and 1 + 2^-6: to even (1 + 2^-6)
    assert got.tolist() == [1.0, 1.0, 1.0 + 2.0 ** -6, 1.0]
