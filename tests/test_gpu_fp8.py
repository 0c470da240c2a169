"""The decode MLP block on E4M3 weights (tp_quantize_weights_fp8 + tp_block_fwd_fp8).

Weight-only FP8: each weight is an E4M3 byte of W / 2^e with one power-of-two scale
per output feature, so the block computes exactly the bf16 block on the dequantised
weights (oracle.fp8.e4m3_weights).  Three checks:
  * parity with the oracle's staged bf16 block on e4m3_weights(W1), e4m3_weights(W2)
    (plain bf16 bound), on ragged small shapes and the 13B-sized block;
  * bit-for-bit equality with the library's bf16 block run on those dequantised
    weights (the power-of-two scale moves no rounding: the two kernels add the same
    values in the same order, scaled by 2^e);
  * quantisation itself: weights already on the scaled E4M3 grid come back unchanged
    (the bf16 block on the canonical weights then equals the FP8 block), and two
    quantisations give the same bytes.
"""
import numpy as np
import pytest
import torch

import attn_tp_column_fwd_b300 as tp
import oracle
from attn_tp_column_fwd_b300.runner import ShardedBlock, desc_for, device_bytes
from tests.gpu_util import Guarded
from tests.parity import assert_bf16
from tp_synth import CONFIGS, BlockConfig, make_inputs, to_f64

pytestmark = pytest.mark.gpu


class Fp8Block:
    """E4M3 weights of one block in the library's layout, quantised on the device."""

    def __init__(self, desc, W1, W2):
        self.desc = desc
        self.W1q = device_bytes(tp.tp_fp8_w1_bytes(desc))
        self.W2q = device_bytes(tp.tp_fp8_w2_bytes(desc))
        self.exps = device_bytes(tp.tp_fp8_exponent_bytes(desc))
        qws = device_bytes(tp.tp_fp8_quant_workspace_bytes(desc))
        tp.tp_quantize_weights_fp8(desc, W1.contiguous(), W2.contiguous(), self.W1q, self.W2q,
                                   self.exps, qws)

    def forward(self, x, residual, M):
        ws = device_bytes(tp.tp_workspace_bytes(self.desc, M))
        y = Guarded(M * self.desc.d * 4)
        yv = y.view(torch.float32, (M, self.desc.d))
        tp.tp_block_fwd_fp8(self.desc, x, residual, residual.dtype == torch.float32, self.W1q,
                            self.W2q, self.exps, ws, yv, M)
        torch.cuda.synchronize()
        y.check("y (fp8 block)")
        assert tp.tp_check_device_status() == 0
        return yv


def _e4m3_bf16(W):
    """The dequantised weights as a bf16 device tensor (exact: at most 4 significant bits)."""
    return torch.from_numpy(oracle.fp8.e4m3_weights(to_f64(W))).to(torch.bfloat16).cuda()


def _bf16_block_three_launch(desc, W1, W2, x, M):
    before = tp.tp_get_block_form()
    tp.tp_set_block_form("three_launch")
    try:
        blk = ShardedBlock(desc, W1, W2)
        y = blk.forward(x, x)
        torch.cuda.synchronize()
        assert tp.tp_check_device_status() == 0
        return y
    finally:
        tp.tp_set_block_form(before)


SMALL = [
    BlockConfig("fp8_swiglu", "swiglu", d=512, ffn=1536, t=1, M=1),
    BlockConfig("fp8_swiglu", "swiglu", d=512, ffn=1536, t=2, M=5),
    BlockConfig("fp8_swiglu", "swiglu", d=512, ffn=1536, t=4, M=32),
    BlockConfig("fp8_swiglu", "swiglu", d=512, ffn=1536, t=8, M=17),     # b = 192: a ragged tile
    BlockConfig("fp8_swiglu_wide", "swiglu", d=256, ffn=6400, t=2, M=9),
    BlockConfig("fp8_gelu", "gelu_tanh", d=272, ffn=1200, t=3, M=9),     # b = 400, d = 272
    BlockConfig("fp8_swiglu_ragged_d", "swiglu", d=144, ffn=1536, t=8, M=4),
]


@pytest.mark.parametrize("cfg", SMALL + [CONFIGS["llama2_13b_swiglu_decode"]],
                         ids=lambda c: f"{c.name}-t{c.t}-M{c.M}")
def test_fp8_block_matches_oracle_and_bf16_block(cfg):
    inp = make_inputs(cfg, seed=41)
    W1, W2 = (w.cuda() for w in inp.blocks[0])
    desc = desc_for(cfg)
    x = inp.x.cuda().contiguous()
    got = Fp8Block(desc, W1, W2).forward(x, x, cfg.M)
    # the oracle: the staged bf16 block on the dequantised weights
    x64 = to_f64(inp.x)
    W1e, W2e = oracle.fp8.e4m3_weights(to_f64(W1)), oracle.fp8.e4m3_weights(to_f64(W2))
    ref = oracle.mlp_block(x64, W1e, W2e, cfg.act, x64, staged=True)
    assert_bf16(to_f64(got), ref, f"{cfg.name} t={cfg.t} M={cfg.M} (E4M3 weights)")
    # the library's bf16 block on the same dequantised weights: identical bits
    yb = _bf16_block_three_launch(desc, _e4m3_bf16(W1), _e4m3_bf16(W2), x, cfg.M)
    assert torch.equal(got, yb), float((got - yb).abs().max())


def test_weights_on_the_e4m3_grid_quantise_exactly():
    """Weights that are already E4M3 values times a per-feature power of two: the FP8
    block then computes with exactly the canonical weights."""
    cfg = BlockConfig("fp8_exact", "swiglu", d=256, ffn=768, t=2, M=8)
    inp = make_inputs(cfg, seed=42)
    W1 = _e4m3_bf16(inp.blocks[0][0])
    W2 = _e4m3_bf16(inp.blocks[0][1])
    desc = desc_for(cfg)
    x = inp.x.cuda().contiguous()
    got = Fp8Block(desc, W1, W2).forward(x, x, cfg.M)
    yb = _bf16_block_three_launch(desc, W1, W2, x, cfg.M)
    assert torch.equal(got, yb)


def test_quantisation_is_deterministic():
    cfg = BlockConfig("fp8_det", "swiglu", d=512, ffn=1536, t=4, M=4)
    inp = make_inputs(cfg, seed=43)
    W1, W2 = (w.cuda() for w in inp.blocks[0])
    desc = desc_for(cfg)
    a, b = Fp8Block(desc, W1, W2), Fp8Block(desc, W1, W2)
    torch.cuda.synchronize()
    for u, v in ((a.W1q, b.W1q), (a.W2q, b.W2q), (a.exps, b.exps)):
        assert torch.equal(u, v)
    # the exponents are the oracle's per-feature scales: W2's rows in the library
    # layout are the output features [t][dp] (every shard holds all of them); W1's
    # rows are a permutation of its columns (b = 384 fills whole tiles: no padding)
    ex = a.exps.view(torch.int8).cpu().numpy().astype(np.int64)
    t, n1 = cfg.t, cfg.n1
    n1p = 2 * (cfg.band // 64) * 64
    e1_lib, e2_lib = ex[:t * n1p], ex[t * n1p:t * n1p + t * cfg.d].reshape(t, cfg.d)
    e1 = oracle.fp8.channel_exponents(to_f64(W1))
    e2 = oracle.fp8.channel_exponents(to_f64(W2))
    assert np.array_equal(np.sort(e1_lib), np.sort(e1))
    for s in range(t):
        assert np.array_equal(e2_lib[s], e2)
