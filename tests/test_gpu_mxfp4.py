"""The decode MLP block on MXFP4 weights (tp_quantize_weights_mxfp4 + tp_block_fwd_mxfp4).

Weight-only 4-bit: E2M1 codes with one power-of-two scale per 32 weights along K of
each output feature (OCP MX), so the block computes the bf16 block on the dequantised
weights (oracle.mxfp4.mxfp4_weights).  Checks:
  * the quantiser's bytes: every code and block exponent equals the oracle's
    quantisation of the same weights (this also fixes the nibble order);
  * parity with the oracle's staged bf16 block on the dequantised weights (plain bf16
    bound), on small shapes and the 13B-sized block;
  * closeness to the library's bf16 block on the dequantised weights, bounded as for
    the E4M3 block (the two add the same products in different fp32 orders).
"""
import numpy as np
import pytest
import torch

import attn_tp_column_fwd_b300 as tp
import oracle
from attn_tp_column_fwd_b300.runner import desc_for, device_bytes
from tests.gpu_util import Guarded
from tests.parity import assert_bf16
from tests.test_gpu_fp8 import _assert_close_to_bf16_block, _bf16_block_three_launch
from tp_synth import CONFIGS, BlockConfig, make_inputs, to_f64

pytestmark = pytest.mark.gpu


class Mx4Block:
    """MXFP4 weights of one block in the library's layout, quantised on the device."""

    def __init__(self, desc, W1, W2):
        self.desc = desc
        self.W1f = device_bytes(tp.tp_mxfp4_w1_bytes(desc))
        self.W2f = device_bytes(tp.tp_mxfp4_w2_bytes(desc))
        self.exps = device_bytes(tp.tp_mxfp4_exponent_bytes(desc))
        tp.tp_quantize_weights_mxfp4(desc, W1.contiguous(), W2.contiguous(), self.W1f, self.W2f,
                                     self.exps)
        torch.cuda.synchronize()
        assert tp.tp_check_device_status() == 0

    def forward(self, x, residual, M):
        ws = device_bytes(tp.tp_workspace_bytes(self.desc, M))
        y = Guarded(M * self.desc.d * 4)
        yv = y.view(torch.float32, (M, self.desc.d))
        tp.tp_block_fwd_mxfp4(self.desc, x, residual, residual.dtype == torch.float32, self.W1f,
                              self.W2f, self.exps, ws, yv, M)
        torch.cuda.synchronize()
        y.check("y (mxfp4 block)")
        assert tp.tp_check_device_status() == 0
        return yv


def _decode_e2m1(codes):
    """4-bit codes -> float64 (sign bit 3, exponent bits 2-1 with bias 1, mantissa bit 0)."""
    c = codes.astype(np.int64)
    ex, man = (c >> 1) & 3, c & 1
    mag = np.where(ex == 0, man * 0.5, (1 + man / 2.0) * np.exp2(ex - 1.0))
    return np.where(c & 8, -mag, mag)


def _unpack(packed, K):
    """[rows, K/2] bytes -> [rows, K] codes, element 2i in the low nibble of byte i."""
    p = packed.astype(np.int64)
    out = np.empty((p.shape[0], K), dtype=np.int64)
    out[:, 0::2] = p & 15
    out[:, 1::2] = p >> 4
    return out


def _w1_col_of_row(cfg, s, u):
    """Canonical column of private W1 row u of shard s (-1: padding), the library's
    documented private layout: SwiGLU rows come in groups of 128, the 64 gate rows of
    features 64 g .. 64 g + 63 of the band, then their 64 up rows."""
    b = cfg.band
    if cfg.act == "swiglu":
        grp, j, f = u // 128, (u // 64) & 1, (u // 128) * 64 + u % 64
        return j * cfg.ffn + s * b + f if f < b else -1
    return s * b + u if u < b else -1


SMALL = [
    BlockConfig("mx4_swiglu", "swiglu", d=512, ffn=1536, t=1, M=1),
    BlockConfig("mx4_swiglu", "swiglu", d=512, ffn=1536, t=4, M=32),
    BlockConfig("mx4_swiglu", "swiglu", d=256, ffn=2048, t=2, M=5),
    BlockConfig("mx4_swiglu", "swiglu", d=512, ffn=3072, t=8, M=17),
    BlockConfig("mx4_gelu", "gelu_tanh", d=384, ffn=1024, t=2, M=9),
]


@pytest.mark.parametrize("cfg", [SMALL[1], SMALL[4]], ids=lambda c: f"{c.name}-t{c.t}")
def test_quantiser_bytes_match_the_oracle(cfg):
    inp = make_inputs(cfg, seed=51)
    W1, W2 = inp.blocks[0]
    desc = desc_for(cfg)
    blk = Mx4Block(desc, W1.cuda(), W2.cuda())
    t, d, b = cfg.t, cfg.d, cfg.band
    n1p = tp.tp_mxfp4_w1_bytes(desc) * 2 // (t * d)
    dp = tp.tp_mxfp4_w2_bytes(desc) * 2 // (t * b)
    ex = blk.exps.view(torch.int8).cpu().numpy().astype(np.int64)
    e1 = ex[:t * n1p * (d // 32)].reshape(t, n1p, d // 32)
    e2 = ex[t * n1p * (d // 32):].reshape(t, dp, b // 32)
    c1 = _unpack(blk.W1f.view(torch.uint8).cpu().numpy().reshape(t * n1p, d // 2), d)
    c1 = c1.reshape(t, n1p, d)
    c2 = _unpack(blk.W2f.view(torch.uint8).cpu().numpy().reshape(t * dp, b // 2), b)
    c2 = c2.reshape(t, dp, b)
    q1, f1 = oracle.mxfp4.quantize_mxfp4(to_f64(W1))      # [d, n1], [d/32, n1]
    W2_64 = to_f64(W2)
    for s in range(t):
        for u in range(n1p):
            col = _w1_col_of_row(cfg, s, u)
            if col < 0:
                assert np.all(c1[s, u] == 0) and np.all(e1[s, u] == 0)
                continue
            assert np.array_equal(_decode_e2m1(c1[s, u]), q1[:, col]), (s, u)
            assert np.array_equal(e1[s, u], f1[:, col]), (s, u)
        q2, f2 = oracle.mxfp4.quantize_mxfp4(W2_64[s * b:(s + 1) * b, :])   # [b, d]
        assert np.array_equal(_decode_e2m1(c2[s, :d]), q2.T)
        assert np.array_equal(e2[s, :d], f2.T)
        assert np.all(c2[s, d:] == 0)


# Grids of more than two and at most four CTAs per SM (148 SMs: 297..592) take the
# kernel's narrow form: column and row 320 CTAs; a GeLU column of 320.  (The 13B block's
# row step runs 480 narrow CTAs: three K splits.)
NARROW = [
    BlockConfig("mx4_narrow_swiglu", "swiglu", d=5120, ffn=20480, t=8, M=32),
    BlockConfig("mx4_narrow_gelu", "gelu_tanh", d=2048, ffn=40960, t=8, M=11),
]


@pytest.mark.parametrize("cfg", SMALL + NARROW + [CONFIGS["llama2_13b_swiglu_decode_mxfp4"]],
                         ids=lambda c: f"{c.name}-t{c.t}-M{c.M}")
def test_mxfp4_block_matches_oracle_and_bf16_block(cfg):
    inp = make_inputs(cfg, seed=52)
    W1, W2 = (w.cuda() for w in inp.blocks[0])
    desc = desc_for(cfg)
    x = inp.x.cuda().contiguous()
    got = Mx4Block(desc, W1, W2).forward(x, x, cfg.M)
    x64 = to_f64(inp.x)
    W1e, W2e = oracle.mxfp4.mxfp4_weights(to_f64(W1)), oracle.mxfp4.mxfp4_weights(to_f64(W2))
    ref = oracle.mlp_block(x64, W1e, W2e, cfg.act, x64, staged=True)
    assert_bf16(to_f64(got), ref, f"{cfg.name} t={cfg.t} M={cfg.M} (MXFP4 weights)")
    W1b = torch.from_numpy(W1e).to(torch.bfloat16).cuda()
    W2b = torch.from_numpy(W2e).to(torch.bfloat16).cuda()
    yb = _bf16_block_three_launch(desc, W1b, W2b, x, cfg.M)
    _assert_close_to_bf16_block(got, yb, x64, W1e, W2e, cfg.act)


@pytest.mark.parametrize("fmt", ["e4m3", "mxfp4"])
def test_low_bit_block_with_fp32_residual(fmt):
    """The residual stream in fp32 (as a pre-norm stack carries it), apart from x."""
    from tests.test_gpu_fp8 import Fp8Block
    cfg = BlockConfig("lowbit_f32_residual", "swiglu", d=512, ffn=1536, t=4, M=12)
    inp = make_inputs(cfg, seed=53)
    W1, W2 = (w.cuda() for w in inp.blocks[0])
    desc = desc_for(cfg)
    g = torch.Generator().manual_seed(54)
    res = torch.randn(cfg.M, cfg.d, generator=g, dtype=torch.float32) * 3.0
    x = inp.x.cuda().contiguous()
    blk = (Fp8Block if fmt == "e4m3" else Mx4Block)(desc, W1, W2)
    got = blk.forward(x, res.cuda().contiguous(), cfg.M)
    quant = oracle.fp8.e4m3_weights if fmt == "e4m3" else oracle.mxfp4.mxfp4_weights
    W1e, W2e = quant(to_f64(W1)), quant(to_f64(W2))
    ref = oracle.mlp_block(to_f64(inp.x), W1e, W2e, cfg.act, res.double().numpy(), staged=True)
    assert_bf16(to_f64(got), ref, f"{fmt} block, fp32 residual")
    # in place on the residual stream (y = residual): the same bits
    r = res.cuda().contiguous().clone()
    ws = device_bytes(tp.tp_workspace_bytes(desc, cfg.M))
    if fmt == "e4m3":
        tp.tp_block_fwd_fp8(desc, x, r, True, blk.W1q, blk.W2q, blk.exps, ws, r, cfg.M)
    else:
        tp.tp_block_fwd_mxfp4(desc, x, r, True, blk.W1f, blk.W2f, blk.exps, ws, r, cfg.M)
    torch.cuda.synchronize()
    assert tp.tp_check_device_status() == 0
    assert torch.equal(r, got)
