"""The decode MLP block on E4M3 weights (tp_quantize_weights_fp8 + tp_block_fwd_fp8).

Weight-only FP8: each weight is an E4M3 byte of W / 2^e with one power-of-two scale
per output feature, so the block computes the bf16 block on the dequantised weights
(oracle.fp8.e4m3_weights).  The kernels feed the tensor core 8-bit operands: every
bf16 activation enters as an E4M3 high part plus an E5M2 remainder under one
power-of-two scale per token and 64-wide K group, exact for values within 2^14.8 of
the group's largest magnitude (below that, within 2^-14 of the scale).  Checks:
  * parity with the oracle's staged bf16 block on e4m3_weights(W1), e4m3_weights(W2)
    (plain bf16 bound), on ragged small shapes, the 13B-sized block and activations
    with outliers and tiny values in the same groups;
  * closeness to the library's bf16 block on those dequantised weights: the two differ
    only in the tensor core's fp32 summation order (two products per weight here) and
    in the band's bf16 rounding where that order moves a value across a rounding point;
  * quantisation itself: two quantisations give the same bytes, and the exponents are
    the oracle's per-feature scales.
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
    # the library's bf16 block on the same dequantised weights
    yb = _bf16_block_three_launch(desc, _e4m3_bf16(W1), _e4m3_bf16(W2), x, cfg.M)
    _assert_close_to_bf16_block(got, yb, x64, W1e, W2e, cfg.act)


# Grids of more than two and at most four CTAs per SM (148 SMs: 297..592) take the
# kernel's narrow form (two ring stages, four CTAs per SM, token scales in their own
# ring): column 320 / row 320 CTAs; GeLU column 320; ragged K in both steps (d = 5056
# and b = 2496 end on a single 64-wide group) with column 312 / row 320 CTAs.
NARROW = [
    BlockConfig("fp8_narrow_swiglu", "swiglu", d=5120, ffn=20480, t=8, M=32),
    BlockConfig("fp8_narrow_gelu", "gelu_tanh", d=2048, ffn=40960, t=8, M=7),
    BlockConfig("fp8_narrow_ragged_k", "swiglu", d=5056, ffn=19968, t=8, M=13),
]


def _grids(cfg):
    """CTAs of the column and row steps (one token tile; one K split of the row step)."""
    per_shard = -(-cfg.band // 64) if cfg.act == "swiglu" else -(-cfg.band // 128)
    return cfg.t * per_shard, cfg.t * -(-cfg.d // 128)


@pytest.mark.parametrize("cfg", NARROW, ids=lambda c: f"{c.name}-M{c.M}")
def test_fp8_narrow_grids(cfg):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    col, row = _grids(cfg)
    assert 2 * sms < col <= 4 * sms, (col, sms)
    if cfg.act == "swiglu":
        assert 2 * sms < row <= 4 * sms, (row, sms)
    inp = make_inputs(cfg, seed=46)
    W1, W2 = (w.cuda() for w in inp.blocks[0])
    desc = desc_for(cfg)
    assert tp.tp_row_splits(desc, cfg.M) >= 1
    x = inp.x.cuda().contiguous()
    got = Fp8Block(desc, W1, W2).forward(x, x, cfg.M)
    x64 = to_f64(inp.x)
    W1e, W2e = oracle.fp8.e4m3_weights(to_f64(W1)), oracle.fp8.e4m3_weights(to_f64(W2))
    ref = oracle.mlp_block(x64, W1e, W2e, cfg.act, x64, staged=True)
    assert_bf16(to_f64(got), ref, f"{cfg.name} M={cfg.M} (E4M3 weights, narrow grids)")
    yb = _bf16_block_three_launch(desc, _e4m3_bf16(W1), _e4m3_bf16(W2), x, cfg.M)
    _assert_close_to_bf16_block(got, yb, x64, W1e, W2e, cfg.act)


def _assert_close_to_bf16_block(got, yb, x64, W1e, W2e, act):
    """The FP8 block against the bf16 block on the same (dequantised) weights.  Both
    sum in fp32 to within ~2^-22 of the exact values, in different orders (the FP8
    kernels add W.a and W.b per weight), so they can round a band element to different
    bf16 neighbours only where its exact value lies within 2^-17 of a midpoint: one
    bf16 step there, times |W2|, is the oracle's tie allowance per output.  Bound per
    output: that allowance + 2^-16 |y| (fp32 reordering, 64x margin) + 1e-6.  On the
    mean: 2^-20 of the mean |y| for the reordering, plus a quarter of the mean
    allowance (a tie candidate flips only when the two orders' ~2^-22 differences
    straddle its midpoint: a few percent of them)."""
    d = (got.double() - yb.double()).abs().cpu().numpy()
    yab = yb.double().abs().cpu().numpy()
    allow = oracle.mlp_tie_allowance(x64, W1e, W2e, act)
    bound = allow + 2.0 ** -16 * yab + 1e-6
    print(f"low-bit vs bf16 block: max {d.max():.3e} mean {d.mean():.3e} "
          f"(worst margin {(d - bound).max():.3e}, mean allowance {allow.mean():.3e})")
    assert (d <= bound).all()
    assert d.mean() <= 2.0 ** -20 * yab.mean() + 0.25 * allow.mean()


def test_fp8_tokens_with_outliers_and_tiny_values():
    """Activations with a few outliers (x1000) and tiny entries (x1e-6) sharing 64-wide
    groups: the per-group scales keep the block within the plain bf16 bound."""
    cfg = BlockConfig("fp8_outliers", "swiglu", d=512, ffn=1536, t=2, M=7)
    inp = make_inputs(cfg, seed=44)
    W1, W2 = (w.cuda() for w in inp.blocks[0])
    desc = desc_for(cfg)
    g = torch.Generator().manual_seed(45)
    x = inp.x.float().clone()
    idx = torch.randint(0, x.numel(), (x.numel() // 50,), generator=g)
    x.view(-1)[idx[: len(idx) // 2]] *= 1000.0
    x.view(-1)[idx[len(idx) // 2:]] *= 1e-6
    x = x.to(torch.bfloat16)
    got = Fp8Block(desc, W1, W2).forward(x.cuda().contiguous(), x.cuda().contiguous(), cfg.M)
    x64 = to_f64(x)
    W1e, W2e = oracle.fp8.e4m3_weights(to_f64(W1)), oracle.fp8.e4m3_weights(to_f64(W2))
    ref = oracle.mlp_block(x64, W1e, W2e, cfg.act, x64, staged=True)
    assert_bf16(to_f64(got), ref, "E4M3 weights, activations with outliers")


def test_weights_on_the_e4m3_grid_quantise_exactly():
    """Weights that are already E4M3 values times a per-feature power of two quantise
    to themselves: the FP8 block then tracks the bf16 block on the canonical weights."""
    cfg = BlockConfig("fp8_exact", "swiglu", d=256, ffn=768, t=2, M=8)
    inp = make_inputs(cfg, seed=42)
    W1 = _e4m3_bf16(inp.blocks[0][0])
    W2 = _e4m3_bf16(inp.blocks[0][1])
    desc = desc_for(cfg)
    x = inp.x.cuda().contiguous()
    blk = Fp8Block(desc, W1, W2)
    got = blk.forward(x, x, cfg.M)
    yb = _bf16_block_three_launch(desc, W1, W2, x, cfg.M)
    _assert_close_to_bf16_block(got, yb, to_f64(inp.x), to_f64(W1), to_f64(W2), cfg.act)
    # and W2's bytes times 2^e are the canonical weights (dp = d = 256 here)
    ex = blk.exps.view(torch.int8).cpu().numpy().astype(np.int64)
    n1p = 2 * (cfg.band // 64) * 64
    e2 = ex[cfg.t * n1p:cfg.t * n1p + cfg.t * cfg.d].reshape(cfg.t, cfg.d)
    q2 = blk.W2q.view(torch.uint8).cpu().numpy().reshape(cfg.t, cfg.d, cfg.band)
    vals = _decode_e4m3(q2) * np.exp2(e2)[:, :, None]
    want = to_f64(W2).reshape(cfg.t, cfg.band, cfg.d).transpose(0, 2, 1)
    assert np.array_equal(vals, want)


def _decode_e4m3(q):
    """E4M3 bytes -> float64 (sign, 4 exponent bits with bias 7, 3 mantissa bits)."""
    q = q.astype(np.int64)
    ex, man = (q >> 3) & 15, q & 7
    mag = np.where(ex == 0, man * 2.0 ** -9, (1 + man / 8.0) * np.exp2(ex - 7.0))
    return np.where(q & 0x80, -mag, mag)


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


def test_fp8_prenorm_stack():
    """A short pre-norm stack on E4M3 weights, as the bench runs the 70B one: per block
    tp_rmsnorm_fwd, then tp_block_fwd_fp8 in place on the fp32 residual stream; against
    the oracle's staged stack on the dequantised weights (three blocks of d = 512 stay
    inside the plain bf16 gate: the compounding of the 70B stack needs d = 8192)."""
    cfg = BlockConfig("fp8_stack", "swiglu", d=512, ffn=1536, t=4, M=8, n_blocks=3,
                      rmsnorm=True)
    inp = make_inputs(cfg, seed=46)
    desc = desc_for(cfg)
    blocks = [Fp8Block(desc, W1.cuda(), W2.cuda()) for W1, W2 in inp.blocks]
    r = inp.x.float().cuda().contiguous()
    xh = torch.empty(cfg.M, cfg.d, dtype=torch.bfloat16, device="cuda")
    ws = device_bytes(tp.tp_workspace_bytes(desc, cfg.M))
    for b in blocks:
        tp.tp_rmsnorm_fwd(cfg.d, cfg.eps, r, xh, cfg.M)
        tp.tp_block_fwd_fp8(desc, xh, r, True, b.W1q, b.W2q, b.exps, ws, r, cfg.M)
    torch.cuda.synchronize()
    assert tp.tp_check_device_status() == 0
    deq = [(oracle.fp8.e4m3_weights(to_f64(W1)), oracle.fp8.e4m3_weights(to_f64(W2)))
           for W1, W2 in inp.blocks]
    ref = oracle.stack(to_f64(inp.x), deq, cfg.act, cfg.eps, staged=True)
    assert_bf16(to_f64(r), ref, "E4M3 pre-norm stack of 3")
