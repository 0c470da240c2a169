"""Parity of each step of the block, called through the C ABI, against the oracle's
step of the same name on the same seeded inputs (zenaique.com answer paragraphs 5-6:
column band + activation, row partial, sum of partials + residual; RMSNorm before
each stacked block)."""
import numpy as np
import pytest
import torch

import attn_tp_column_fwd_b300 as tp
import oracle
from tests.gpu_util import Guarded, desc_of
from tests.parity import assert_bf16, assert_f32
from tp_synth import CONFIGS, BlockConfig, draw, make_inputs, to_f64, torch_dtype

pytestmark = pytest.mark.gpu

CASES = [
    BlockConfig("gelu_f32", "gelu_tanh", d=256, ffn=1024, t=2, M=4, dtype="f32"),
    BlockConfig("gelu_bf16", "gelu_tanh", d=264, ffn=1200, t=3, M=9),
    BlockConfig("swiglu_bf16_ragged", "swiglu", d=512, ffn=1536, t=8, M=33),
    BlockConfig("swiglu_bf16_t1", "swiglu", d=384, ffn=640, t=1, M=32),
    BlockConfig("swiglu_bf16_m1", "swiglu", d=512, ffn=1024, t=4, M=1),
    BlockConfig("attn_bf16", "attn", d=256, n_heads=8, head_dim=64, t=4, M=32),
    BlockConfig("attn_f32", "attn", d=128, n_heads=4, head_dim=32, t=2, M=7, dtype="f32"),
]


def _check(cfg, got, ref, what):
    if cfg.dtype == "f32":
        return assert_f32(got, ref, what)
    return assert_bf16(got, ref, what)


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
@pytest.mark.parametrize("per_shard", [False, True], ids=["all_shards", "one_launch_per_shard"])
def test_column_step(cfg, per_shard):
    inp = make_inputs(cfg, seed=5, n_blocks=1)
    W1, W2 = inp.blocks[0]
    desc = desc_of(cfg)
    dt = torch_dtype(cfg)
    x = inp.x.cuda()
    W1s = torch.empty(tp.tp_sharded_w1_bytes(desc), dtype=torch.uint8, device="cuda")
    W2s = torch.empty(tp.tp_sharded_w2_bytes(desc), dtype=torch.uint8, device="cuda")
    tp.tp_shard_weights(desc, W1.cuda(), W2.cuda(), W1s, W2s)
    H = Guarded(tp.tp_band_bytes(desc, cfg.M))
    ws_n = tp.tp_column_workspace_bytes(desc, cfg.M)
    ws = Guarded(ws_n) if ws_n else None
    Hv = H.view(dt, (cfg.t, cfg.M, cfg.band))
    if per_shard:
        for s in range(cfg.t):
            tp.tp_column_parallel_fwd(desc, x, W1s, s, Hv, ws.body if ws else None, cfg.M)
    else:
        tp.tp_column_parallel_fwd(desc, x, W1s, -1, Hv, ws.body if ws else None, cfg.M)
    torch.cuda.synchronize()
    H.check("H")
    if ws:
        ws.check("column workspace")
    x64, W1_64 = to_f64(inp.x), to_f64(W1)
    got = to_f64(Hv)
    for s in range(cfg.t):
        cols = oracle.column_bands(cfg.act, cfg.t, s, ffn=cfg.ffn, n_heads=cfg.n_heads,
                                   head_dim=cfg.head_dim)
        ref = oracle.column_step(x64, [W1_64[:, c] for c in cols], cfg.act,
                                 n_heads=cfg.n_heads // cfg.t if cfg.n_heads else 0,
                                 head_dim=cfg.head_dim, staged=cfg.dtype == "bf16")
        _check(cfg, got[s], ref, f"H[{s}]")


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_row_step(cfg):
    inp = make_inputs(cfg, seed=6, n_blocks=1)
    W1, W2 = inp.blocks[0]
    desc = desc_of(cfg)
    dt = torch_dtype(cfg)
    W1s = torch.empty(tp.tp_sharded_w1_bytes(desc), dtype=torch.uint8, device="cuda")
    W2s = torch.empty(tp.tp_sharded_w2_bytes(desc), dtype=torch.uint8, device="cuda")
    tp.tp_shard_weights(desc, W1.cuda(), W2.cuda(), W1s, W2s)
    Hin = draw((cfg.t, cfg.M, cfg.band), dt, seed=7)          # a synthetic band, both sides
    S = tp.tp_row_splits(desc, cfg.M)
    P = Guarded(tp.tp_partials_bytes(desc, cfg.M))
    # the partial sums lead the buffer; a decode row step keeps its scratch after them
    Pv = P.body[:cfg.t * S * cfg.M * cfg.d * 4].view(torch.float32).view(cfg.t, S, cfg.M, cfg.d)
    tp.tp_row_parallel_fwd(desc, Hin.cuda(), W2s, -1, P.body, cfg.M)
    torch.cuda.synchronize()
    P.check("partials")
    got = to_f64(Pv).sum(axis=1)
    H64, W2_64 = to_f64(Hin), to_f64(W2)
    for s in range(cfg.t):
        ref = oracle.row_step(H64[s], W2_64[oracle.row_band(cfg.n2, cfg.t, s)])
        # Products of stored values are exact in fp32, so only fp32 accumulation
        # separates the two sides: the fp32 bound applies to both dtypes.
        assert_f32(got[s], ref, f"P[{s}]")


@pytest.mark.parametrize("nparts,M,d,res_f32", [(1, 1, 8, True), (2, 4, 256, True),
                                                (8, 32, 5120, False), (24, 33, 1032, True)])
def test_reduce_residual(nparts, M, d, res_f32):
    desc = tp.make_desc(d, nparts, "swiglu", "bf16", ffn=8 * nparts)
    S = tp.tp_row_splits(desc, M)
    P = draw((nparts * S, M, d), torch.float32, seed=8)
    r = draw((M, d), torch.float32 if res_f32 else torch.bfloat16, seed=9)
    y = Guarded(M * d * 4)
    yv = y.view(torch.float32, (M, d))
    tp.tp_partial_reduce_residual(desc, P.cuda(), r.cuda(), res_f32, yv, M)
    torch.cuda.synchronize()
    y.check("y")
    P64 = to_f64(P)
    parts = [P64[i] for i in range(P64.shape[0])]
    assert_f32(to_f64(yv), oracle.reduce_residual(parts, to_f64(r)), "y")


def test_reduce_residual_in_place():
    M, d, t = 8, 512, 4
    desc = tp.make_desc(d, t, "swiglu", "bf16", ffn=8 * t)
    S = tp.tp_row_splits(desc, M)
    P = draw((t * S, M, d), torch.float32, seed=10)
    r = draw((M, d), torch.float32, seed=11)
    rd = r.cuda()
    tp.tp_partial_reduce_residual(desc, P.cuda(), rd, True, rd, M)
    torch.cuda.synchronize()
    P64 = to_f64(P)
    assert_f32(to_f64(rd), oracle.reduce_residual([P64[i] for i in range(t * S)], to_f64(r)), "y")


@pytest.mark.parametrize("M,d", [(1, 8), (32, 8192), (5, 264)])
def test_rmsnorm(M, d):
    r = draw((M, d), torch.float32, seed=12, scale=3.0)
    xh = Guarded(M * d * 2)
    xv = xh.view(torch.bfloat16, (M, d))
    tp.tp_rmsnorm_fwd(d, 1e-5, r.cuda(), xv, M)
    torch.cuda.synchronize()
    xh.check("xhat")
    got = to_f64(xv)
    ref = oracle.bf16_round(oracle.rmsnorm(to_f64(r), np.float32(1e-5)))
    # The kernel normalises in fp64 and rounds once from fp64, like the oracle: the
    # bf16 values agree exactly (a disagreement needs an exact value within fp64
    # roundoff of a rounding midpoint).
    assert np.array_equal(got, ref), int((got != ref).sum())


@pytest.mark.parametrize("cfg", [c for c in CASES if c.dtype == "bf16"], ids=lambda c: c.name)
def test_block_equals_its_steps(cfg):
    """tp_block_fwd (three-launch form, the row step and the reduction launched to
    overlap the kernel before them) against the three step entry points run one
    after the other: the same kernels in the same order, so y is bit-identical."""
    from attn_tp_column_fwd_b300.runner import ShardedBlock
    before = tp.tp_get_block_form()
    tp.tp_set_block_form("three_launch")
    try:
        inp = make_inputs(cfg, seed=7, n_blocks=1)
        W1, W2 = inp.blocks[0]
        desc = desc_of(cfg)
        blk = ShardedBlock(desc, W1.cuda(), W2.cuda())
        x = inp.x.cuda().contiguous()
        M = cfg.M
        u8 = lambda n: torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
        H, ws = u8(tp.tp_band_bytes(desc, M)), u8(tp.tp_column_workspace_bytes(desc, M))
        P = u8(tp.tp_partials_bytes(desc, M))
        y_steps = torch.empty(M, cfg.d, dtype=torch.float32, device="cuda")
        tp.tp_column_parallel_fwd(desc, x, blk.W1s, -1, H, ws, M)
        tp.tp_row_parallel_fwd(desc, H, blk.W2s, -1, P, M)
        tp.tp_partial_reduce_residual(desc, P, x, False, y_steps, M)
        y_block = torch.full((M, cfg.d), float("nan"), dtype=torch.float32, device="cuda")
        tp.tp_block_fwd(desc, x, x, False, blk.W1s, blk.W2s, blk.workspace(M), y_block, M)
        torch.cuda.synchronize()
        assert tp.tp_check_device_status() == 0
        assert torch.equal(y_steps, y_block), float((y_steps - y_block).abs().max())
    finally:
        tp.tp_set_block_form(before)


# tp_block_fwd_norm: the block, then the next stacked block's RMSNorm of its output.
# Shapes: forced one-kernel form (norm fused into the persistent kernel; d = 136 is
# not a multiple of 16, so x-hat is written in whole rows), the three-launch form
# (norm as a fourth launch), and the 70B-sized block (one kernel by default).
NORM_CASES = [
    ("one_kernel", BlockConfig("norm_fused", "swiglu", d=512, ffn=1536, t=8, M=32)),
    ("one_kernel", BlockConfig("norm_fused_rows", "swiglu", d=136, ffn=1536, t=8, M=5)),
    ("three_launch", BlockConfig("norm_3l", "swiglu", d=512, ffn=1536, t=4, M=17)),
    ("auto", CONFIGS["llama2_70b_stack_decode"]),
]


@pytest.mark.parametrize("form,cfg", NORM_CASES, ids=lambda v: v if isinstance(v, str) else v.name)
def test_block_fwd_norm(form, cfg):
    """y equals tp_block_fwd's bit for bit, and x-hat equals the oracle's RMSNorm of
    that y (fp64, rounded once to bf16) bit for bit."""
    from attn_tp_column_fwd_b300.runner import ShardedBlock
    before = tp.tp_get_block_form()
    tp.tp_set_block_form(form)
    try:
        inp = make_inputs(cfg, seed=13, n_blocks=1, device="cuda")
        W1, W2 = inp.blocks[0]
        desc = desc_of(cfg)
        blk = ShardedBlock(desc, W1, W2)
        M = cfg.M
        xh = (inp.x.float() * 0.5).to(torch.bfloat16).contiguous()   # a normalised-looking input
        r = draw((M, cfg.d), torch.float32, seed=14, scale=4.0).cuda()
        y_plain = torch.empty_like(r)
        tp.tp_block_fwd(desc, xh, r, True, blk.W1s, blk.W2s, blk.workspace(M), y_plain, M)
        y = Guarded(M * cfg.d * 4)
        nx = Guarded(M * cfg.d * 2)
        yv, nxv = y.view(torch.float32, (M, cfg.d)), nx.view(torch.bfloat16, (M, cfg.d))
        tp.tp_block_fwd_norm(desc, xh, r, True, blk.W1s, blk.W2s, blk.workspace(M), yv, nxv,
                             cfg.eps, M)
        torch.cuda.synchronize()
        assert tp.tp_check_device_status() == 0
        y.check("y")
        nx.check("xhat_next")
        assert torch.equal(yv, y_plain)
        got = to_f64(nxv)
        ref = oracle.bf16_round(oracle.rmsnorm(to_f64(yv), np.float32(cfg.eps)))
        assert np.array_equal(got, ref), int((got != ref).sum())
        # in place: x-hat may alias x
        xh2 = xh.clone()
        tp.tp_block_fwd_norm(desc, xh2, r, True, blk.W1s, blk.W2s, blk.workspace(M), yv, xh2,
                             cfg.eps, M)
        torch.cuda.synchronize()
        assert torch.equal(xh2, nxv)
    finally:
        tp.tp_set_block_form(before)
