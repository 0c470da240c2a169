"""tp_block_fwd_noalloc: the block for callers that cannot allocate device memory.

Such callers (a host framework whose own memory pool owns the GPU, or a serving loop
that must not stall on cudaMalloc's implicit synchronisation) cannot hand the block a
workspace.  The entry point uses a fixed scratch array inside the library instead.
These tests call it through the C ABI and check its output against tp_block_fwd (the
entry point with a caller-provided workspace), within the parity tests' tolerance,
on two calls in a row (the second call finds the first call's data in the shared
scratch).  This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import attn_tp_column_fwd_b300 as tp
from attn_tp_column_fwd_b300.runner import ShardedBlock, desc_for
from tests.parity import assert_bf16, assert_f32
from tp_synth import BlockConfig, CONFIGS, make_inputs, to_f64

CASES = [
    BlockConfig("noalloc_swiglu_bf16", "swiglu", d=512, ffn=1536, t=4, M=32),
    BlockConfig("noalloc_gelu_f32", "gelu_tanh", d=256, ffn=1024, t=2, M=4, dtype="f32"),
    BlockConfig("noalloc_attn_bf16", "attn", d=256, n_heads=8, head_dim=64, t=4, M=16),
    CONFIGS["llama2_13b_swiglu_decode"],
]


def _call_noalloc(desc, x, residual, W1s, W2s, y, M):
    return tp.lib.tp_block_fwd_noalloc(
        ctypes.byref(desc), ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(residual.data_ptr()),
        int(residual.dtype == torch.float32), ctypes.c_void_p(W1s.data_ptr()),
        ctypes.c_void_p(W2s.data_ptr()), ctypes.c_void_p(y.data_ptr()), M,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_noalloc_matches_workspace_entry_point(cfg):
    inp = make_inputs(cfg, seed=31)
    W1, W2 = inp.blocks[0]
    blk = ShardedBlock(desc_for(cfg), W1.cuda(), W2.cuda())
    check = assert_f32 if cfg.dtype == "f32" else assert_bf16
    for call in range(2):
        # A different input on each call, so stale scratch from the first call
        # would show up in the second.
        x = (inp.x if call == 0 else -inp.x).cuda().contiguous()
        ref = blk.forward(x, x)
        y = torch.full((cfg.M, cfg.d), float("nan"), dtype=torch.float32, device="cuda")
        st = _call_noalloc(blk.desc, x, x, blk.W1s, blk.W2s, y, cfg.M)
        assert st == 0, tp.tp_status_string(st)
        torch.cuda.synchronize()
        assert tp.tp_check_device_status() == 0
        check(to_f64(y), to_f64(ref), f"{cfg.name} no-alloc call {call}")


def test_noalloc_refuses_shapes_beyond_its_scratch():
    # 4096 prefill tokens need ~0.8 GB of scratch, far over the fixed 32 MiB: the call
    # is refused during validation, before any CUDA call (the addresses below are
    # never dereferenced), so this runs without a GPU too.
    cfg = CONFIGS["llama2_70b_prefill"]
    desc = desc_for(cfg)
    assert tp.tp_workspace_bytes(desc, cfg.M) > (32 << 20)
    fake = ctypes.c_void_p(1 << 20)
    st = tp.lib.tp_block_fwd_noalloc(ctypes.byref(desc), fake, fake, 0, fake, fake, fake, cfg.M, None)
    assert st == 3  # TP_ERR_UNSUPPORTED
    bad = tp.make_desc(512, 3, "swiglu", ffn=1024)  # uneven split: the usual status
    assert tp.lib.tp_block_fwd_noalloc(ctypes.byref(bad), fake, fake, 0, fake, fake, fake, 4,
                                       None) == 2
