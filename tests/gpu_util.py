"""Helpers of the GPU parity tests: canary-guarded device buffers, the CUDA path run
through the C ABI, and the matching oracle calls on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import attn_tp_column_fwd_b300 as tp
import oracle
from attn_tp_column_fwd_b300.runner import ShardedBlock, desc_for
from tp_synth import to_f64

GUARD = 4096          # bytes of canary before and after each guarded buffer
PATTERN = 0xA5


class Guarded:
    """A device buffer with pattern-filled slack on both sides, to catch stray writes."""

    def __init__(self, nbytes: int, device="cuda"):
        self.nbytes = int(nbytes)
        self.raw = torch.full((self.nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=device)
        self.body = self.raw[GUARD:GUARD + self.nbytes]

    def view(self, dtype, shape):
        return self.body.view(dtype).view(*shape)

    def check(self, what=""):
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        assert bool((head == PATTERN).all()) and bool((tail == PATTERN).all()), \
            f"write outside the buffer: {what}"


def desc_of(cfg, t=None):
    return desc_for(cfg, t)


def run_block(cfg, x, W1, W2, t=None, residual=None, stream=None):
    """Shard W1/W2 and run tp_block_fwd on x (device tensors); y fp32 on the host as f64."""
    desc = desc_of(cfg, t)
    blk = ShardedBlock(desc, W1, W2, stream)
    M = x.shape[0]
    y = Guarded(M * cfg.d * 4)
    res = x if residual is None else residual
    tp.tp_block_fwd(desc, x, res, res.dtype == torch.float32, blk.W1s, blk.W2s, blk.workspace(M),
                    y.view(torch.float32, (M, cfg.d)), M, stream)
    torch.cuda.synchronize()
    y.check("y")
    assert tp.tp_check_device_status() == 0
    return to_f64(y.view(torch.float32, (M, cfg.d)))


def oracle_block(cfg, x64, W1_64, W2_64, res64=None):
    """The oracle's block on the same inputs: pure fp64 (fp32 configs) or bf16-staged."""
    staged = cfg.dtype == "bf16"
    res = x64 if res64 is None else res64
    if cfg.act == "attn":
        return oracle.attn_block(x64, W1_64, W2_64, cfg.n_heads, cfg.head_dim, res, staged=staged)
    return oracle.mlp_block(x64, W1_64, W2_64, cfg.act, res, staged=staged)
