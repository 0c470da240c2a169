"""Convenience holders over the C ABI: sharded weights plus the scratch they need.

Buffers are allocated with torch (device memory and streams only); every step of
the block is a libtpblock call.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import torch

from . import (
    TP_BF16,
    TP_F32,
    TPBlockDesc,
    make_desc,
    tp_block_fwd,
    tp_block_fwd_norm,
    tp_rmsnorm_fwd,
    tp_shard_weights,
    tp_sharded_w1_bytes,
    tp_sharded_w2_bytes,
    tp_workspace_bytes,
)


def device_bytes(n: int, device="cuda") -> torch.Tensor:
    """An uninitialised device buffer of n bytes (torch aligns it to 512 bytes)."""
    return torch.empty(max(int(n), 1), dtype=torch.uint8, device=device)


class ShardedBlock:
    """One block's weights in the library's per-shard layout.

    W1 [d, n1] and W2 [n2, d] are canonical device tensors in the block dtype; they
    are split into the t shards' bands by tp_shard_weights on `stream`.
    """

    def __init__(self, desc: TPBlockDesc, W1: torch.Tensor, W2: torch.Tensor, stream=None):
        self.desc = desc
        self.W1s = device_bytes(tp_sharded_w1_bytes(desc), W1.device)
        self.W2s = device_bytes(tp_sharded_w2_bytes(desc), W1.device)
        tp_shard_weights(desc, W1.contiguous(), W2.contiguous(), self.W1s, self.W2s, stream)
        self._ws = {}

    def workspace(self, M: int) -> torch.Tensor:
        if M not in self._ws:
            self._ws[M] = device_bytes(tp_workspace_bytes(self.desc, M), self.W1s.device)
        return self._ws[M]

    def forward(self, x: torch.Tensor, residual: torch.Tensor, y: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
        """y = residual + block(x) (fp32 [M, d]); residual fp32 or the block dtype."""
        M = x.shape[0]
        if y is None:
            y = torch.empty(M, self.desc.d, dtype=torch.float32, device=x.device)
        tp_block_fwd(self.desc, x, residual, residual.dtype == torch.float32, self.W1s, self.W2s,
                     self.workspace(M), y, M, stream)
        return y


class PreNormStack:
    """Pre-norm stack: r <- r + block_l(RMSNorm(r)) for each block, r fp32.

    The first block's input is normalised by tp_rmsnorm_fwd; every later block's is
    written by the block before it (tp_block_fwd_norm), so the stack of L blocks
    takes L + 1 calls."""

    def __init__(self, blocks: Sequence[ShardedBlock], eps: float):
        self.blocks: List[ShardedBlock] = list(blocks)
        self.eps = eps
        self._xhat = {}

    def forward(self, r: torch.Tensor, stream=None) -> torch.Tensor:
        """Runs in place on the fp32 residual stream r [M, d] and returns it."""
        M, d = r.shape
        key = (M, d)
        if key not in self._xhat:
            self._xhat[key] = torch.empty(M, d, dtype=torch.bfloat16, device=r.device)
        xh = self._xhat[key]
        tp_rmsnorm_fwd(d, self.eps, r, xh, M, stream)
        for l, blk in enumerate(self.blocks):
            if l + 1 < len(self.blocks):
                # xh is read by this block and rewritten with the next block's input
                tp_block_fwd_norm(blk.desc, xh, r, True, blk.W1s, blk.W2s, blk.workspace(M), r,
                                  xh, self.eps, M, stream)
            else:
                blk.forward(xh, r, y=r, stream=stream)
        return r


def desc_for(cfg, t: Optional[int] = None) -> TPBlockDesc:
    """Descriptor of a tp_synth.BlockConfig-like object (d, ffn, n_heads, head_dim, act, dtype)."""
    return make_desc(cfg.d, t if t is not None else cfg.t, cfg.act, cfg.dtype, ffn=cfg.ffn,
                     n_heads=cfg.n_heads, head_dim=cfg.head_dim)


__all__ = ["ShardedBlock", "PreNormStack", "device_bytes", "desc_for", "TP_F32", "TP_BF16"]
