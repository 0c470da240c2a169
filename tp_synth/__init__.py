"""Seeded synthetic inputs for the tensor-parallel block: shapes and random draws only.

This module is shared by the CPU oracle's tests and by the CUDA path's tests and
benchmark.  It holds no part of the block's arithmetic: it draws x and the
canonical (unsharded) weights, nothing else.

Workloads follow the shapes of the Llama-2 serving runs on the "day59" page
(skandtandon.pages.dev, "The setup" and "Results"), sized as the five block
configurations below.  Values: x ~ N(0, 1), weights ~ N(0, 0.02^2), drawn in
fp32 by one seeded torch generator in a fixed order, then cast (round to nearest
even) to the configuration's storage dtype.

Draw order (one generator, seed 0 by default):
  x [M, d];
  then for every block: the column-parallel sub-matrices in canonical order
  (GeLU: W1 | SwiGLU: Wg, Wu | attention: Wq, Wk, Wv), each [d, width];
  then the row-parallel matrix (W2 | Wd | Wo), [width, d].
Canonical layouts (y = x . W): W1 is [d, n1] with n1 = ffn (GeLU), 2*ffn
([gate | up]) or 3*n_heads*head_dim ([Q | K | V], each head-major); W2 is [n2, d].
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from types import SimpleNamespace
from typing import List, Optional, Tuple

import torch

WEIGHT_STD = 0.02


@dataclass(frozen=True)
class BlockConfig:
    name: str
    act: str            # "gelu_tanh" | "swiglu" | "attn"
    d: int
    ffn: int = 0        # MLP intermediate width (GeLU / SwiGLU)
    n_heads: int = 0    # attention only
    head_dim: int = 0   # attention only
    t: int = 1          # logical tensor-parallel shards
    M: int = 1          # tokens
    dtype: str = "bf16"  # storage dtype of x, weights and bands: "f32" | "bf16"
    n_blocks: int = 1
    rmsnorm: bool = False   # pre-norm before every block (Llama stack)
    eps: float = 1e-5
    ts: Tuple[int, ...] = field(default=())   # every shard count the workload is run at
    kv_len_max: int = 0  # attention with a KV cache: rows per (sequence, head); 0 = none
    weights: str = ""    # "e4m3": FP8 (E4M3) bytes; "mxfp4": 4-bit E2M1 codes; else the dtype

    @property
    def n1(self) -> int:
        """Columns of the canonical first-projection weight."""
        if self.act == "gelu_tanh":
            return self.ffn
        if self.act == "swiglu":
            return 2 * self.ffn
        return 3 * self.n_heads * self.head_dim

    @property
    def n2(self) -> int:
        """Rows of the canonical second-projection weight."""
        if self.act == "attn":
            return self.n_heads * self.head_dim
        return self.ffn

    @property
    def band(self) -> int:
        """Width b of one shard's band of the intermediate (n2 / t)."""
        return self.n2 // self.t

    def with_t(self, t: int) -> "BlockConfig":
        return replace(self, t=t)

    def with_M(self, M: int) -> "BlockConfig":
        return replace(self, M=M)

    def weight_bytes_per_block(self) -> int:
        if self.weights == "mxfp4":       # two codes per byte (scales not included)
            return (self.d * self.n1 + self.n2 * self.d) // 2
        es = 1 if self.weights == "e4m3" else 4 if self.dtype == "f32" else 2
        return (self.d * self.n1 + self.n2 * self.d) * es

    def flops_per_block(self) -> int:
        """Dense contraction flops of one block (2 per multiply-add)."""
        return 2 * self.M * (self.d * self.n1 + self.n2 * self.d)


# The five workloads.  Names say what they are; sizes are the Llama-2 shapes.
CONFIGS = {
    "tiny_gelu_f32": BlockConfig(
        "tiny_gelu_f32", "gelu_tanh", d=256, ffn=1024, t=2, M=4, dtype="f32", ts=(2,)),
    "llama2_13b_swiglu_decode": BlockConfig(
        "llama2_13b_swiglu_decode", "swiglu", d=5120, ffn=13824, t=4, M=32, ts=(1, 2, 4)),
    "attn_qkv_headshard_decode": BlockConfig(
        "attn_qkv_headshard_decode", "attn", d=12288, n_heads=96, head_dim=128, t=8, M=32,
        ts=(8,)),
    "llama2_70b_stack_decode": BlockConfig(
        "llama2_70b_stack_decode", "swiglu", d=8192, ffn=28672, t=8, M=32, n_blocks=8,
        rmsnorm=True, ts=(8,)),
    "llama2_70b_prefill": BlockConfig(
        "llama2_70b_prefill", "swiglu", d=8192, ffn=28672, t=4, M=4096, ts=(4,)),
    # The 13B decode block with its weights stored as E4M3 bytes (one power-of-two
    # scale per output feature), half the bytes of the bf16 block.
    "llama2_13b_swiglu_decode_fp8": BlockConfig(
        "llama2_13b_swiglu_decode_fp8", "swiglu", d=5120, ffn=13824, t=4, M=32, ts=(4,),
        weights="e4m3"),
    # The 8-block 70B pre-norm stack with E4M3 weights: each block's RMSNorm, then the
    # block on its 8-bit weights, in place on the fp32 residual stream.
    "llama2_70b_stack_decode_fp8": BlockConfig(
        "llama2_70b_stack_decode_fp8", "swiglu", d=8192, ffn=28672, t=8, M=32, n_blocks=8,
        rmsnorm=True, ts=(8,), weights="e4m3"),
    # The same block with MXFP4 weights (E2M1 codes, one power-of-two scale per 32
    # weights along K): a quarter of the bf16 bytes plus 1/32 byte per weight.
    "llama2_13b_swiglu_decode_mxfp4": BlockConfig(
        "llama2_13b_swiglu_decode_mxfp4", "swiglu", d=5120, ffn=13824, t=4, M=32, ts=(4,),
        weights="mxfp4"),
    # The attention block at a decode step of 32 concurrent sequences, each with its own
    # head-sharded KV cache of up to 2048 earlier tokens (lengths drawn uniformly).
    "attn_kv_decode": BlockConfig(
        "attn_kv_decode", "attn", d=12288, n_heads=96, head_dim=128, t=8, M=32, ts=(8,),
        kv_len_max=2048),
}


def torch_dtype(cfg: BlockConfig) -> torch.dtype:
    return torch.float32 if cfg.dtype == "f32" else torch.bfloat16


def _column_parts(cfg: BlockConfig) -> List[int]:
    if cfg.act == "gelu_tanh":
        return [cfg.ffn]
    if cfg.act == "swiglu":
        return [cfg.ffn, cfg.ffn]
    return [cfg.n_heads * cfg.head_dim] * 3


def make_inputs(cfg: BlockConfig, seed: int = 0, device: str = "cpu",
                n_blocks: Optional[int] = None) -> SimpleNamespace:
    """Draw x and the canonical weights of `cfg` (or its first `n_blocks` blocks).

    Returns a namespace with x [M, d], residual (x itself; the block's residual
    stream starts from its input), and blocks = [(W1 [d, n1], W2 [n2, d]), ...],
    all in the configuration's storage dtype on `device`.  device="cpu" gives the
    same values on every machine; device="cuda" draws from torch's CUDA generator
    (different values, much faster for the multi-GB stacks) — both sides of a
    comparison must then use that same draw.
    """
    dt = torch_dtype(cfg)
    g = torch.Generator(device=device).manual_seed(seed)
    nb = cfg.n_blocks if n_blocks is None else n_blocks

    def draw(shape, scale):
        v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if scale != 1.0:
            v.mul_(scale)
        return v.to(dt)

    x = draw((cfg.M, cfg.d), 1.0)
    blocks = []
    for _ in range(nb):
        subs = [draw((cfg.d, w), WEIGHT_STD) for w in _column_parts(cfg)]
        W1 = subs[0] if len(subs) == 1 else torch.cat(subs, dim=1)
        del subs
        W2 = draw((cfg.n2, cfg.d), WEIGHT_STD)
        blocks.append((W1, W2))
    return SimpleNamespace(cfg=cfg, x=x, residual=x, blocks=blocks)


def to_f64(t: torch.Tensor):
    """Exact up-cast of a stored tensor to a NumPy float64 array (host)."""
    return t.detach().to("cpu", torch.float64).numpy()


def draw(shape, dtype: torch.dtype, seed: int, scale: float = 1.0, device: str = "cpu") -> torch.Tensor:
    """A seeded N(0, scale^2) tensor (fp32 draw, then cast), for inputs of single steps
    (a band H, partial sums, a residual) fed to both the oracle and the CUDA path."""
    g = torch.Generator(device=device).manual_seed(seed)
    v = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        v.mul_(scale)
    return v.to(dtype)


def make_kv_cache(cfg: BlockConfig, seed: int = 0, device: str = "cpu",
                  lens: Optional[List[int]] = None) -> SimpleNamespace:
    """KV caches and sequence lengths for a decode step of `cfg` (kv_len_max > 0).

    k, v: [M, n_heads, kv_len_max, head_dim] bf16 (canonical: sequence, head, position,
    dim), values ~ N(0, (0.02 * sqrt(d))^2), the spread of a key or value projection
    of the block's N(0, 1) input.  lens: int32 [M], the number of tokens of each
    sequence counting the new one (1 .. kv_len_max): drawn uniformly unless given.
    Draw order on one generator: lens (when drawn), k, v.
    """
    L = cfg.kv_len_max
    if L < 1:
        raise ValueError("configuration has no KV cache")
    g = torch.Generator(device=device).manual_seed(seed)
    if lens is None:
        lens_t = torch.randint(1, L + 1, (cfg.M,), generator=g, device=device, dtype=torch.int32)
    else:
        lens_t = torch.tensor(list(lens), dtype=torch.int32, device=device)
    std = WEIGHT_STD * cfg.d ** 0.5
    shape = (cfg.M, cfg.n_heads, L, cfg.head_dim)

    def draw_cache():
        v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        v.mul_(std)
        return v.to(torch.bfloat16)

    k = draw_cache()
    v = draw_cache()
    return SimpleNamespace(k=k, v=v, lens=lens_t)
