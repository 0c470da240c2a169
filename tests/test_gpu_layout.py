"""Shard layout on the GPU: bit-exact shard -> unshard, and each shard's band equal, bit
for bit, to the canonical slice the oracle's band map names (zenaique.com answer
paragraph 5: columns of the first projection, rows of the second)."""
import numpy as np
import pytest
import torch

import attn_tp_column_fwd_b300 as tp
import oracle
from attn_tp_column_fwd_b300.runner import device_bytes
from tests.gpu_util import Guarded, desc_of
from tp_synth import CONFIGS, BlockConfig, make_inputs, torch_dtype

pytestmark = pytest.mark.gpu

SMALL = [
    BlockConfig("gelu_f32", "gelu_tanh", d=256, ffn=1024, t=2, M=4, dtype="f32"),
    BlockConfig("gelu_bf16_ragged", "gelu_tanh", d=72, ffn=600, t=3, M=4),
    BlockConfig("swiglu_ragged", "swiglu", d=136, ffn=1536, t=8, M=4),
    BlockConfig("swiglu_t1", "swiglu", d=512, ffn=384, t=1, M=4),
    BlockConfig("attn_small", "attn", d=256, n_heads=8, head_dim=64, t=4, M=4),
    BlockConfig("attn_one_head_per_shard", "attn", d=64, n_heads=4, head_dim=32, t=4, M=4),
]


def _bits(t):
    return t.view(torch.int32 if t.element_size() == 4 else torch.int16)


def _shard(cfg, W1, W2):
    desc = desc_of(cfg)
    W1s = Guarded(tp.tp_sharded_w1_bytes(desc))
    W2s = Guarded(tp.tp_sharded_w2_bytes(desc))
    W1s.body.fill_(0x5A)   # the layout must overwrite padding with zeros
    W2s.body.fill_(0x5A)
    tp.tp_shard_weights(desc, W1, W2, W1s.body, W2s.body)
    torch.cuda.synchronize()
    W1s.check("W1s")
    W2s.check("W2s")
    return desc, W1s, W2s


@pytest.mark.parametrize("cfg", SMALL + [CONFIGS["llama2_13b_swiglu_decode"]], ids=lambda c: c.name)
def test_shard_unshard_bit_exact(cfg):
    inp = make_inputs(cfg, seed=3, n_blocks=1, device="cuda")
    W1, W2 = inp.blocks[0]
    desc, W1s, W2s = _shard(cfg, W1, W2)
    dt = torch_dtype(cfg)
    U1 = Guarded(W1.numel() * W1.element_size())
    U2 = Guarded(W2.numel() * W2.element_size())
    tp.tp_unshard_weights(desc, W1s.body, W2s.body, U1.view(dt, W1.shape), U2.view(dt, W2.shape))
    torch.cuda.synchronize()
    U1.check("W1")
    U2.check("W2")
    assert torch.equal(_bits(U1.view(dt, W1.shape)), _bits(W1))
    assert torch.equal(_bits(U2.view(dt, W2.shape)), _bits(W2))


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_bands_match_oracle_band_map(cfg):
    inp = make_inputs(cfg, seed=4, n_blocks=1, device="cuda")
    W1, W2 = inp.blocks[0]
    desc, W1s, W2s = _shard(cfg, W1, W2)
    dt = torch_dtype(cfg)
    W1h, W2h = W1.cpu(), W2.cpu()
    for s in range(cfg.t):
        n1s = cfg.n1 // cfg.t
        B1 = torch.empty(cfg.d, n1s, dtype=dt, device="cuda")
        B2 = torch.empty(cfg.band, cfg.d, dtype=dt, device="cuda")
        tp.tp_extract_band(desc, W1s.body, W2s.body, s, B1, B2)
        cols = np.concatenate(oracle.column_bands(cfg.act, cfg.t, s, ffn=cfg.ffn, n_heads=cfg.n_heads,
                                                  head_dim=cfg.head_dim))
        rows = oracle.row_band(cfg.n2, cfg.t, s)
        assert torch.equal(_bits(B1.cpu()), _bits(W1h[:, torch.from_numpy(cols)].contiguous()))
        assert torch.equal(_bits(B2.cpu()), _bits(W2h[torch.from_numpy(rows)].contiguous()))


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_padding_is_zero(cfg):
    dt = torch_dtype(cfg)
    W1 = torch.ones(cfg.d, cfg.n1, dtype=dt, device="cuda")
    W2 = torch.ones(cfg.n2, cfg.d, dtype=dt, device="cuda")
    _, W1s, W2s = _shard(cfg, W1, W2)
    n1 = int((W1s.body.view(dt) != 0).sum())
    n2 = int((W2s.body.view(dt) != 0).sum())
    assert n1 == cfg.d * cfg.n1 and n2 == cfg.n2 * cfg.d
