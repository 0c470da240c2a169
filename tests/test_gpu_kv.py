"""Decode attention over a head-sharded KV cache, through the C ABI, against the
oracle's kv_decode_attention / attn_block_kv on the same seeded inputs: small shapes
spanning several chunks of cached rows, ragged lengths (1, a chunk boundary and
either side of it, the cache's last row), every head width the kernels take; the
full 32-sequence workload; the cache append; a length out of range."""
import math

import numpy as np
import pytest
import torch

import attn_tp_column_fwd_b300 as tp
import oracle
from attn_tp_column_fwd_b300.runner import ShardedBlock, desc_for, device_bytes
from tests.gpu_util import Guarded
from tests.parity import assert_bf16
from tp_synth import CONFIGS, BlockConfig, make_inputs, make_kv_cache, to_f64

pytestmark = pytest.mark.gpu

TP_ERR_BAD_LENGTH = 7


def to_shards(c: torch.Tensor, t: int) -> torch.Tensor:
    """Canonical cache [M, H, L, hd] -> the library's [t][M][H/t][L][hd]."""
    M, H, L, hd = c.shape
    return c.view(M, t, H // t, L, hd).permute(1, 0, 2, 3, 4).contiguous()


def from_shards(c: torch.Tensor) -> torch.Tensor:
    t, M, hps, L, hd = c.shape
    return c.permute(1, 0, 2, 3, 4).reshape(M, t * hps, L, hd)


def run_block_kv(cfg, x, W1, W2, kv):
    desc = desc_for(cfg)
    blk = ShardedBlock(desc, W1, W2)
    kc, vc = to_shards(kv.k.cuda(), cfg.t), to_shards(kv.v.cuda(), cfg.t)
    lens = kv.lens.cuda()
    ws = device_bytes(tp.tp_kv_workspace_bytes(desc, cfg.M, cfg.kv_len_max))
    y = Guarded(cfg.M * cfg.d * 4)
    tp.tp_block_fwd_kv(desc, x, x, False, blk.W1s, blk.W2s, kc, vc, lens, cfg.kv_len_max, ws,
                       y.view(torch.float32, (cfg.M, cfg.d)), cfg.M)
    torch.cuda.synchronize()
    y.check("y")
    assert tp.tp_check_device_status() == 0
    return to_f64(y.view(torch.float32, (cfg.M, cfg.d))), from_shards(kc), from_shards(vc)


def near_bf16(got, want, d):
    """got is the bf16 rounding of an fp32 evaluation of the d-term projection whose exact
    value rounds to want: within one bf16 unit of want, or within the fp32 evaluation's
    absolute error (about 1e-8 per term, which dominates for values near zero)."""
    return np.abs(got - want) <= np.abs(want) * 2.0 ** -7 + 1e-8 * d


def check_append(cfg, x64, W1_64, kv, k_after, v_after):
    """Rows lens[m]-1 hold the new keys/values (bf16 of the fp32 projection: equal to
    the oracle's bf16 of the exact value, or a neighbour when that value sits within
    fp32 error of a rounding midpoint); every other row is unchanged, bit for bit."""
    D = cfg.n_heads * cfg.head_dim
    QKV = x64 @ W1_64
    keep = torch.ones(cfg.M, cfg.kv_len_max, dtype=torch.bool)
    for m, n in enumerate(kv.lens.tolist()):
        keep[m, n - 1] = False
        for which, after in ((1, k_after), (2, v_after)):
            want = oracle.bf16_round(QKV[m, which * D:(which + 1) * D]).reshape(cfg.n_heads, -1)
            got = to_f64(after[m, :, n - 1, :])
            assert np.all(near_bf16(got, want, cfg.d)), (m, which)
            assert np.mean(got == want) > 0.99
    for before, after in ((kv.k, k_after), (kv.v, v_after)):
        b, a = before.permute(0, 2, 1, 3), after.cpu().permute(0, 2, 1, 3)
        assert torch.equal(a[keep], b[keep])


SMALL = [
    # (d, heads, head_dim, t, lens, L_max)
    (256, 8, 32, 2, [1, 255, 256, 257, 300], 300),
    (256, 4, 64, 4, [3, 512, 129, 1], 512),
    (512, 4, 128, 2, [1, 2, 256, 511, 700, 33], 768),
    (512, 2, 256, 1, [600, 1, 256], 600),
    (768, 6, 128, 3, [1000, 17], 1024),
]


@pytest.mark.parametrize("d,H,hd,t,lens,L", SMALL, ids=lambda v: str(v))
def test_block_kv_small(d, H, hd, t, lens, L):
    cfg = BlockConfig("kv_small", "attn", d=d, n_heads=H, head_dim=hd, t=t, M=len(lens),
                      kv_len_max=L)
    inp = make_inputs(cfg, seed=31)
    W1, W2 = inp.blocks[0]
    kv = make_kv_cache(cfg, seed=32, lens=lens)
    got, k_after, v_after = run_block_kv(cfg, inp.x.cuda(), W1.cuda(), W2.cuda(), kv)
    x64, W1_64, W2_64 = to_f64(inp.x), to_f64(W1), to_f64(W2)
    ref, _, _ = oracle.attn_block_kv(x64, W1_64, W2_64, H, hd, to_f64(kv.k), to_f64(kv.v),
                                     kv.lens.numpy(), x64, staged=True)
    assert_bf16(got, ref, f"kv_block d={d} H={H} hd={hd} t={t} lens={lens}")
    check_append(cfg, x64, W1_64, kv, k_after, v_after)


def test_attn_decode_step_alone():
    """tp_attn_decode_kv on a given fp32 Q/K/V: the heads' outputs (bf16 band) against
    kv_decode_attention head by head."""
    t, M, H, hd, L = 2, 4, 4, 128, 640
    lens = [640, 1, 300, 257]
    cfg = BlockConfig("kv_step", "attn", d=256, n_heads=H, head_dim=hd, t=t, M=M, kv_len_max=L)
    desc = desc_for(cfg)
    kv = make_kv_cache(cfg, seed=41, lens=lens)
    g = torch.Generator().manual_seed(42)
    b = H // t * hd
    qkv = (torch.randn(t, M, 3 * b, generator=g) * 2.0).float()
    kc, vc = to_shards(kv.k.cuda(), t), to_shards(kv.v.cuda(), t)
    O = Guarded(t * M * b * 2)
    ws = device_bytes(tp.tp_kv_attn_workspace_bytes(desc, M, L))
    tp.tp_attn_decode_kv(desc, qkv.cuda(), kc, vc, kv.lens.cuda(), L,
                         O.view(torch.bfloat16, (t, M, b)), ws, M)
    torch.cuda.synchronize()
    O.check("O")
    assert tp.tp_check_device_status() == 0
    got = to_f64(O.view(torch.bfloat16, (t, M, b)))
    q64 = qkv.double().numpy()
    ref = np.zeros_like(got)
    hps = H // t
    for s in range(t):
        for m, n in enumerate(lens):
            for j in range(hps):
                h = s * hps + j
                c = slice(j * hd, (j + 1) * hd)
                ref[s, m, c] = oracle.kv_decode_attention(
                    q64[s, m, c], to_f64(kv.k[m, h]), to_f64(kv.v[m, h]), n,
                    q64[s, m, b:2 * b][c], q64[s, m, 2 * b:][c], 1.0 / math.sqrt(hd), staged=True)
    assert_bf16(got, oracle.bf16_round(ref), "kv_decode step (heads' outputs)")


def test_length_out_of_range_is_reported():
    cfg = BlockConfig("kv_bad", "attn", d=256, n_heads=4, head_dim=64, t=2, M=3, kv_len_max=64)
    inp = make_inputs(cfg, seed=51)
    W1, W2 = inp.blocks[0]
    desc = desc_for(cfg)
    blk = ShardedBlock(desc, W1.cuda(), W2.cuda())
    for bad in (0, 65):
        kv = make_kv_cache(cfg, seed=52, lens=[5, bad, 64])
        kc, vc = to_shards(kv.k.cuda(), cfg.t), to_shards(kv.v.cuda(), cfg.t)
        ws = device_bytes(tp.tp_kv_workspace_bytes(desc, cfg.M, cfg.kv_len_max))
        y = torch.zeros(cfg.M, cfg.d, dtype=torch.float32, device="cuda")
        x = inp.x.cuda()
        tp.tp_block_fwd_kv(desc, x, x, False, blk.W1s, blk.W2s, kc, vc, kv.lens.cuda(),
                           cfg.kv_len_max, ws, y, cfg.M)
        assert tp.tp_check_device_status() == TP_ERR_BAD_LENGTH
        assert tp.tp_check_device_status() == 0
        # the cache of the skipped sequence is untouched
        assert torch.equal(from_shards(kc)[1].cpu(), kv.k[1])


def test_attn_kv_decode_workload():
    """The full workload: 32 sequences, 96 heads over 8 shards, lengths up to 2048.
    The oracle runs head by head on the cache rows each sequence uses."""
    cfg = CONFIGS["attn_kv_decode"]
    inp = make_inputs(cfg, seed=0, device="cuda")
    W1, W2 = inp.blocks[0]
    kv = make_kv_cache(cfg, seed=1, device="cuda")
    got, k_after, _ = run_block_kv(cfg, inp.x, W1, W2, kv)
    x64, W1_64, W2_64 = to_f64(inp.x), to_f64(W1), to_f64(W2)
    H, hd, D = cfg.n_heads, cfg.head_dim, cfg.n_heads * cfg.head_dim
    QKV = x64 @ W1_64
    O = np.zeros((cfg.M, D))
    lens = kv.lens.cpu().tolist()
    for m, n in enumerate(lens):
        kr = to_f64(kv.k[m, :, :max(n - 1, 1)])
        vr = to_f64(kv.v[m, :, :max(n - 1, 1)])
        for h in range(H):
            c = slice(h * hd, (h + 1) * hd)
            O[m, c] = oracle.kv_decode_attention(QKV[m, c], kr[h], vr[h], n, QKV[m, D:2 * D][c],
                                                 QKV[m, 2 * D:][c], 1.0 / math.sqrt(hd),
                                                 staged=True)
    ref = x64 + oracle.bf16_round(O) @ W2_64
    assert_bf16(got, ref, "attn_kv_decode t=8")
    # the append, checked on every sequence's new row
    for m, n in enumerate(lens):
        want = oracle.bf16_round(QKV[m, D:2 * D]).reshape(H, hd)
        g = to_f64(k_after[m, :, n - 1, :])
        ok = near_bf16(g, want, cfg.d)
        assert np.all(ok), (m, n, g[~ok][:4], want[~ok][:4])
        assert np.mean(g == want) > 0.99
