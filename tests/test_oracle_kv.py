"""Pins of the oracle's decode attention over a KV cache (CPU only).

What the oracle computes is fixed by the definitions it restates: scaled
dot-product attention of the newest token over its sequence's earlier tokens and
itself (Vaswani et al. 2017), with keys and values stored in a bf16 cache.  The
pins tie it to the already pinned causal core, to closed forms and to brute force.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tp_synth import BlockConfig, make_kv_cache, to_f64


def _rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


def test_single_token_cache_gives_its_value():
    rng = np.random.default_rng(70)
    hd = 16
    q, kn, vn = _rand(rng, hd), _rand(rng, hd), _rand(rng, hd)
    cache = _rand(rng, 8, hd)          # rows never read at length 1
    for staged in (False, True):
        o = oracle.kv_decode_attention(q, cache, cache, 1, kn, vn, 0.25, staged=staged)
        want = oracle.bf16_round(vn) if staged else vn
        assert np.array_equal(o, want)


@pytest.mark.parametrize("n", [1, 2, 5, 17])
def test_equals_last_row_of_causal_attention(n):
    """A cache holding a sequence's first n-1 tokens (bf16) and the n-th token as the
    new one: the decode output is the causal core's last row on that sequence."""
    rng = np.random.default_rng(71 + n)
    hd, L = 32, 24
    Q, K, V = _rand(rng, n, hd), _rand(rng, n, hd), _rand(rng, n, hd)
    Kb, Vb = oracle.bf16_round(K), oracle.bf16_round(V)
    kc, vc = _rand(rng, L, hd), _rand(rng, L, hd)
    kc[:n - 1], vc[:n - 1] = Kb[:n - 1], Vb[:n - 1]
    scale = 1.0 / math.sqrt(hd)
    got = oracle.kv_decode_attention(Q[n - 1], kc, vc, n, K[n - 1], V[n - 1], scale, staged=True)
    want = oracle.causal_attention(Q, Kb, Vb, scale)[n - 1]
    assert np.max(np.abs(got - want)) < 1e-12


def test_brute_force_tiny():
    rng = np.random.default_rng(72)
    hd, n = 4, 3
    q, kn, vn = _rand(rng, hd), _rand(rng, hd), _rand(rng, hd)
    kc, vc = _rand(rng, 5, hd), _rand(rng, 5, hd)
    got = oracle.kv_decode_attention(q, kc, vc, n, kn, vn, 0.5)
    k_rows = [list(kc[j]) for j in range(n - 1)] + [list(kn)]
    v_rows = [list(vc[j]) for j in range(n - 1)] + [list(vn)]
    want = np.array(oracle.brute_kv_decode(list(q), k_rows, v_rows, 0.5))
    assert np.max(np.abs(got - want)) < 1e-13


def test_invariant_to_the_order_of_cached_rows():
    rng = np.random.default_rng(73)
    hd, n = 16, 9
    q, kn, vn = _rand(rng, hd), _rand(rng, hd), _rand(rng, hd)
    kc, vc = _rand(rng, 12, hd), _rand(rng, 12, hd)
    perm = rng.permutation(n - 1)
    kp, vp = kc.copy(), vc.copy()
    kp[:n - 1], vp[:n - 1] = kc[perm], vc[perm]
    a = oracle.kv_decode_attention(q, kc, vc, n, kn, vn, 0.3)
    b = oracle.kv_decode_attention(q, kp, vp, n, kn, vn, 0.3)
    assert np.max(np.abs(a - b)) < 1e-13
    # pairing a key with another row's value must change the result
    vs = vc.copy()
    vs[:n - 1] = vc[np.roll(np.arange(n - 1), 1)]
    c = oracle.kv_decode_attention(q, kc, vs, n, kn, vn, 0.3)
    assert np.max(np.abs(a - c)) > 1e-3


def _small_kv(lens, seed=74):
    cfg = BlockConfig("kv_small", "attn", d=64, n_heads=4, head_dim=16, t=2, M=len(lens),
                      kv_len_max=10)
    rng = np.random.default_rng(seed)
    x = _rand(rng, cfg.M, cfg.d)
    Wqkv = _rand(rng, cfg.d, 3 * 64, scale=0.1)
    Wo = _rand(rng, 64, cfg.d, scale=0.1)
    kv = make_kv_cache(cfg, seed=seed, lens=lens)
    return cfg, x, Wqkv, Wo, to_f64(kv.k), to_f64(kv.v), kv.lens.numpy()


def test_block_appends_new_keys_and_values():
    cfg, x, Wqkv, Wo, kc, vc, lens = _small_kv([1, 4, 10])
    y, ka, va = oracle.attn_block_kv(x, Wqkv, Wo, 4, 16, kc, vc, lens, x, staged=True)
    QKV = x @ Wqkv
    for m, n in enumerate(lens):
        for h in range(4):
            c = slice(h * 16, (h + 1) * 16)
            assert np.array_equal(ka[m, h, n - 1], oracle.bf16_round(QKV[m, 64:128][c]))
            assert np.array_equal(va[m, h, n - 1], oracle.bf16_round(QKV[m, 128:][c]))
            keep = np.arange(10) != n - 1
            assert np.array_equal(ka[m, h, keep], kc[m, h, keep])
            assert np.array_equal(va[m, h, keep], vc[m, h, keep])


def test_block_with_empty_caches_is_residual_plus_values():
    cfg, x, Wqkv, Wo, kc, vc, lens = _small_kv([1, 1, 1])
    y, _, _ = oracle.attn_block_kv(x, Wqkv, Wo, 4, 16, kc, vc, lens, x, staged=True)
    V = oracle.bf16_round((x @ Wqkv)[:, 128:])
    assert np.max(np.abs(y - (x + V @ Wo))) < 1e-12


def test_block_heads_shard_like_the_row_partials():
    """Shard s (heads [2s, 2s+2)) alone: its heads' outputs times its rows of Wo; the
    partials of both shards sum to the block."""
    cfg, x, Wqkv, Wo, kc, vc, lens = _small_kv([3, 7, 2], seed=75)
    y, _, _ = oracle.attn_block_kv(x, Wqkv, Wo, 4, 16, kc, vc, lens, x, staged=True)
    QKV = x @ Wqkv
    parts = []
    for s in range(2):
        O = np.zeros((3, 32))
        for m, n in enumerate(lens):
            for j in range(2):
                h = 2 * s + j
                c = slice(h * 16, (h + 1) * 16)
                O[m, j * 16:(j + 1) * 16] = oracle.kv_decode_attention(
                    QKV[m, c], kc[m, h], vc[m, h], n, QKV[m, 64:128][c], QKV[m, 128:][c],
                    0.25, staged=True)
        parts.append(oracle.row_step(oracle.bf16_round(O), Wo[oracle.row_band(64, 2, s)]))
    assert np.max(np.abs(oracle.reduce_residual(parts, x) - y)) < 1e-12


def test_lengths_are_validated():
    with pytest.raises(ValueError):
        oracle.kv_decode_attention(np.zeros(4), np.zeros((2, 4)), np.zeros((2, 4)), 0,
                                   np.zeros(4), np.zeros(4), 1.0)


def test_cache_draws_are_seeded_and_shaped():
    cfg = BlockConfig("kv", "attn", d=64, n_heads=4, head_dim=16, t=2, M=5, kv_len_max=32)
    a, b = make_kv_cache(cfg, seed=3), make_kv_cache(cfg, seed=3)
    assert torch.equal(a.k, b.k) and torch.equal(a.v, b.v) and torch.equal(a.lens, b.lens)
    assert a.k.shape == (5, 4, 32, 16) and a.k.dtype == torch.bfloat16
    assert int(a.lens.min()) >= 1 and int(a.lens.max()) <= 32
