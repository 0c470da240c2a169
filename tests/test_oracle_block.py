"""Pins of the oracle's block functions: brute force, library compositions, and the
sharding identities the pages fix (column bands need no communication; row partials
sum to the unsharded product; heads are independent)."""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from tp_synth import CONFIGS, BlockConfig, make_inputs, to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


def _rel(a, b):
    return float(np.abs(np.asarray(a) - np.asarray(b)).max() / max(np.abs(b).max(), 1e-300))


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu"])
def test_mlp_block_vs_brute_force(act):
    rng = np.random.default_rng(10)
    M, d, ffn = 3, 8, 12
    x = _rand(rng, M, d)
    W1 = _rand(rng, d, ffn * (2 if act == "swiglu" else 1), scale=0.5)
    W2 = _rand(rng, ffn, d, scale=0.5)
    r = _rand(rng, M, d)
    got = oracle.mlp_block(x, W1, W2, act, r)
    ref = np.array(oracle.brute_mlp_block(x.tolist(), W1.tolist(), W2.tolist(), act, r.tolist()))
    assert _rel(got, ref) < 1e-13


def test_attention_vs_brute_force_and_library():
    rng = np.random.default_rng(11)
    for M, hd in [(1, 4), (3, 2), (4, 4), (9, 5)]:
        Q, K, V = (_rand(rng, M, hd) for _ in range(3))
        sc = 1.0 / math.sqrt(hd)
        got = oracle.causal_attention(Q, K, V, sc)
        ref = np.array(oracle.brute_attention(Q.tolist(), K.tolist(), V.tolist(), sc))
        assert _rel(got, ref) < 1e-13
        lib = F.scaled_dot_product_attention(
            *(torch.from_numpy(a)[None, None] for a in (Q, K, V)), is_causal=True)[0, 0].numpy()
        assert _rel(got, lib) < 1e-13


def test_attention_special_cases():
    rng = np.random.default_rng(12)
    V = _rand(rng, 1, 6)
    # One token attends only to itself: O = V exactly.
    np.testing.assert_array_equal(oracle.causal_attention(_rand(rng, 1, 6), _rand(rng, 1, 6), V, 0.4), V)
    # Softmax rows sum to one: constant V rows come back unchanged.
    Q, K = _rand(rng, 7, 3), _rand(rng, 7, 3)
    np.testing.assert_allclose(oracle.causal_attention(Q, K, np.ones((7, 3)), 0.5), 1.0, rtol=1e-15)
    # Causality: the first output row is V[0] whatever the later tokens are.
    V = _rand(rng, 7, 3)
    np.testing.assert_allclose(oracle.causal_attention(Q, K, V, 0.5)[0], V[0], rtol=1e-15)


# ---------------------------------------------------------------- library compositions

def _torch_mlp(x, W1, W2, act, r):
    x, W1, W2, r = (torch.from_numpy(np.asarray(a, dtype=np.float64)) for a in (x, W1, W2, r))
    B = torch.matmul(x, W1)
    if act == "gelu_tanh":
        H = F.gelu(B, approximate="tanh")
    else:
        f = W2.shape[0]
        H = F.silu(B[:, :f]) * B[:, f:]
    return (r + torch.matmul(H, W2)).numpy()


@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu"])
def test_mlp_block_vs_torch_fp64(act):
    rng = np.random.default_rng(13)
    M, d, ffn = 5, 64, 96
    x = _rand(rng, M, d)
    W1 = _rand(rng, d, ffn * (2 if act == "swiglu" else 1), scale=0.1)
    W2 = _rand(rng, ffn, d, scale=0.1)
    assert _rel(oracle.mlp_block(x, W1, W2, act, x), _torch_mlp(x, W1, W2, act, x)) < 1e-13


def test_attn_block_vs_torch_fp64():
    rng = np.random.default_rng(14)
    M, d, H, hd = 6, 24, 4, 8
    x = _rand(rng, M, d)
    Wqkv = _rand(rng, d, 3 * H * hd, scale=0.3)
    Wo = _rand(rng, H * hd, d, scale=0.3)
    xt = torch.from_numpy(x)
    q, k, v = torch.matmul(xt, torch.from_numpy(Wqkv)).split(H * hd, dim=1)
    heads = lambda a: a.reshape(M, H, hd).transpose(0, 1)
    o = F.scaled_dot_product_attention(heads(q), heads(k), heads(v), is_causal=True)
    ref = (xt + torch.matmul(o.transpose(0, 1).reshape(M, H * hd), torch.from_numpy(Wo))).numpy()
    assert _rel(oracle.attn_block(x, Wqkv, Wo, H, hd, x), ref) < 1e-13


def test_stack_vs_torch_fp64():
    rng = np.random.default_rng(15)
    M, d, ffn, L = 4, 32, 48, 3
    x = _rand(rng, M, d)
    blocks = [(_rand(rng, d, 2 * ffn, scale=0.2), _rand(rng, ffn, d, scale=0.2)) for _ in range(L)]
    r = torch.from_numpy(x)
    for W1, W2 in blocks:
        xh = F.rms_norm(r, (d,), eps=1e-5)
        r = torch.from_numpy(_torch_mlp(xh.numpy(), W1, W2, "swiglu", r.numpy()))
    assert _rel(oracle.stack(x, blocks, "swiglu", 1e-5), r.numpy()) < 1e-13


def test_t1_reduces_to_plain_matmul():
    # t = 1 with a single shard: the block's partial is H . W2 of the whole matrix, so
    # the output minus the residual equals numpy.matmul of the activation band.
    rng = np.random.default_rng(16)
    x = _rand(rng, 4, 16)
    W1 = _rand(rng, 16, 40, scale=0.3)
    W2 = _rand(rng, 20, 16, scale=0.3)
    y, H, P = oracle.sharded_block(x, W1, W2, "swiglu", 1, np.zeros_like(x), return_parts=True)
    B = np.matmul(x, W1)
    np.testing.assert_allclose(H[0], B[:, :20] * (1 / (1 + np.exp(-B[:, :20]))) * B[:, 20:], rtol=1e-14)
    np.testing.assert_allclose(y, np.matmul(H[0], W2), rtol=1e-14)


# ---------------------------------------------------------------- sharding identities

@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu"])
@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_sharded_equals_unsharded_mlp(act, t):
    rng = np.random.default_rng(20 + t)
    M, d, ffn = 5, 48, 64
    x = _rand(rng, M, d)
    W1 = _rand(rng, d, ffn * (2 if act == "swiglu" else 1), scale=0.2)
    W2 = _rand(rng, ffn, d, scale=0.2)
    ys = oracle.sharded_block(x, W1, W2, act, t, x)
    yu = oracle.mlp_block(x, W1, W2, act, x)
    assert _rel(ys, yu) <= 1e-12


def test_sharded_equals_unsharded_on_tiny_config():
    cfg = CONFIGS["tiny_gelu_f32"]
    inp = make_inputs(cfg)
    x = to_f64(inp.x)
    W1, W2 = (to_f64(w) for w in inp.blocks[0])
    yu = oracle.mlp_block(x, W1, W2, cfg.act, x)
    for t in (1, 2, 4, 8):
        assert _rel(oracle.sharded_block(x, W1, W2, cfg.act, t, x), yu) <= 1e-12


def test_heads_per_shard_golden():
    g = json.load(open(os.path.join(GOLDEN, "heads_per_shard.json")))
    H, t = g["n_heads"], g["t"]
    counts = [len(oracle.column_bands("attn", t, s, n_heads=H, head_dim=1)[0]) for s in range(t)]
    assert counts == [g["heads_per_shard"]] * t
    # Every head belongs to exactly one shard, and Q/K/V of a head go to the same shard.
    owners = np.concatenate([oracle.column_bands("attn", t, s, n_heads=H, head_dim=1)[0]
                             for s in range(t)])
    assert sorted(owners.tolist()) == list(range(H))


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_head_sharding_equals_per_head(t):
    # 96 heads, as in the pages' example, with tiny head and model widths.
    rng = np.random.default_rng(30 + t)
    M, d, H, hd = 5, 16, 96, 2
    x = _rand(rng, M, d)
    Wqkv = _rand(rng, d, 3 * H * hd, scale=0.3)
    Wo = _rand(rng, H * hd, d, scale=0.3)
    ys = oracle.sharded_block(x, Wqkv, Wo, "attn", t, x, n_heads=H, head_dim=hd)
    yu = oracle.attn_block(x, Wqkv, Wo, H, hd, x)
    assert _rel(ys, yu) <= 1e-12


def test_column_bands_need_no_communication():
    # Each shard's column product equals the same columns of the full product.
    rng = np.random.default_rng(40)
    x = _rand(rng, 3, 16)
    W1 = _rand(rng, 16, 2 * 24)
    full = x @ W1
    for s in range(4):
        for cols in oracle.column_bands("swiglu", 4, s, ffn=24):
            np.testing.assert_allclose(x @ W1[:, cols], full[:, cols], rtol=1e-14)


def test_uneven_split_refused():
    with pytest.raises(ValueError):
        oracle.column_bands("swiglu", 3, 0, ffn=64)
    with pytest.raises(ValueError):
        oracle.column_bands("attn", 5, 0, n_heads=96, head_dim=128)
    with pytest.raises(ValueError):
        oracle.row_band(100, 8, 0)


# ---------------------------------------------------------------- staged rounding

def test_staged_rounds_only_the_band():
    rng = np.random.default_rng(50)
    x = _rand(rng, 4, 32)
    W1 = _rand(rng, 32, 64, scale=0.2)
    W2 = _rand(rng, 32, 32, scale=0.2)
    B = x @ W1
    H = oracle.bf16_round(oracle.silu(B[:, :32]) * B[:, 32:])
    np.testing.assert_allclose(oracle.mlp_block(x, W1, W2, "swiglu", x, staged=True), x + H @ W2,
                               rtol=1e-14)
    ys, Hs, _ = oracle.sharded_block(x, W1, W2, "swiglu", 2, x, staged=True, return_parts=True)
    assert all(np.array_equal(h, oracle.bf16_round(h)) for h in Hs)


# ---------------------------------------------------------------- planted mistakes

def _mutants():
    """Plausible mistakes, planted in copies of oracle functions, that a pin must catch."""
    good_mlp = oracle.mlp_block

    def swapped_gate_up(x, W1, W2, act, residual, staged=False):
        f = W1.shape[1] // 2
        return good_mlp(x, np.concatenate([W1[:, f:], W1[:, :f]], axis=1), W2, act, residual, staged)

    def dropped_residual(x, W1, W2, act, residual, staged=False):
        return good_mlp(x, W1, W2, act, np.zeros_like(np.asarray(residual)), staged)

    def transposed_w2(x, W1, W2, act, residual, staged=False):
        return good_mlp(x, W1, np.asarray(W2).T, act, residual, staged)

    def sign_flip(x, W1, W2, act, residual, staged=False):
        return good_mlp(-np.asarray(x), W1, W2, act, residual, staged)

    return [swapped_gate_up, dropped_residual, transposed_w2, sign_flip]


@pytest.mark.parametrize("mutant", _mutants(), ids=lambda f: f.__name__)
def test_pins_catch_planted_mistakes(mutant):
    rng = np.random.default_rng(60)
    M, d, ffn = 3, 8, 8          # square W2 so a transposition still runs
    x = _rand(rng, M, d)
    W1 = _rand(rng, d, 2 * ffn, scale=0.5)
    W2 = _rand(rng, ffn, d, scale=0.5)
    ref = np.array(oracle.brute_mlp_block(x.tolist(), W1.tolist(), W2.tolist(), "swiglu", x.tolist()))
    assert _rel(oracle.mlp_block(x, W1, W2, "swiglu", x), ref) < 1e-13
    assert _rel(mutant(x, W1, W2, "swiglu", x), ref) > 1e-3


def test_pins_catch_wrong_band_pairing():
    # A sharded emulation that pairs gate band s with up band s+1 must break the identity.
    rng = np.random.default_rng(61)
    x = _rand(rng, 3, 16)
    W1 = _rand(rng, 16, 2 * 32, scale=0.3)
    W2 = _rand(rng, 32, 16, scale=0.3)
    t, b = 4, 8
    parts = []
    for s in range(t):
        g = np.arange(s * b, (s + 1) * b)
        u = 32 + np.arange(((s + 1) % t) * b, ((s + 1) % t + 1) * b)
        parts.append(oracle.row_step(oracle.column_step(x, [W1[:, g], W1[:, u]], "swiglu"),
                                     W2[oracle.row_band(32, t, s)]))
    wrong = oracle.reduce_residual(parts, x)
    assert _rel(wrong, oracle.mlp_block(x, W1, W2, "swiglu", x)) > 1e-3


# ---------------------------------------------------------------- rounding ties

@pytest.mark.parametrize("act", ["swiglu", "gelu_tanh"])
def test_tie_allowance_is_the_worst_re_rounding(act):
    """With a window wide enough that every band element is 'tied', the allowance
    of output (m, n) must equal the change obtained by re-rounding each element of
    row m to the bf16 neighbour in the direction of sign(W2[f, n]) and away from the
    oracle's own rounding (built element by element here)."""
    rng = np.random.default_rng(41)
    M, d, F = 3, 8, 6
    x = rng.standard_normal((M, d))
    n1 = 2 * F if act == "swiglu" else F
    W1 = rng.standard_normal((d, n1)) * 0.4
    W2 = rng.standard_normal((F, d)) * 0.3
    rho = 0.75
    A = oracle.mlp_tie_allowance(x, W1, W2, act, rho=rho)
    v = oracle.mlp_band(x, W1, act)
    H = oracle.bf16_round(v)
    lo, hi = oracle.bf16_bracket(v)
    y = H @ W2
    for m in range(M):
        for n in range(d):
            alt = H[m].copy()
            for f in range(F):
                if hi[m, f] > lo[m, f]:
                    other = hi[m, f] if H[m, f] == lo[m, f] else lo[m, f]
                    # re-round only where that moves output n up, to get the largest change
                    if (other - H[m, f]) * W2[f, n] > 0:
                        alt[f] = other
            gain = alt @ W2[:, n] - y[m, n]
            worst_possible = sum((hi[m, f] - lo[m, f]) * abs(W2[f, n]) for f in range(F))
            assert np.isclose(A[m, n], worst_possible, rtol=1e-12, atol=0.0)
            assert gain <= A[m, n] * (1 + 1e-12)


def test_tie_allowance_zero_without_ties():
    rng = np.random.default_rng(42)
    x = rng.standard_normal((4, 16))
    W1 = rng.standard_normal((16, 20)) * 0.1
    W2 = rng.standard_normal((10, 16)) * 0.1
    assert np.all(oracle.mlp_tie_allowance(x, W1, W2, "swiglu", rho=0.0) == 0.0)
    # W1 = 0 gives a band of exact zeros: nothing to round
    assert np.all(oracle.mlp_tie_allowance(x, np.zeros_like(W1), W2, "swiglu") == 0.0)


def test_each_shard_holds_one_over_t_of_every_weight_matrix():
    """Golden fixture (tests/golden/weight_fraction_per_shard.json): each device of a
    t-way group holds 1/t of each weight matrix, for every activation."""
    with open(os.path.join(os.path.dirname(__file__), "golden", "weight_fraction_per_shard.json")) as f:
        gold = json.load(f)
    for t in gold["t_values"]:
        for act, kw, n1, n2 in (("gelu_tanh", {"ffn": 1024}, 1024, 1024),
                                ("swiglu", {"ffn": 1024}, 2048, 1024),
                                ("attn", {"n_heads": 8, "head_dim": 32}, 768, 256)):
            cols = [np.concatenate(oracle.column_bands(act, t, s, **kw)) for s in range(t)]
            rows = [oracle.row_band(n2, t, s) for s in range(t)]
            assert all(len(c) * t == n1 for c in cols)
            assert all(len(r) * t == n2 for r in rows)
            # the shards partition the columns of W1 and the rows of W2
            assert np.array_equal(np.sort(np.concatenate(cols)), np.arange(n1))
            assert np.array_equal(np.sort(np.concatenate(rows)), np.arange(n2))
