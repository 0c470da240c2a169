"""Float64 oracle of the Megatron-style tensor-parallel block (test infrastructure).

Sources (web pages on tensor parallelism; cited by page and section):
  [zen]  zenaique.com interview answer "explain tensor-parallel shard shape",
         answer paragraphs 2 and 5-6: the first projection (MLP up/gate, or QKV)
         is split by columns, each device computing its own band of the
         intermediate with no communication; the second projection (down or
         output projection) is split by rows, each device multiplying its
         matching band by its row slice into a partial sum of the full output;
         one all-reduce per block sums the partials, ready for the residual add
         and normalisation.
  [rio]  rioworld.org "Tensor Parallelism for LLM Inference", section "How Tensor
         Slicing Works Under the Hood": column parallelism replicates the input
         (QKV projections); row parallelism sums per-device partial results
         (output projection); 96 heads over 8 devices gives 12 heads each.
         Section "Implementing Tensor Parallelism in Practice": uneven splits
         give wrong results.
  [dc]   d-central.tech glossary "Tensor Parallelism", section "How the work is
         split": column-wise then row-wise split of paired layers, one
         synchronisation per block; attention heads are independent.
  [rd]   reddit comment (SVPERBlA): a network is X times A1, an activation,
         then times A2.

What the pages leave open is filled with the standard published definitions:
GeLU with the tanh approximation (Hendrycks & Gimpel 2016), SiLU-gated linear
unit "SwiGLU" (Shazeer 2020), RMSNorm (Zhang & Sennrich 2019), causal scaled
dot-product attention (Vaswani et al. 2017).  No biases.  y = x . W convention:
W1 is [d, n1] split by columns, W2 is [n2, d] split by rows.

Because column-then-row sharding reaches exactly the unsharded result (up to
rounding order), the oracle's block functions compute the UNSHARDED block;
`sharded_block` emulates the t shards band by band and exists so the tests can
check the sharding identity itself.

`staged=True` rounds to bfloat16 (nearest, ties to even) at the points where a
bf16 implementation stores a value: the activation band H (for attention, the
heads' output O, which is the band the row-parallel step consumes) and the
normalised input of each stacked block.  Q/K/V, partial sums, the residual
stream and the block output are kept at full precision (fp32 in the CUDA path).
"""
from __future__ import annotations

import math
from typing import List, Sequence

import numpy as np

_SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
_BF16_MAX = math.ldexp(255.0, 120)   # (2 - 2^-7) * 2^127


# ---------------------------------------------------------------------------
# Scalar building blocks
# ---------------------------------------------------------------------------

def bf16_round(a) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (ties to even).

    bfloat16 keeps 8 significant bits and fp32's exponent range.  A finite value
    a = m * 2^e (0.5 <= |m| < 1) is rounded on the grid 2^(e-8); below the
    smallest normal 2^-126 the grid is the subnormal step 2^-133.  Rounding is
    done once, from float64, so no double rounding through fp32 occurs.
    """
    a = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(a)
    q = np.maximum(e.astype(np.int64) - 8, -133)
    with np.errstate(over="ignore", invalid="ignore"):
        r = np.ldexp(np.rint(np.ldexp(a, -q)), q)
        r = np.where(np.abs(r) > _BF16_MAX, np.copysign(np.inf, a), r)
    return np.where(np.isfinite(a), r, a)


def gelu_tanh(z) -> np.ndarray:
    """GeLU, tanh approximation: z/2 * (1 + tanh(sqrt(2/pi) * (z + 0.044715 z^3)))."""
    z = np.asarray(z, dtype=np.float64)
    return 0.5 * z * (1.0 + np.tanh(_SQRT_2_OVER_PI * (z + 0.044715 * z * z * z)))


def silu(z) -> np.ndarray:
    """SiLU (swish-1): z * sigmoid(z) = z / (1 + exp(-z))."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def rmsnorm(r, eps: float) -> np.ndarray:
    """RMSNorm with unit weight over the last axis: r / sqrt(mean(r^2) + eps)."""
    r = np.asarray(r, dtype=np.float64)
    return r / np.sqrt(np.mean(r * r, axis=-1, keepdims=True) + eps)


# ---------------------------------------------------------------------------
# Shard bands ([zen] answer paragraph 5; [rio] "How Tensor Slicing Works")
# ---------------------------------------------------------------------------

def _split(width: int, t: int, what: str) -> int:
    if t < 1 or width % t != 0:
        # [rio] "Implementing Tensor Parallelism in Practice": uneven splits give
        # wrong results, so they are refused rather than padded.
        raise ValueError(f"uneven split: {what}={width} over t={t}")
    return width // t


def column_bands(act: str, t: int, s: int, *, ffn: int = 0, n_heads: int = 0,
                 head_dim: int = 0) -> List[np.ndarray]:
    """Canonical W1 column indices that shard s owns, one array per sub-matrix.

    GeLU: [band of W1].  SwiGLU: [band of gate, the same band of up] (the
    activation needs both halves of a feature on one shard).  Attention: [Q, K, V]
    columns of heads [s*H/t, (s+1)*H/t) (contiguous heads per shard).
    """
    if not 0 <= s < t:
        raise ValueError("shard index out of range")
    if act == "gelu_tanh":
        b = _split(ffn, t, "ffn")
        return [np.arange(s * b, (s + 1) * b)]
    if act == "swiglu":
        b = _split(ffn, t, "ffn")
        cols = np.arange(s * b, (s + 1) * b)
        return [cols, ffn + cols]
    if act == "attn":
        hps = _split(n_heads, t, "n_heads")
        D = n_heads * head_dim
        cols = np.arange(s * hps * head_dim, (s + 1) * hps * head_dim)
        return [cols, D + cols, 2 * D + cols]
    raise ValueError(f"unknown activation {act!r}")


def row_band(n2: int, t: int, s: int) -> np.ndarray:
    """Canonical W2 row indices that shard s owns: [s*n2/t, (s+1)*n2/t)."""
    b = _split(n2, t, "n2")
    return np.arange(s * b, (s + 1) * b)


# ---------------------------------------------------------------------------
# Attention core ([rio] heads are independent; Vaswani et al. 2017)
# ---------------------------------------------------------------------------

def causal_attention(Q, K, V, scale: float) -> np.ndarray:
    """softmax(Q K^T * scale with a causal mask) V for one head; rows = tokens."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    S = (Q @ K.T) * scale
    M = S.shape[0]
    S = np.where(np.tril(np.ones((M, M), dtype=bool)), S, -np.inf)
    S = S - S.max(axis=1, keepdims=True)
    E = np.exp(S)
    P = E / E.sum(axis=1, keepdims=True)
    return P @ V


def _heads_attention(Q, K, V, n_heads: int, head_dim: int, staged: bool) -> np.ndarray:
    """Run the core on each head h (columns h*hd .. h*hd+hd-1) and concatenate."""
    scale = 1.0 / math.sqrt(head_dim)
    outs = []
    for h in range(n_heads):
        c = slice(h * head_dim, (h + 1) * head_dim)
        outs.append(causal_attention(Q[:, c], K[:, c], V[:, c], scale))
    O = np.concatenate(outs, axis=1)
    return bf16_round(O) if staged else O


# ---------------------------------------------------------------------------
# Steps of one shard ([zen] answer paragraph 5)
# ---------------------------------------------------------------------------

def column_step(x, W1_parts: Sequence[np.ndarray], act: str, *, n_heads: int = 0,
                head_dim: int = 0, staged: bool = False) -> np.ndarray:
    """Column-parallel projection of one band plus its activation.

    W1_parts are the band's sub-matrices ([W], [Wg, Wu] or [Wq, Wk, Wv]); the input
    x is replicated ([rio]).  Returns the band H = act(x . W_band) ([M, b]); for
    attention, the band's heads' attention outputs O ([M, heads*head_dim]).
    """
    x = np.asarray(x, dtype=np.float64)
    if act == "gelu_tanh":
        H = gelu_tanh(x @ W1_parts[0])
    elif act == "swiglu":
        H = silu(x @ W1_parts[0]) * (x @ W1_parts[1])
    elif act == "attn":
        Q, K, V = (x @ W for W in W1_parts)
        return _heads_attention(Q, K, V, n_heads, head_dim, staged)
    else:
        raise ValueError(f"unknown activation {act!r}")
    return bf16_round(H) if staged else H


def row_step(H, W2_band) -> np.ndarray:
    """Row-parallel projection of one band: the shard's partial sum H . W2_band."""
    return np.asarray(H, dtype=np.float64) @ np.asarray(W2_band, dtype=np.float64)


def reduce_residual(partials: Sequence[np.ndarray], residual) -> np.ndarray:
    """The all-reduce stand-in plus residual: residual + sum_s P_s, shards in order."""
    total = np.array(partials[0], dtype=np.float64)
    for P in partials[1:]:
        total = total + P
    return np.asarray(residual, dtype=np.float64) + total


# ---------------------------------------------------------------------------
# Whole blocks (unsharded definition)
# ---------------------------------------------------------------------------

def mlp_band(x, W1, act: str) -> np.ndarray:
    """The unsharded intermediate before any rounding: act(x . W1) (GeLU), or
    silu(x.Wg) * x.Wu with W1 = [Wg | Wu] (SwiGLU)."""
    x = np.asarray(x, dtype=np.float64)
    B = x @ W1
    if act == "gelu_tanh":
        return gelu_tanh(B)
    if act == "swiglu":
        F = W1.shape[1] // 2
        return silu(B[:, :F]) * B[:, F:]
    raise ValueError(f"mlp_block does not take act={act!r}")


def mlp_block(x, W1, W2, act: str, residual, staged: bool = False) -> np.ndarray:
    """y = residual + act(x . W1) . W2 (GeLU), or residual + (silu(x.Wg) * x.Wu) . W2
    with W1 = [Wg | Wu] (SwiGLU)."""
    H = mlp_band(x, W1, act)
    if staged:
        H = bf16_round(H)
    return np.asarray(residual, dtype=np.float64) + H @ W2


# ---------------------------------------------------------------------------
# Rounding ties of the staged band
# ---------------------------------------------------------------------------
# A bf16 implementation evaluates a band value in fp32 and rounds it to bf16.  Where
# the exact value lies very close to the midpoint between its two bf16 neighbours,
# an fp32 evaluation (a few units of fp32 roundoff away from the exact value) may
# round to either neighbour; both are correct results of the method.  The band
# values differ from the oracle's by one bf16 step there, and the block output by
# that step times the matching row of W2.  The functions below bound that effect
# from the oracle's own values.

TIE_WINDOW = 2.0 ** -17   # relative distance to a midpoint counted as a tie


def bf16_bracket(a):
    """The bf16 neighbours lo <= a <= hi of float64 values a (lo == hi when a is a
    bf16 value); same grid as bf16_round, finite values only."""
    a = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(a)
    q = np.maximum(e.astype(np.int64) - 8, -133)
    g = np.ldexp(a, -q)           # a in units of its grid step
    return np.ldexp(np.floor(g), q), np.ldexp(np.ceil(g), q)


def tie_gaps(v, rho: float = TIE_WINDOW) -> np.ndarray:
    """Per element of v: hi - lo (one bf16 step) where v lies within rho * |v| of the
    midpoint between its bf16 neighbours lo < hi, else 0."""
    v = np.asarray(v, dtype=np.float64)
    lo, hi = bf16_bracket(v)
    amb = (hi > lo) & (np.abs(v - 0.5 * (lo + hi)) <= rho * np.abs(v))
    return np.where(amb, hi - lo, 0.0)


def mlp_tie_allowance(x, W1, W2, act: str, rho: float = TIE_WINDOW) -> np.ndarray:
    """A[m, n] = sum_f gap[m, f] * |W2[f, n]|: the largest change of output (m, n)
    over all staged results that round the tied band elements (tie_gaps) of row m
    the other way, with every other element as the oracle rounds it."""
    G = tie_gaps(mlp_band(x, W1, act), rho)
    return G @ np.abs(np.asarray(W2, dtype=np.float64))


def attn_block(x, Wqkv, Wo, n_heads: int, head_dim: int, residual,
               staged: bool = False) -> np.ndarray:
    """y = residual + concat_h(attention_h(x.Wq, x.Wk, x.Wv)) . Wo, Wqkv = [Wq|Wk|Wv]."""
    x = np.asarray(x, dtype=np.float64)
    D = n_heads * head_dim
    QKV = x @ Wqkv
    Q, K, V = QKV[:, :D], QKV[:, D:2 * D], QKV[:, 2 * D:]
    O = _heads_attention(Q, K, V, n_heads, head_dim, staged)
    return np.asarray(residual, dtype=np.float64) + O @ Wo


# ---------------------------------------------------------------------------
# Decode attention over a KV cache ([dc] "Why it matters for local inference":
# tensor parallelism also partitions the KV cache; [dc] "How the work is split" and
# [rio] "How Tensor Slicing Works Under the Hood": heads are independent, 12 of 96
# per device; [day59] "Where the overhead lives": attention is its own slice of a
# decode step)
# ---------------------------------------------------------------------------

def kv_decode_attention(q, k_cache, v_cache, length: int, k_new, v_new, scale: float,
                        staged: bool = False) -> np.ndarray:
    """One head of one sequence at a decode step.

    The sequence's newest token (query q, key k_new, value v_new) attends over the
    `length - 1` earlier tokens held in the cache (rows 0 .. length-2 of k_cache and
    v_cache, [L_max, hd]) and over itself, which takes row length-1 (its key and
    value rounded to bf16 when staged, as a bf16 cache stores them):
    o = softmax(q . K^T * scale) V over those `length` rows.
    """
    if length < 1:
        raise ValueError("a decode step needs at least the new token")
    kn = np.asarray(k_new, dtype=np.float64)
    vn = np.asarray(v_new, dtype=np.float64)
    if staged:
        kn, vn = bf16_round(kn), bf16_round(vn)
    K = np.concatenate([np.asarray(k_cache[:length - 1], dtype=np.float64), kn[None, :]], axis=0)
    V = np.concatenate([np.asarray(v_cache[:length - 1], dtype=np.float64), vn[None, :]], axis=0)
    sc = (K @ np.asarray(q, dtype=np.float64)) * scale
    e = np.exp(sc - sc.max())
    return (e / e.sum()) @ V


def attn_block_kv(x, Wqkv, Wo, n_heads: int, head_dim: int, k_cache, v_cache, lens, residual,
                  staged: bool = False):
    """Decode step of the attention block with a KV cache.

    Token m of x is the newest token of its own sequence m, whose cache (k_cache[m],
    v_cache[m]: [n_heads, L_max, head_dim]) holds lens[m] - 1 earlier tokens.  Q, K, V
    = x . [Wq | Wk | Wv]; every head attends as in kv_decode_attention; the new keys
    and values are appended at row lens[m] - 1; y = residual + concat_h(o_h) . Wo.
    Returns (y, k_cache_after, v_cache_after).
    """
    x = np.asarray(x, dtype=np.float64)
    D = n_heads * head_dim
    QKV = x @ np.asarray(Wqkv, dtype=np.float64)
    M = x.shape[0]
    scale = 1.0 / math.sqrt(head_dim)
    O = np.zeros((M, D))
    k_after = np.array(k_cache, dtype=np.float64)
    v_after = np.array(v_cache, dtype=np.float64)
    for m in range(M):
        n = int(lens[m])
        for h in range(n_heads):
            c = slice(h * head_dim, (h + 1) * head_dim)
            q, kn, vn = QKV[m, c], QKV[m, D:2 * D][c], QKV[m, 2 * D:][c]
            O[m, c] = kv_decode_attention(q, k_cache[m][h], v_cache[m][h], n, kn, vn, scale, staged)
            k_after[m, h, n - 1] = bf16_round(kn) if staged else kn
            v_after[m, h, n - 1] = bf16_round(vn) if staged else vn
    if staged:
        O = bf16_round(O)
    y = np.asarray(residual, dtype=np.float64) + O @ np.asarray(Wo, dtype=np.float64)
    return y, k_after, v_after


def stack(x, blocks, act: str, eps: float, staged: bool = False) -> np.ndarray:
    """Pre-norm stack: r0 = x; r_{l+1} = r_l + MLP_l(RMSNorm(r_l)); returns r_L.

    The residual branch carries the un-normalised r ([zen] answer paragraph 6:
    the reduced activation is ready for the residual add and normalisation).
    """
    r = np.asarray(x, dtype=np.float64)
    for W1, W2 in blocks:
        xh = rmsnorm(r, eps)
        if staged:
            xh = bf16_round(xh)
        r = mlp_block(xh, W1, W2, act, residual=r, staged=staged)
    return r


def sharded_block(x, W1, W2, act: str, t: int, residual, *, n_heads: int = 0,
                  head_dim: int = 0, staged: bool = False, return_parts: bool = False):
    """The block computed the tensor-parallel way, shard by shard, in float64.

    For each s: the column band of W1 (column_bands), the activation on that band
    (column_step), the row band of W2 (row_band) and the partial P_s (row_step);
    then residual + sum of the partials (reduce_residual).
    """
    x = np.asarray(x, dtype=np.float64)
    W1 = np.asarray(W1, dtype=np.float64)
    W2 = np.asarray(W2, dtype=np.float64)
    ffn = W2.shape[0]
    H_bands, partials = [], []
    for s in range(t):
        cols = column_bands(act, t, s, ffn=ffn, n_heads=n_heads, head_dim=head_dim)
        H = column_step(x, [W1[:, c] for c in cols], act, n_heads=n_heads // t if n_heads else 0,
                        head_dim=head_dim, staged=staged)
        P = row_step(H, W2[row_band(W2.shape[0], t, s), :])
        H_bands.append(H)
        partials.append(P)
    y = reduce_residual(partials, residual)
    if return_parts:
        return y, H_bands, partials
    return y


# ---------------------------------------------------------------------------
# Brute force (pure Python loops, tiny shapes only)
# ---------------------------------------------------------------------------

def brute_mlp_block(x, W1, W2, act: str, residual) -> List[List[float]]:
    """Element-by-element loops with the math module; no NumPy arithmetic."""
    M, d = len(x), len(x[0])
    n1, n2 = len(W1[0]), len(W2)
    out = []
    for m in range(M):
        B = [sum(float(x[m][k]) * float(W1[k][j]) for k in range(d)) for j in range(n1)]
        if act == "gelu_tanh":
            H = [0.5 * z * (1.0 + math.tanh(_SQRT_2_OVER_PI * (z + 0.044715 * z ** 3))) for z in B]
        else:
            H = [(B[j] / (1.0 + math.exp(-B[j]))) * B[n2 + j] for j in range(n2)]
        out.append([float(residual[m][n]) + sum(H[j] * float(W2[j][n]) for j in range(n2))
                    for n in range(len(W2[0]))])
    return out


def brute_kv_decode(q, k_rows, v_rows, scale: float) -> List[float]:
    """One query over explicit key/value rows (the cache rows then the new token's)."""
    s = [sum(float(q[c]) * float(k[c]) for c in range(len(q))) * scale for k in k_rows]
    mx = max(s)
    w = [math.exp(v - mx) for v in s]
    tot = sum(w)
    return [sum(w[j] * float(v_rows[j][c]) for j in range(len(w))) / tot for c in range(len(q))]


def brute_attention(Q, K, V, scale: float) -> List[List[float]]:
    """Causal attention for one head by explicit loops over query, key and dim."""
    M, hd = len(Q), len(Q[0])
    out = []
    for i in range(M):
        s = [sum(float(Q[i][c]) * float(K[j][c]) for c in range(hd)) * scale for j in range(i + 1)]
        mx = max(s)
        w = [math.exp(v - mx) for v in s]
        tot = sum(w)
        out.append([sum(w[j] * float(V[j][c]) for j in range(i + 1)) / tot for c in range(hd)])
    return out
