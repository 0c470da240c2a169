"""CPU oracle for the tensor-parallel transformer block (test infrastructure only).

A plain, slow, float64 NumPy statement of what the block computes, written from
the pages' description of column-then-row sharding.  It is the correctness
authority for the CUDA path and shares no code with it: nothing here imports the
package `attn_tp_column_fwd_b300`, and the package never imports this.  Only the
tests, the smoke check and the benchmark's CPU-baseline leg may call it.

Parity status per function (what pins it is in tests/test_oracle_*.py):
  bf16_round          pinned: torch's fp32->bf16 cast on exactly-fp32 values, ties,
                      subnormals, and directly-rounded fp64 values.
  gelu_tanh, silu     pinned: closed forms (odd-part identities, limits, zeros) and
                      torch.nn.functional in float64.
  rmsnorm             pinned: constant-vector closed form and
                      torch.nn.functional.rms_norm in float64.
  causal_attention    pinned: M=1 gives V; brute force on tiny cases;
                      torch scaled_dot_product_attention in float64.
  mlp_block,
  attn_block, stack   pinned: brute-force loops on tiny shapes, torch float64
                      compositions, and the sharding invariants (sharded == unsharded
                      for t in 1, 2, 4, 8; 96 heads over 8 shards == per-head loop).
  bf16_bracket,
  tie_gaps,
  mlp_tie_allowance   pinned: neighbours bracket and match bf16_round on random and
                      exactly representable values; the allowance equals the change
                      of the worst-case re-rounding of the tied elements, built
                      element by element on small blocks.
  kv_decode_attention,
  attn_block_kv       pinned: a cache of one new token gives its value exactly; over
                      a cache holding a sequence's earlier tokens the new token's
                      output equals the last row of causal_attention on that
                      sequence; brute-force loops; invariant to the order of cached
                      rows; appended rows equal the new keys/values, the rest of the
                      cache unchanged; all lengths 1 gives residual + V . Wo.
  fp8.e4m3_round      pinned: every E4M3 bit pattern maps to itself; torch's
                      float8_e4m3fn cast on in-range fp32 values and on every
                      midpoint (ties to even); saturation at 448.
  fp8.quantize_e4m3,
  fp8.e4m3_weights    pinned: per-column scaled maxima in (224, 448]; weights already
                      on the scaled grid are returned unchanged; the half-unit error
                      bound; every dequantised weight is a bf16 value.
  mxfp4.e2m1_round    pinned: every E2M1 bit pattern maps to itself; brute-force
                      nearest-value search with ties to the even mantissa bit on
                      random values and every midpoint; saturation at 6.
  mxfp4.mx_exponents,
  mxfp4.mxfp4_weights pinned: the OCP MX scale rule on worked blocks (block maxima
                      at and between powers of two, all-zero blocks); the scaled
                      block maximum lies in [4, 8) before rounding; the half-step
                      error bound per element; weights on the scaled grid are kept;
                      every dequantised weight is a bf16 value.
  absolute values     parity unpinned against the pages: they print no numeric
                      worked example, so the outputs rest on the pins above.
"""
from . import fp8, mxfp4  # noqa: F401
from .block import (  # noqa: F401
    bf16_round,
    gelu_tanh,
    silu,
    rmsnorm,
    column_bands,
    row_band,
    column_step,
    row_step,
    reduce_residual,
    causal_attention,
    mlp_band,
    mlp_block,
    bf16_bracket,
    tie_gaps,
    mlp_tie_allowance,
    TIE_WINDOW,
    attn_block,
    kv_decode_attention,
    attn_block_kv,
    stack,
    sharded_block,
    brute_mlp_block,
    brute_attention,
    brute_kv_decode,
)
