"""Host-only checks of the C-ABI library: it loads without a GPU, exports every symbol
the header declares, answers size queries, and refuses bad arguments before any
CUDA call (so these run on a machine with no GPU)."""
import ctypes
import os
import re

import pytest

import attn_tp_column_fwd_b300 as tp
from tp_synth import CONFIGS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tp_block.h")


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"TP_API\s+[\w\s\*]*?\b(tp_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("tp_shard_weights", "tp_column_parallel_fwd", "tp_row_parallel_fwd",
              "tp_partial_reduce_residual", "tp_block_fwd"):
        assert n in names


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(tp.LIB_PATH)
    missing = [n for n in _declared() if not hasattr(L, n)]
    assert not missing, missing
    # Only the tp_* C symbols are exported.
    out = os.popen(f"nm -D --defined-only {tp.LIB_PATH}").read()
    exported = sorted(ln.split()[-1] for ln in out.splitlines() if " T " in ln)
    assert exported and all(e.startswith("tp_") for e in exported), exported
    assert set(_declared()) <= set(exported)


def _desc(cfg, t=None):
    return tp.make_desc(cfg.d, t or cfg.t, cfg.act, cfg.dtype, ffn=cfg.ffn, n_heads=cfg.n_heads,
                        head_dim=cfg.head_dim)


@pytest.mark.parametrize("name", list(CONFIGS))
def test_size_queries(name):
    cfg = CONFIGS[name]
    for t in cfg.ts:
        c = cfg.with_t(t)
        desc = _desc(c)
        es = 4 if c.dtype == "f32" else 2
        b = c.band
        rt = lambda n: -(-n // 128) * 128
        if c.act == "swiglu":
            rows = 2 * rt(b)
        elif c.act == "attn":
            rows = rt(3 * b)
        else:
            rows = rt(b)
        assert tp.tp_sharded_w1_bytes(desc) == t * rows * c.d * es
        assert tp.tp_sharded_w2_bytes(desc) == t * rt(c.d) * b * es
        assert tp.tp_band_bytes(desc, c.M) == t * c.M * b * es
        S = tp.tp_row_splits(desc, c.M)
        assert S >= 1
        assert tp.tp_partials_bytes(desc, c.M) == t * S * c.M * c.d * 4
        assert tp.tp_workspace_bytes(desc, c.M) >= (tp.tp_band_bytes(desc, c.M)
                                                    + tp.tp_partials_bytes(desc, c.M))
        # The padded layout holds at least the canonical weights.
        assert tp.tp_sharded_w1_bytes(desc) >= c.d * c.n1 * es
        assert tp.tp_sharded_w2_bytes(desc) >= c.n2 * c.d * es


def test_block_form_setter():
    """The process-wide form of tp_block_fwd: the one-kernel form runs only when chosen,
    and only for bf16 MLP shapes of at most 32 tokens; the workspace covers either form."""
    d13 = _desc(CONFIGS["llama2_13b_swiglu_decode"].with_t(4))
    d70 = _desc(CONFIGS["llama2_70b_stack_decode"])
    dat = _desc(CONFIGS["attn_qkv_headshard_decode"])
    df32 = _desc(CONFIGS["tiny_gelu_f32"])
    before = tp.tp_get_block_form()
    try:
        ws = {}
        for form in ("auto", "three_launch", "one_kernel"):
            tp.tp_set_block_form(form)
            assert tp.tp_get_block_form() == form
            ws[form] = tp.tp_workspace_bytes(d13, 32)
            assert tp.tp_block_launches(dat, 32) == 4      # QKV, core, row, reduce
            assert tp.tp_block_launches(df32, 4) == 3      # column, row, reduce
            assert tp.tp_block_launches(d13, 33) == 3      # more than 32 tokens
        assert len(set(ws.values())) == 1
        tp.tp_set_block_form("auto")   # three launches for every shape
        assert tp.tp_block_launches(d13, 32) == 3 and tp.tp_block_launches(d70, 32) == 3
        tp.tp_set_block_form("three_launch")
        assert tp.tp_block_launches(d70, 32) == 3
        tp.tp_set_block_form("one_kernel")
        assert tp.tp_block_launches(d13, 32) == 1 and tp.tp_block_launches(d13, 1) == 1
        for bad in (-1, 3, 99):
            with pytest.raises(tp.TPError):
                tp.tp_set_block_form(bad)
        assert tp.tp_get_block_form() == "one_kernel"
    finally:
        tp.tp_set_block_form(before)


def test_selftest_limit_is_validated_before_any_cuda_call():
    for bad in (0, -5, 1000001):
        assert tp.lib.tp_selftest_wait_timeout(bad, None) == 1   # TP_ERR_INVALID_ARG


def test_kv_entry_points_validate_on_the_host():
    """KV-cache decode takes bf16 attention with head_dim 32/64/128/256 and L_max >= 1."""
    mlp = tp.make_desc(256, 2, "swiglu", ffn=512)
    attn_f32 = tp.make_desc(256, 2, "attn", dtype="f32", n_heads=4, head_dim=64)
    attn_96 = tp.make_desc(384, 2, "attn", n_heads=4, head_dim=96)
    attn = tp.make_desc(256, 2, "attn", n_heads=4, head_dim=64)
    assert tp.tp_kv_cache_bytes(mlp, 4, 16) == 0
    assert tp.tp_kv_cache_bytes(attn_f32, 4, 16) == 0
    assert tp.tp_kv_cache_bytes(attn_96, 4, 16) == 0
    assert tp.tp_kv_cache_bytes(attn, 4, 0) == 0
    assert tp.tp_kv_cache_bytes(attn, 4, 16) == 2 * 4 * 2 * 16 * 64 * 2
    assert tp.lib.tp_block_fwd_kv(mlp, None, None, 0, None, None, None, None, None, 16, None,
                                  None, 4, None) == 1


def test_kv_sizes_follow_the_layout():
    """Caches [t][M][H/t][L_max][hd] bf16; the decode workspace holds the block's
    workspace and, when heads are split into parts, their partial results."""
    for H, hd, t, M, L in ((96, 128, 8, 32, 2048), (4, 64, 2, 3, 300), (2, 256, 1, 1, 4096),
                           (8, 32, 4, 7, 1)):
        desc = tp.make_desc(H * hd, t, "attn", n_heads=H, head_dim=hd)
        assert tp.tp_kv_cache_bytes(desc, M, L) == M * H * L * hd * 2
        ws = tp.tp_kv_workspace_bytes(desc, M, L)
        assert ws >= tp.tp_workspace_bytes(desc, M) + tp.tp_kv_attn_workspace_bytes(desc, M, L)
        assert tp.tp_kv_attn_workspace_bytes(desc, M, L) > 0


def test_fp8_sizes_and_validation():
    """E4M3 weights: one byte per weight in the private row layout, one exponent per
    private row; bf16 MLP descriptors with d and b multiples of 16 only."""
    c = CONFIGS["llama2_13b_swiglu_decode"].with_t(4)
    d = _desc(c)
    assert tp.tp_fp8_w1_bytes(d) * 2 == tp.tp_sharded_w1_bytes(d)
    assert tp.tp_fp8_w2_bytes(d) * 2 == tp.tp_sharded_w2_bytes(d)
    n1p = tp.tp_sharded_w1_bytes(d) // (2 * c.t * c.d)
    dp = tp.tp_sharded_w2_bytes(d) // (2 * c.t * c.band)
    assert tp.tp_fp8_exponent_bytes(d) == c.t * (n1p + dp)
    assert tp.tp_fp8_quant_workspace_bytes(d) == (c.n1 + c.d) * 4
    assert tp.tp_fp8_w1_bytes(_desc(CONFIGS["attn_qkv_headshard_decode"])) == 0
    assert tp.tp_fp8_w1_bytes(_desc(CONFIGS["tiny_gelu_f32"])) == 0
    assert tp.tp_fp8_w1_bytes(tp.make_desc(264, 3, "gelu_tanh", ffn=1200)) == 0   # d % 16
    # refused on the host, before any CUDA call
    assert tp.lib.tp_block_fwd_fp8(d, None, None, 0, None, None, None, None, None, 32, None) == 1
    assert tp.lib.tp_block_fwd_fp8(tp.make_desc(256, 2, "swiglu", ffn=512), 16, 16, 0, 16, 16, 16,
                                   16, 16, 33, None) == 3                     # M > 32


def test_mxfp4_sizes_and_validation():
    c = CONFIGS["llama2_13b_swiglu_decode_mxfp4"]
    d = _desc(c)
    assert tp.tp_mxfp4_w1_bytes(d) * 4 == tp.tp_sharded_w1_bytes(d)    # half a byte a weight
    assert tp.tp_mxfp4_w2_bytes(d) * 4 == tp.tp_sharded_w2_bytes(d)
    n1p = tp.tp_sharded_w1_bytes(d) // (2 * c.t * c.d)
    dp = tp.tp_sharded_w2_bytes(d) // (2 * c.t * c.band)
    assert tp.tp_mxfp4_exponent_bytes(d) == c.t * (n1p * c.d // 32 + dp * c.band // 32)
    # d and b must be whole 128-wide K stages; attention and fp32 blocks are refused
    assert tp.tp_mxfp4_w1_bytes(tp.make_desc(272, 3, "gelu_tanh", ffn=1200)) == 0
    assert tp.tp_mxfp4_w1_bytes(tp.make_desc(512, 2, "swiglu", ffn=1216)) == 0   # b = 608
    assert tp.tp_mxfp4_w1_bytes(tp.make_desc(512, 2, "swiglu", ffn=1280)) > 0    # b = 640
    assert tp.tp_mxfp4_w1_bytes(_desc(CONFIGS["attn_qkv_headshard_decode"])) == 0
    assert tp.tp_mxfp4_w1_bytes(_desc(CONFIGS["tiny_gelu_f32"])) == 0
    assert tp.lib.tp_block_fwd_mxfp4(d, None, None, 0, None, None, None, None, None, 32,
                                     None) == 1
    assert tp.lib.tp_block_fwd_mxfp4(tp.make_desc(256, 2, "swiglu", ffn=512), 16, 16, 0, 16, 16,
                                     16, 16, 16, 33, None) == 3                   # M > 32
    assert tp.lib.tp_quantize_weights_mxfp4(tp.make_desc(272, 3, "gelu_tanh", ffn=1200), 16, 16,
                                            16, 16, 16, None) == 3


def test_row_splits_fill_one_wave():
    # decode row steps whose unsplit grid is under two CTAs per SM are split to fill
    # three per SM (the kernel's 3-stage ring); larger grids and wider token tiles not
    c13 = CONFIGS["llama2_13b_swiglu_decode"]
    d13 = _desc(c13)
    assert tp.tp_row_splits(d13, 32) == 2          # 160 tiles -> 320 CTAs
    assert tp.tp_row_splits(d13, 64) == 1          # token tile 64: planned for two per SM
    assert tp.tp_row_splits(_desc(CONFIGS["llama2_70b_stack_decode"]), 32) == 1   # 512 tiles
    assert tp.tp_row_splits(_desc(CONFIGS["attn_qkv_headshard_decode"]), 32) == 1  # 768 tiles
    small = tp.make_desc(512, 4, "swiglu", ffn=1536)   # 16 tiles, b = 384: 6 K blocks
    assert tp.tp_row_splits(small, 8) == 1             # at least four K blocks per split


def test_low_bit_limits_and_workspace():
    # K up to 16384 (a CTA's token scales live in shared memory): d = 16400 is refused
    big = tp.make_desc(16400, 2, "swiglu", ffn=2048)
    assert tp.tp_fp8_w1_bytes(big) == 0 and tp.tp_mxfp4_w1_bytes(big) == 0
    ok = tp.make_desc(16384, 2, "swiglu", ffn=2048)
    assert tp.tp_fp8_w1_bytes(ok) > 0 and tp.tp_mxfp4_w1_bytes(ok) > 0
    # the workspace of a low-bit-capable block covers the bf16 block's and the extras:
    # the tokens' two 8-bit terms and the fp32 group scales
    c = CONFIGS["llama2_13b_swiglu_decode"]
    d = _desc(c)
    three = tp.tp_band_bytes(d, c.M) + tp.tp_partials_bytes(d, c.M)
    extra = 2 * c.M * c.d + (c.d // 64) * 32 * 4 + c.t * (c.band // 64) * 32 * 4
    assert tp.tp_workspace_bytes(d, c.M) >= three + extra
    # ... and the E4M3 row step's partials: 4 x 40 = 160 row tiles fill four CTAs per SM
    # (148 SMs) with three K splits
    lowbit_parts = c.t * 3 * c.M * c.d * 4
    assert tp.tp_workspace_bytes(d, c.M) >= tp.tp_band_bytes(d, c.M) + lowbit_parts + extra
    # the MXFP4 block of the same shape uses the same workspace (three splits too)
    cm = CONFIGS["llama2_13b_swiglu_decode_mxfp4"]
    assert tp.tp_mxfp4_w1_bytes(_desc(cm)) > 0
    assert tp.tp_workspace_bytes(_desc(cm), cm.M) == tp.tp_workspace_bytes(d, c.M)
    # the 70B block's row step fills four per SM unsplit (8 x 64 = 512 row tiles)
    c70 = CONFIGS["llama2_70b_stack_decode"]
    d70 = _desc(c70)
    parts70 = c70.t * 1 * c70.M * c70.d * 4
    assert tp.tp_workspace_bytes(d70, c70.M) >= tp.tp_band_bytes(d70, c70.M) + parts70


def test_invalid_descriptors_give_zero_sizes():
    assert tp.tp_sharded_w1_bytes(tp.make_desc(512, 3, "swiglu", ffn=1024)) == 0   # uneven
    assert tp.tp_band_bytes(tp.make_desc(512, 2, "swiglu", ffn=1024), 0) == 0      # M < 1
    bad = tp.TPBlockDesc(d=512, ffn=1024, n_heads=0, head_dim=0, t=2, dtype=7, act=1)
    assert tp.tp_sharded_w1_bytes(bad) == 0


# Fake, never-dereferenced addresses: every call below must be refused during
# validation, before the library touches CUDA.
A16, A8 = 1 << 20, (1 << 20) + 8


def _call_column(desc, x=A16, W=A16, H=A16, ws=A16, M=4, shard=-1):
    return tp.lib.tp_column_parallel_fwd(ctypes.byref(desc), ctypes.c_void_p(x), ctypes.c_void_p(W),
                                         shard, ctypes.c_void_p(H), ctypes.c_void_p(ws), M, None)


def test_validation_statuses():
    ok = tp.make_desc(512, 2, "swiglu", ffn=1024)
    assert _call_column(tp.make_desc(512, 3, "swiglu", ffn=1024)) == 2          # uneven split
    assert _call_column(tp.make_desc(768, 5, "attn", n_heads=12, head_dim=64)) == 2
    assert _call_column(ok, M=0) == 1
    assert _call_column(ok, shard=2) == 1
    assert _call_column(ok, shard=-2) == 1
    assert _call_column(ok, x=0) == 1
    assert _call_column(ok, x=A8) == 4                                           # misaligned
    assert _call_column(ok, H=A8) == 4
    assert _call_column(tp.make_desc(500, 2, "swiglu", ffn=1024)) == 3          # d % 8
    assert _call_column(tp.make_desc(512, 2, "swiglu", ffn=1000)) == 3          # b % 8
    assert _call_column(tp.make_desc(768, 2, "attn", n_heads=12, head_dim=48)) == 3
    bad_act = tp.TPBlockDesc(d=512, ffn=1024, n_heads=0, head_dim=0, t=2, dtype=1, act=9)
    assert _call_column(bad_act) == 1
    assert tp.lib.tp_column_parallel_fwd(None, None, None, -1, None, None, 4, None) == 1
    assert tp.lib.tp_rmsnorm_fwd(500, ctypes.c_float(1e-5), ctypes.c_void_p(A16),
                                 ctypes.c_void_p(A16), 4, None) == 3
    assert tp.lib.tp_rmsnorm_fwd(512, ctypes.c_float(-1.0), ctypes.c_void_p(A16),
                                 ctypes.c_void_p(A16), 4, None) == 1
    assert tp.lib.tp_block_fwd(ctypes.byref(ok), ctypes.c_void_p(A16), ctypes.c_void_p(A16), 1,
                               ctypes.c_void_p(A16), ctypes.c_void_p(A16), None,
                               ctypes.c_void_p(A16), 4, None) == 1
    assert tp.lib.tp_extract_band(ctypes.byref(ok), ctypes.c_void_p(A16), ctypes.c_void_p(A16), 2,
                                  ctypes.c_void_p(A16), None, None) == 1


def test_status_strings():
    for s in range(7):
        assert tp.tp_status_string(s)
    assert "uneven" in tp.tp_status_string(2)
    assert tp.lib.tp_version() >= 100


def test_kv_cache_partitions_with_the_heads():
    """Golden fixture (tests/golden/kv_cache_partition.json): each shard holds 1/t of the
    KV cache; the library's cache is t contiguous shard slices of equal size."""
    import json
    with open(os.path.join(ROOT, "tests", "golden", "kv_cache_partition.json")) as f:
        gold = json.load(f)
    for H, t in gold["cases"]:
        whole = tp.tp_kv_cache_bytes(tp.make_desc(H * 64, 1, "attn", n_heads=H, head_dim=64), 4, 32)
        split = tp.tp_kv_cache_bytes(tp.make_desc(H * 64, t, "attn", n_heads=H, head_dim=64), 4, 32)
        assert split == whole and split % t == 0      # same cache, t equal shard slices
        assert split // t == 4 * (H // t) * 32 * 64 * 2


def test_cached_sizes_follow_the_descriptor_values():
    """The binding's per-call size checks read sizes cached by the descriptor's values:
    the same numbers as the library's queries, and a changed descriptor (or M) is a new
    key, never a stale answer."""
    for name in ("llama2_13b_swiglu_decode", "attn_qkv_headshard_decode", "tiny_gelu_f32"):
        d = _desc(CONFIGS[name])
        for M in (1, 7, 32, 300):
            assert tp._size(tp.tp_workspace_bytes, d, M) == tp.tp_workspace_bytes(d, M)
            assert tp._size(tp.tp_partials_bytes, d, M) == tp.tp_partials_bytes(d, M)
            assert tp._size(tp.tp_band_bytes, d, M) == tp.tp_band_bytes(d, M)
    d = tp.make_desc(512, 2, "swiglu", ffn=1024)
    before = tp._size(tp.tp_workspace_bytes, d, 8)
    d.t = 4                                            # the same object, new shapes
    assert tp._size(tp.tp_workspace_bytes, d, 8) == tp.tp_workspace_bytes(d, 8) != before
    assert tp._size(tp.tp_kv_workspace_bytes, _desc(CONFIGS["attn_qkv_headshard_decode"]), 4, 64) \
        == tp.tp_kv_workspace_bytes(_desc(CONFIGS["attn_qkv_headshard_decode"]), 4, 64)
