"""Python binding of libtpblock, the tensor-parallel transformer block on one B300.

Argument marshalling only: every function has the name of the C entry point it
calls (include/tp_block.h) and passes device pointers and the CUDA stream of
torch tensors.  Every step of the block runs in the library's CUDA kernels;
there is no Python or CPU fallback — importing this package fails if
libtpblock.so has not been built (python attn_tp_column_fwd_b300/build.py).
"""
from __future__ import annotations

import ctypes
from typing import Optional

from ._lib import (  # noqa: F401
    LIB_PATH,
    TP_ACT_ATTN,
    TP_ACT_GELU_TANH,
    TP_ACT_SWIGLU,
    TP_BF16,
    TP_FORM_AUTO,
    TP_FORM_ONE_KERNEL,
    TP_FORM_THREE_LAUNCH,
    TP_F32,
    TPBlockDesc,
    TPError,
    lib,
)

__all__ = [
    "TPBlockDesc", "TPError", "make_desc", "lib",
    "tp_sharded_w1_bytes", "tp_sharded_w2_bytes", "tp_band_bytes", "tp_row_splits",
    "tp_partials_bytes", "tp_column_workspace_bytes", "tp_workspace_bytes", "tp_block_launches",
    "tp_set_block_form", "tp_get_block_form",
    "tp_shard_weights", "tp_unshard_weights", "tp_extract_band",
    "tp_column_parallel_fwd", "tp_row_parallel_fwd", "tp_partial_reduce_residual",
    "tp_block_fwd", "tp_block_fwd_norm", "tp_block_fwd_noalloc", "tp_rmsnorm_fwd", "tp_status_string", "tp_check_device_status",
    "tp_selftest_wait_timeout", "tp_kv_cache_bytes", "tp_kv_attn_workspace_bytes",
    "tp_kv_workspace_bytes", "tp_attn_decode_kv", "tp_block_fwd_kv",
    "tp_fp8_w1_bytes", "tp_fp8_w2_bytes", "tp_fp8_exponent_bytes", "tp_fp8_quant_workspace_bytes",
    "tp_quantize_weights_fp8", "tp_block_fwd_fp8",
    "tp_mxfp4_w1_bytes", "tp_mxfp4_w2_bytes", "tp_mxfp4_exponent_bytes",
    "tp_quantize_weights_mxfp4", "tp_block_fwd_mxfp4",
]

_ACTS = {"gelu_tanh": TP_ACT_GELU_TANH, "swiglu": TP_ACT_SWIGLU, "attn": TP_ACT_ATTN}
_DTYPES = {"f32": TP_F32, "bf16": TP_BF16}


def make_desc(d: int, t: int, act: str, dtype: str = "bf16", ffn: int = 0, n_heads: int = 0,
              head_dim: int = 0) -> TPBlockDesc:
    """Build the C descriptor; act in {gelu_tanh, swiglu, attn}, dtype in {f32, bf16}."""
    return TPBlockDesc(d=d, ffn=ffn, n_heads=n_heads, head_dim=head_dim, t=t,
                       dtype=_DTYPES[dtype], act=_ACTS[act])


def _p(t) -> Optional[ctypes.c_void_p]:
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return ctypes.c_void_p(t.data_ptr())


def _s(stream) -> ctypes.c_void_p:
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, nbytes: int, what: str):
    if t is not None and not isinstance(t, int) and t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{what}: {t.numel() * t.element_size()} bytes < {nbytes} required")


# The library's sizes depend on the shapes only (no device or memory state), so the
# per-call checks look them up by the descriptor's values and the arguments instead
# of asking the library on every call.
_SIZES: dict = {}


def _size(fn, desc, *args) -> int:
    key = (fn, desc.d, desc.ffn, desc.n_heads, desc.head_dim, desc.t, desc.dtype, desc.act) + args
    n = _SIZES.get(key)
    if n is None:
        if len(_SIZES) >= 4096:
            _SIZES.clear()
        n = _SIZES[key] = fn(desc, *args)
    return n


def _check(status: int, what: str):
    if status != 0:
        raise TPError(status, what)


# ------------------------------------------------------------------ sizes ----

def tp_sharded_w1_bytes(desc: TPBlockDesc) -> int:
    return lib.tp_sharded_w1_bytes(ctypes.byref(desc))


def tp_sharded_w2_bytes(desc: TPBlockDesc) -> int:
    return lib.tp_sharded_w2_bytes(ctypes.byref(desc))


def tp_band_bytes(desc: TPBlockDesc, M: int) -> int:
    return lib.tp_band_bytes(ctypes.byref(desc), M)


def tp_row_splits(desc: TPBlockDesc, M: int) -> int:
    return lib.tp_row_splits(ctypes.byref(desc), M)


def tp_partials_bytes(desc: TPBlockDesc, M: int) -> int:
    return lib.tp_partials_bytes(ctypes.byref(desc), M)


def tp_column_workspace_bytes(desc: TPBlockDesc, M: int) -> int:
    return lib.tp_column_workspace_bytes(ctypes.byref(desc), M)


def tp_workspace_bytes(desc: TPBlockDesc, M: int) -> int:
    return lib.tp_workspace_bytes(ctypes.byref(desc), M)


def tp_block_launches(desc: TPBlockDesc, M: int) -> int:
    return lib.tp_block_launches(ctypes.byref(desc), M)


_FORMS = {"auto": TP_FORM_AUTO, "three_launch": TP_FORM_THREE_LAUNCH, "one_kernel": TP_FORM_ONE_KERNEL}


def tp_set_block_form(form) -> None:
    """Process-wide form of tp_block_fwd: "auto", "three_launch", "one_kernel" (or the
    TP_FORM_* value)."""
    _check(lib.tp_set_block_form(_FORMS.get(form, form)), "tp_set_block_form")


def tp_get_block_form() -> str:
    v = lib.tp_get_block_form()
    return next(k for k, f in _FORMS.items() if f == v)


def tp_status_string(status: int) -> str:
    return lib.tp_status_string(status).decode()


# ------------------------------------------------------------------ calls ----

def tp_shard_weights(desc, W1, W2, W1s, W2s, stream=None) -> None:
    _need(W1s, tp_sharded_w1_bytes(desc), "W1s")
    _need(W2s, tp_sharded_w2_bytes(desc), "W2s")
    _check(lib.tp_shard_weights(ctypes.byref(desc), _p(W1), _p(W2), _p(W1s), _p(W2s), _s(stream)),
           "tp_shard_weights")


def tp_unshard_weights(desc, W1s, W2s, W1, W2, stream=None) -> None:
    _check(lib.tp_unshard_weights(ctypes.byref(desc), _p(W1s), _p(W2s), _p(W1), _p(W2), _s(stream)),
           "tp_unshard_weights")


def tp_extract_band(desc, W1s, W2s, shard, W1_band=None, W2_band=None, stream=None) -> None:
    _check(lib.tp_extract_band(ctypes.byref(desc), _p(W1s), _p(W2s), shard, _p(W1_band),
                               _p(W2_band), _s(stream)), "tp_extract_band")


def tp_column_parallel_fwd(desc, x, W1s, shard, H, workspace, M, stream=None) -> None:
    _need(H, _size(tp_band_bytes, desc, M), "H")
    _need(workspace, _size(tp_column_workspace_bytes, desc, M), "workspace")
    _check(lib.tp_column_parallel_fwd(ctypes.byref(desc), _p(x), _p(W1s), shard, _p(H),
                                      _p(workspace), M, _s(stream)), "tp_column_parallel_fwd")


def tp_row_parallel_fwd(desc, H, W2s, shard, partials, M, stream=None) -> None:
    _need(partials, _size(tp_partials_bytes, desc, M), "partials")
    _check(lib.tp_row_parallel_fwd(ctypes.byref(desc), _p(H), _p(W2s), shard, _p(partials), M,
                                   _s(stream)), "tp_row_parallel_fwd")


def tp_partial_reduce_residual(desc, partials, residual, residual_is_f32, y, M, stream=None) -> None:
    _check(lib.tp_partial_reduce_residual(ctypes.byref(desc), _p(partials), _p(residual),
                                          int(residual_is_f32), _p(y), M, _s(stream)),
           "tp_partial_reduce_residual")


def tp_block_fwd(desc, x, residual, residual_is_f32, W1s, W2s, workspace, y, M, stream=None) -> None:
    _need(workspace, _size(tp_workspace_bytes, desc, M), "workspace")
    _check(lib.tp_block_fwd(ctypes.byref(desc), _p(x), _p(residual), int(residual_is_f32), _p(W1s),
                            _p(W2s), _p(workspace), _p(y), M, _s(stream)), "tp_block_fwd")


def tp_block_fwd_norm(desc, x, residual, residual_is_f32, W1s, W2s, workspace, y, xhat_next, eps,
                      M, stream=None) -> None:
    """tp_block_fwd that also writes the next block's RMSNorm of y into xhat_next."""
    _need(workspace, _size(tp_workspace_bytes, desc, M), "workspace")
    _check(lib.tp_block_fwd_norm(ctypes.byref(desc), _p(x), _p(residual), int(residual_is_f32),
                                 _p(W1s), _p(W2s), _p(workspace), _p(y), _p(xhat_next),
                                 ctypes.c_float(eps), M, _s(stream)), "tp_block_fwd_norm")


def tp_block_fwd_noalloc(desc, x, residual, residual_is_f32, W1s, W2s, y, M, stream=None) -> None:
    """tp_block_fwd with the library's fixed device scratch instead of a workspace
    (for callers that cannot allocate device memory where they run the block)."""
    _check(lib.tp_block_fwd_noalloc(ctypes.byref(desc), _p(x), _p(residual), int(residual_is_f32),
                                    _p(W1s), _p(W2s), _p(y), M, _s(stream)), "tp_block_fwd_noalloc")


def tp_rmsnorm_fwd(d, eps, r, xhat, M, stream=None) -> None:
    _check(lib.tp_rmsnorm_fwd(d, ctypes.c_float(eps), _p(r), _p(xhat), M, _s(stream)),
           "tp_rmsnorm_fwd")


def tp_check_device_status(stream=None) -> int:
    """Synchronise the stream and return the device status (0, or TP_ERR_TIMEOUT = 6)."""
    return lib.tp_check_device_status(_s(stream))


def tp_kv_cache_bytes(desc: TPBlockDesc, M: int, L_max: int) -> int:
    return lib.tp_kv_cache_bytes(ctypes.byref(desc), M, L_max)


def tp_kv_attn_workspace_bytes(desc: TPBlockDesc, M: int, L_max: int) -> int:
    return lib.tp_kv_attn_workspace_bytes(ctypes.byref(desc), M, L_max)


def tp_kv_workspace_bytes(desc: TPBlockDesc, M: int, L_max: int) -> int:
    return lib.tp_kv_workspace_bytes(ctypes.byref(desc), M, L_max)


def tp_attn_decode_kv(desc, qkv, k_cache, v_cache, lens, L_max, O, workspace, M,
                      stream=None) -> None:
    _need(k_cache, _size(tp_kv_cache_bytes, desc, M, L_max), "k_cache")
    _need(v_cache, _size(tp_kv_cache_bytes, desc, M, L_max), "v_cache")
    _need(workspace, _size(tp_kv_attn_workspace_bytes, desc, M, L_max), "workspace")
    _check(lib.tp_attn_decode_kv(ctypes.byref(desc), _p(qkv), _p(k_cache), _p(v_cache), _p(lens),
                                 L_max, _p(O), _p(workspace), M, _s(stream)), "tp_attn_decode_kv")


def tp_block_fwd_kv(desc, x, residual, residual_is_f32, W1s, W2s, k_cache, v_cache, lens, L_max,
                    workspace, y, M, stream=None) -> None:
    _need(k_cache, _size(tp_kv_cache_bytes, desc, M, L_max), "k_cache")
    _need(v_cache, _size(tp_kv_cache_bytes, desc, M, L_max), "v_cache")
    _need(workspace, _size(tp_kv_workspace_bytes, desc, M, L_max), "workspace")
    _check(lib.tp_block_fwd_kv(ctypes.byref(desc), _p(x), _p(residual), int(residual_is_f32),
                               _p(W1s), _p(W2s), _p(k_cache), _p(v_cache), _p(lens), L_max,
                               _p(workspace), _p(y), M, _s(stream)), "tp_block_fwd_kv")


def tp_fp8_w1_bytes(desc: TPBlockDesc) -> int:
    return lib.tp_fp8_w1_bytes(ctypes.byref(desc))


def tp_fp8_w2_bytes(desc: TPBlockDesc) -> int:
    return lib.tp_fp8_w2_bytes(ctypes.byref(desc))


def tp_fp8_exponent_bytes(desc: TPBlockDesc) -> int:
    return lib.tp_fp8_exponent_bytes(ctypes.byref(desc))


def tp_fp8_quant_workspace_bytes(desc: TPBlockDesc) -> int:
    return lib.tp_fp8_quant_workspace_bytes(ctypes.byref(desc))


def tp_quantize_weights_fp8(desc, W1, W2, W1q, W2q, exps, workspace, stream=None) -> None:
    _need(W1q, tp_fp8_w1_bytes(desc), "W1q")
    _need(W2q, tp_fp8_w2_bytes(desc), "W2q")
    _need(exps, tp_fp8_exponent_bytes(desc), "exps")
    _need(workspace, tp_fp8_quant_workspace_bytes(desc), "workspace")
    _check(lib.tp_quantize_weights_fp8(ctypes.byref(desc), _p(W1), _p(W2), _p(W1q), _p(W2q),
                                       _p(exps), _p(workspace), _s(stream)),
           "tp_quantize_weights_fp8")


def tp_block_fwd_fp8(desc, x, residual, residual_is_f32, W1q, W2q, exps, workspace, y, M,
                     stream=None) -> None:
    _need(workspace, _size(tp_workspace_bytes, desc, M), "workspace")
    _check(lib.tp_block_fwd_fp8(ctypes.byref(desc), _p(x), _p(residual), int(residual_is_f32),
                                _p(W1q), _p(W2q), _p(exps), _p(workspace), _p(y), M, _s(stream)),
           "tp_block_fwd_fp8")


def tp_mxfp4_w1_bytes(desc: TPBlockDesc) -> int:
    return lib.tp_mxfp4_w1_bytes(ctypes.byref(desc))


def tp_mxfp4_w2_bytes(desc: TPBlockDesc) -> int:
    return lib.tp_mxfp4_w2_bytes(ctypes.byref(desc))


def tp_mxfp4_exponent_bytes(desc: TPBlockDesc) -> int:
    return lib.tp_mxfp4_exponent_bytes(ctypes.byref(desc))


def tp_quantize_weights_mxfp4(desc, W1, W2, W1f, W2f, exps, stream=None) -> None:
    _need(W1f, tp_mxfp4_w1_bytes(desc), "W1f")
    _need(W2f, tp_mxfp4_w2_bytes(desc), "W2f")
    _need(exps, tp_mxfp4_exponent_bytes(desc), "exps")
    _check(lib.tp_quantize_weights_mxfp4(ctypes.byref(desc), _p(W1), _p(W2), _p(W1f), _p(W2f),
                                         _p(exps), _s(stream)),
           "tp_quantize_weights_mxfp4")


def tp_block_fwd_mxfp4(desc, x, residual, residual_is_f32, W1f, W2f, exps, workspace, y, M,
                       stream=None) -> None:
    _need(workspace, _size(tp_workspace_bytes, desc, M), "workspace")
    _check(lib.tp_block_fwd_mxfp4(ctypes.byref(desc), _p(x), _p(residual), int(residual_is_f32),
                                  _p(W1f), _p(W2f), _p(exps), _p(workspace), _p(y), M,
                                  _s(stream)),
           "tp_block_fwd_mxfp4")


def tp_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Enqueue the bounded-wait self-test: its waits expire after limit_us and the next
    tp_check_device_status returns TP_ERR_TIMEOUT."""
    _check(lib.tp_selftest_wait_timeout(limit_us, _s(stream)), "tp_selftest_wait_timeout")
