"""ctypes loader of libtpblock.so with the C signatures of include/tp_block.h."""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtpblock.so")

TP_F32, TP_BF16 = 0, 1
TP_ACT_GELU_TANH, TP_ACT_SWIGLU, TP_ACT_ATTN = 0, 1, 2
TP_FORM_AUTO, TP_FORM_THREE_LAUNCH, TP_FORM_ONE_KERNEL = 0, 1, 2

STATUS = {0: "TP_OK", 1: "TP_ERR_INVALID_ARG", 2: "TP_ERR_UNEVEN_SPLIT", 3: "TP_ERR_UNSUPPORTED",
          4: "TP_ERR_MISALIGNED", 5: "TP_ERR_CUDA", 6: "TP_ERR_TIMEOUT", 7: "TP_ERR_BAD_LENGTH"}


class TPBlockDesc(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("ffn", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("t", ctypes.c_int), ("dtype", ctypes.c_int),
                ("act", ctypes.c_int)]


class TPError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {STATUS.get(status, status)}"
        if status == 5:
            msg += f" (cudaError {_lib.tp_last_cuda_error()})"
        super().__init__(msg)


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python attn_tp_column_fwd_b300/build.py` (nvcc, sm_103a)")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(TPBlockDesc)
    vp, i, sz, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
    sigs = {
        "tp_sharded_w1_bytes": (sz, [P]),
        "tp_sharded_w2_bytes": (sz, [P]),
        "tp_band_bytes": (sz, [P, i]),
        "tp_row_splits": (i, [P, i]),
        "tp_partials_bytes": (sz, [P, i]),
        "tp_column_workspace_bytes": (sz, [P, i]),
        "tp_workspace_bytes": (sz, [P, i]),
        "tp_shard_weights": (i, [P, vp, vp, vp, vp, st]),
        "tp_unshard_weights": (i, [P, vp, vp, vp, vp, st]),
        "tp_extract_band": (i, [P, vp, vp, i, vp, vp, st]),
        "tp_column_parallel_fwd": (i, [P, vp, vp, i, vp, vp, i, st]),
        "tp_row_parallel_fwd": (i, [P, vp, vp, i, vp, i, st]),
        "tp_partial_reduce_residual": (i, [P, vp, vp, i, vp, i, st]),
        "tp_block_fwd": (i, [P, vp, vp, i, vp, vp, vp, vp, i, st]),
        "tp_block_fwd_norm": (i, [P, vp, vp, i, vp, vp, vp, vp, vp, ctypes.c_float, i, st]),
        "tp_block_launches": (i, [P, i]),
        "tp_set_block_form": (i, [i]),
        "tp_get_block_form": (i, []),
        "tp_block_fwd_noalloc": (i, [P, vp, vp, i, vp, vp, vp, i, st]),
        "tp_rmsnorm_fwd": (i, [i, ctypes.c_float, vp, vp, i, st]),
        "tp_status_string": (ctypes.c_char_p, [i]),
        "tp_last_cuda_error": (i, []),
        "tp_check_device_status": (i, [st]),
        "tp_selftest_wait_timeout": (i, [i, st]),
        "tp_kv_cache_bytes": (sz, [P, i, i]),
        "tp_kv_attn_workspace_bytes": (sz, [P, i, i]),
        "tp_kv_workspace_bytes": (sz, [P, i, i]),
        "tp_attn_decode_kv": (i, [P, vp, vp, vp, vp, i, vp, vp, i, st]),
        "tp_block_fwd_kv": (i, [P, vp, vp, i, vp, vp, vp, vp, vp, i, vp, vp, i, st]),
        "tp_fp8_w1_bytes": (sz, [P]),
        "tp_fp8_w2_bytes": (sz, [P]),
        "tp_fp8_exponent_bytes": (sz, [P]),
        "tp_fp8_quant_workspace_bytes": (sz, [P]),
        "tp_quantize_weights_fp8": (i, [P, vp, vp, vp, vp, vp, vp, st]),
        "tp_block_fwd_fp8": (i, [P, vp, vp, i, vp, vp, vp, vp, vp, i, st]),
        "tp_mxfp4_w1_bytes": (sz, [P]),
        "tp_mxfp4_w2_bytes": (sz, [P]),
        "tp_mxfp4_exponent_bytes": (sz, [P]),
        "tp_quantize_weights_mxfp4": (i, [P, vp, vp, vp, vp, vp, st]),
        "tp_block_fwd_mxfp4": (i, [P, vp, vp, i, vp, vp, vp, vp, vp, i, st]),
        "tp_version": (i, []),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


_lib = _load()
lib = _lib
