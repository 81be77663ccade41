"""ctypes declarations of the C interface in include/attn.h.

Loading fails loudly when the shared library has not been built: there is no
fallback implementation.
"""

import ctypes
import os

from .build import LIB_PATH

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4
ATTN_ERR_WORKSPACE = 5

ATTN_BF16 = 0
ATTN_FP32 = 1
ATTN_FP8_E4M3 = 2

ATTN_STALL_NONE = 0
ATTN_STALL_FWD_SOFTMAX = 1
ATTN_STALL_BWD_COMPUTE = 2

# every function the header declares, with its ctypes signature
EXPORTS = {
    "attn_workspace_size": (ctypes.c_size_t, [ctypes.c_void_p, ctypes.c_int]),
    "attn_fwd": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_size_t, ctypes.c_void_p]),
    "attn_bwd": (ctypes.c_int, [ctypes.c_void_p] * 11 + [ctypes.c_size_t, ctypes.c_void_p]),
    "attn_bwd_preprocess": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_size_t, ctypes.c_void_p]),
    "attn_bwd_main": (ctypes.c_int, [ctypes.c_void_p] * 8 + [ctypes.c_size_t, ctypes.c_void_p]),
    "attn_bwd_dq": (ctypes.c_int, [ctypes.c_void_p] * 3 + [ctypes.c_size_t, ctypes.c_void_p]),
    "attn_bwd_noalloc": (ctypes.c_int, [ctypes.c_void_p] * 11),
    "attn_decode_workspace_size": (ctypes.c_size_t, [ctypes.c_void_p, ctypes.c_int32]),
    "attn_decode": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32] + [ctypes.c_void_p] * 6
                    + [ctypes.c_size_t, ctypes.c_void_p]),
    "attn_selftest_timeout": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p]),
    "attn_debug_stall": (ctypes.c_int, [ctypes.c_int32, ctypes.c_uint64]),
    "attn_check": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "attn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "attn_last_error": (ctypes.c_char_p, []),
}


class AttnParams(ctypes.Structure):
    """Mirror of `attn_params`."""

    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("N", ctypes.c_int32),
        ("d", ctypes.c_int32), ("dtype", ctypes.c_int32), ("scale", ctypes.c_float),
        ("causal", ctypes.c_int32), ("dropout_p", ctypes.c_float),
        ("philox_seed", ctypes.c_uint64), ("philox_offset", ctypes.c_uint64),
        ("key_lens", ctypes.c_void_p), ("block_mask", ctypes.c_void_p),
        ("block_mask_head_stride", ctypes.c_int64),
        ("stride_b", ctypes.c_int64), ("stride_h", ctypes.c_int64),
        ("stride_n", ctypes.c_int64),
        ("H_kv", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("kv_stride_b", ctypes.c_int64), ("kv_stride_h", ctypes.c_int64),
        ("kv_stride_n", ctypes.c_int64),
        ("q_descale", ctypes.c_float), ("k_descale", ctypes.c_float),
        ("v_descale", ctypes.c_float), ("reserved2", ctypes.c_int32),
    ]


class AttnError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{message} (status {status})")
        self.status = status


_lib = None


def lib():
    """The loaded shared library; raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"CUDA library {LIB_PATH} is not built; run "
                "`python -m exact_attention_12_gb300.build` (needs nvcc)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def check_status(status, what):
    if status != ATTN_OK:
        detail = lib().attn_last_error().decode(errors="replace")
        raise AttnError(status, f"{what}: {detail}")
