"""ctypes view of libhb.so (include/hb.h). Marshalling only."""

from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libhb.so")

c_int32 = ctypes.c_int32
c_int64 = ctypes.c_int64
c_size_t = ctypes.c_size_t
c_void_p = ctypes.c_void_p

HB_OK = 0
STATUS_NAMES = {
    0: "HB_OK",
    1: "HB_ERR_INVALID_ARG",
    2: "HB_ERR_UNSUPPORTED_SHAPE",
    3: "HB_ERR_MISALIGNED",
    4: "HB_ERR_CUDA",
    5: "HB_ERR_DEVICE_BOUNDS",
    6: "HB_ERR_TIMEOUT",
    7: "HB_ERR_WORKSPACE",
}


class HBConfig(ctypes.Structure):
    """Mirror of ``hb_config``."""

    _fields_ = [
        ("num_heads", c_int32),
        ("head_dim", c_int32),
        ("feat_half", c_int32),
        ("block_len", c_int32),
        ("dtype", c_int32),
        ("merge", c_int32),
        ("scale", ctypes.c_float),
    ]


_P = ctypes.POINTER(HBConfig)

# name -> (restype, argtypes), in the order of include/hb.h
SIGNATURES = {
    "hb_feature_map": (c_int32, [_P, c_int64, c_void_p, c_void_p, c_void_p, c_void_p]),
    "hb_block_attend": (c_int32, [_P, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_void_p]),
    "hb_block_attend_commit": (c_int32, [_P, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_int32, c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_void_p]),
    "hb_block_attend_commit_layers": (c_int32, [_P, c_int32, c_int32, c_void_p, c_void_p,
                                                c_void_p, c_void_p, c_void_p, c_void_p,
                                                c_int32, c_void_p, c_void_p, c_void_p,
                                                c_void_p, c_void_p]),
    "hb_block_attend_commit_s16": (c_int32, [_P, c_int32, c_void_p, c_void_p, c_void_p,
                                             c_void_p, c_void_p, c_void_p, c_void_p, c_int32,
                                             c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "hb_prefill_attend": (c_int32, [_P, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_int64,
                                    c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_int32,
                                    c_void_p, c_void_p]),
    "hb_block_attend_ex": (c_int32, [_P, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_void_p, c_void_p]),
    "hb_prefill_attend_ex": (c_int32, [_P, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_int64, c_void_p, c_void_p, c_int32, c_void_p,
                                       c_void_p, c_void_p, c_int32, c_void_p, c_void_p]),
    "hb_commit_block": (c_int32, [_P, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_int32, c_void_p]),
    "hb_prefill_state": (c_int32, [_P, c_int32, c_void_p, c_void_p, c_void_p, c_int64, c_void_p,
                                   c_int64,
                                   c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_void_p,
                                   c_size_t, c_void_p]),
    "hb_prefill_workspace_size": (c_size_t, [_P, c_int32, c_int64]),
    "hb_prefill_state_noalloc": (c_int32, [_P, c_int32, c_void_p, c_void_p, c_void_p, c_int64,
                                           c_void_p, c_int64, c_void_p, c_void_p, c_void_p,
                                           c_int32, c_int32, c_void_p]),
    "hb_state_zero": (c_int32, [_P, c_int32, c_void_p, c_void_p, c_void_p, c_int32, c_void_p]),
    "hb_state_to_bf16": (c_int32, [_P, c_int32, c_void_p, c_void_p, c_void_p, c_int32,
                                   c_void_p]),
    "hb_state_to_fp8": (c_int32, [_P, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_int32, c_void_p]),
    "hb_block_attend_s8": (c_int32, [_P, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_void_p,
                                     c_void_p, c_void_p]),
    "hb_block_attend_s16": (c_int32, [_P, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                                      c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_void_p,
                                      c_void_p]),
    "hb_state_copy": (c_int32, [_P, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_int32,
                                c_void_p]),
    "hb_softmax_kv_attend": (c_int32, [_P, c_int32, c_void_p, c_void_p, c_int64, c_void_p, c_int64,
                                       c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                       c_void_p]),
    "hb_softmax_kv_workspace_size": (c_size_t, [_P, c_int32, c_int64]),
    "hb_softmax_kv_attend_paged": (c_int32, [_P, c_int32, c_void_p, c_void_p, c_int64, c_int32,
                                             c_void_p, c_int32, c_void_p, c_int64, c_void_p,
                                             c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                             c_void_p]),
    "hb_set_wait_limit": (c_int32, [ctypes.c_uint64]),
    "hb_get_device_status": (c_int32, [c_void_p]),
    "hb_status_string": (ctypes.c_char_p, [c_int32]),
}

_lock = threading.Lock()
_lib = None


def load():
    """Loads libhb.so; raises if it has not been built (there is no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -m linear_attention_diffusion_feature_b300.build)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib
