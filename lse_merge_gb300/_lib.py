"""ctypes view of libskv.so (include/skv.h).  Argument marshalling only."""
from __future__ import annotations

import ctypes
import os
from ctypes import c_float, c_int, c_int32, c_int64, c_size_t, c_void_p

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libskv.so")

SKV_OK, SKV_ERR_INVALID_ARG, SKV_ERR_UNSUPPORTED, SKV_ERR_CUDA, SKV_ERR_TIMEOUT, SKV_ERR_BAD_ANCHORS, \
    SKV_ERR_WORKSPACE = range(7)
SKV_FP32, SKV_BF16 = 0, 1

# every symbol include/skv.h declares, with (restype, argtypes)
SIGNATURES = {
    "skv_chunk_costs": (c_int, [c_void_p, c_void_p, c_void_p]),
    "skv_lpt_order": (c_int, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p]),
    "skv_contiguous_order": (c_int, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p]),
    "skv_zigzag_loads": (c_int, [c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_void_p]),
    "skv_workspace_bytes": (c_size_t, [c_void_p, c_int]),
    "skv_attn_fwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                             c_size_t, c_void_p]),
    "skv_lse_merge": (c_int, [c_void_p, c_void_p, c_int32, c_int64, c_int32, c_void_p, c_int, c_void_p, c_void_p]),
    "skv_lse_merge_bwd": (c_int, [c_void_p, c_void_p, c_int32, c_int64, c_int32, c_void_p, c_int, c_void_p, c_void_p,
                                  c_void_p, c_void_p]),
    "skv_lse_merge_oproj": (c_int, [c_void_p, c_void_p, c_int32, c_int64, c_int32, c_int32, c_void_p, c_int32,
                                    c_void_p, c_void_p, c_void_p, c_void_p]),
    "skv_attn_bwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                             c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "skv_stream_status": (c_int, [c_void_p]),
    "skv_status_str": (ctypes.c_char_p, [c_int]),
    "skv_set_wait_limit": (c_int, [c_int64]),
    "skv_launch_count": (ctypes.c_uint64, []),
    "skv_set_kernel_timing": (c_int, [c_int]),
    "skv_kernel_times": (c_int, [c_void_p, c_int]),
    "skv_attn_fwd_static": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_void_p]),
    "skv_block_local_fwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "skv_block_local_bwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_void_p, c_void_p, c_void_p, c_void_p]),
}


class SkvProblem(ctypes.Structure):
    """Mirror of struct skv_problem."""
    _fields_ = [
        ("B", c_int32), ("n_blocks", c_int32), ("n_heads", c_int32), ("head_dim", c_int32),
        ("S", c_int64), ("m", c_int32), ("P", c_int32), ("J", c_int32),
        ("s", c_void_p), ("a", c_void_p), ("dtype", c_int), ("scale", c_float), ("n_kv_heads", c_int32),
    ]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libskv.so; raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libskv.so is not built ({path}); run `python -m lse_merge_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
