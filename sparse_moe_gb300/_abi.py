"""ctypes declarations for include/sparse_moe.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os

from . import build as _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_NOT_LOADED = 5
MOE_ERR_DEVICE_TIMEOUT = 6
MOE_ERR_RANGE = 7

MOE_W_BF16 = 0
MOE_W_INT4_SYM_G64 = 1
MOE_W_INT4_AFFINE_G64 = 2

# Every function the header declares, with its C signature.
vp = ctypes.c_void_p
i32 = ctypes.c_int
i64 = ctypes.c_int64


class MoeConfig(ctypes.Structure):
    _fields_ = [("hidden", i32), ("n_experts", i32), ("top_k", i32), ("inter", i32),
                ("shared_inter", i32), ("n_layers", i32), ("max_chunk_rows", i32),
                ("wfmt", i32)]


class MoeWeights(ctypes.Structure):
    _fields_ = [("router_w", vp), ("router_b", vp), ("gate_up", vp), ("gate_up_scale", vp),
                ("down", vp), ("down_scale", vp), ("sh_gate_up", vp), ("sh_gate_up_scale", vp),
                ("sh_down", vp), ("sh_down_scale", vp), ("sh_gate_w", vp),
                ("down_f16", vp), ("sh_down_f16", vp),
                ("gate_up_bias", vp), ("down_bias", vp), ("sh_gate_up_bias", vp),
                ("sh_down_bias", vp)]


class MoeKernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", i64), ("total_ms", ctypes.c_double)]


SIGNATURES = {
    "moe_workspace_size": (i32, [ctypes.POINTER(MoeConfig), ctypes.POINTER(ctypes.c_size_t)]),
    "moe_ctx_create": (i32, [ctypes.POINTER(MoeConfig), i32, vp, ctypes.c_size_t,
                             ctypes.POINTER(vp)]),
    "moe_ctx_destroy": (i32, [vp]),
    "moe_load_weights": (i32, [vp, i32, ctypes.POINTER(MoeWeights)]),
    "moe_route": (i32, [vp, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]),
    "moe_forward_prefill": (i32, [vp, i32, vp, i32, vp, vp]),
    "moe_forward_decode": (i32, [vp, i32, vp, vp, vp]),
    "moe_forward_decode_layers": (i32, [vp, i32, i32, vp, ctypes.c_size_t, vp, ctypes.c_size_t,
                                        vp]),
    "moe_decode_routing": (i32, [vp, vp, vp, vp, vp]),
    "moe_forward_rows": (i32, [vp, i32, vp, i32, vp, vp]),
    "moe_rows_routing": (i32, [vp, vp, vp, vp, vp]),
    "moe_forward_prefill_host": (i32, [vp, i32, vp, i32, vp, vp]),
    "moe_forward_decode_host": (i32, [vp, i32, vp, vp, vp]),
    "moe_forward_decode_noalloc": (i32, [ctypes.POINTER(MoeConfig), ctypes.POINTER(MoeWeights), vp,
                                         vp, vp]),
    "moe_convert_bf16_to_f16": (i32, [vp, vp, ctypes.c_size_t, vp]),
    "moe_dequant_int4": (i32, [vp, vp, vp, vp, ctypes.c_size_t, i32, i32, i32, vp]),
    "moe_check_device": (i32, [vp, ctypes.POINTER(ctypes.c_int32)]),
    "moe_profile_enable": (i32, [vp, i32]),
    "moe_profile_read": (i32, [vp, ctypes.POINTER(MoeKernelStat), i32, ctypes.POINTER(i32)]),
    "moe_decode_phase_read": (i32, [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]),
    "moe_launch_count": (i64, [vp]),
    "moe_last_error": (ctypes.c_char_p, [vp]),
    "moe_status_string": (ctypes.c_char_p, [i32]),
}

_lib = None


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Loads the in-tree library (building it first if it is missing or stale).
    Raises if it cannot be built or loaded: there is no fallback path."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB_PATH
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(path):
        raise ImportError(f"sparse_moe_gb300: native library missing at {path}")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
