"""ctypes loader for libmf.so (the C ABI in include/mf.h).

There is no fallback: if the CUDA library cannot be built or loaded, every call
raises.  Nothing here computes; it only declares the C signatures.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

STATUS_NAMES = {
    0: "MF_OK",
    1: "MF_ERR_INVALID_ARG",
    2: "MF_ERR_UNSUPPORTED",
    3: "MF_ERR_OVERFLOW",
    4: "MF_ERR_CUDA",
    5: "MF_ERR_TIMEOUT",
    6: "MF_ERR_BAD_SEQLENS",
}

# every function the header declares, with (restype, argtypes)
_p, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "mf_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "mf_version": (_i32, []),
    "mf_pack_size": (ctypes.c_int, [_p, _i32, _p, _p]),
    "mf_pack": (ctypes.c_int, [_p, _i32, _p, _p, _p]),
    "mf_rope2d_qk": (ctypes.c_int, [_p, _p, _p, _p, _p, _i32, _i32, _i32, _p]),
    "mf_attn_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "mf_attn_workspace_bytes_ds": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "mf_varlen_attn_fwd": (ctypes.c_int, [_p, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _i32, _f32,
                                          _p, _p, _p, _sz, _p]),
    "mf_varlen_attn_fwd_fused_rope": (ctypes.c_int, [_p, _p, _p, _p, _p, _i32, _i32, _i32, _i32,
                                                     _i32, _f32, _p, _p, _p, _sz, _p]),
    "mf_varlen_attn_bwd": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _p, _p, _i32, _i32, _i32, _i32,
                                          _i32, _f32, _p, _p, _p, _p, _sz, _p]),
    "mf_varlen_attn_bwd_after_fwd": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _p, _p, _i32, _i32,
                                                    _i32, _i32, _i32, _i32, _f32, _p, _p, _p, _p,
                                                    _sz, _p]),
    "mf_varlen_attn_fwd_fp8": (ctypes.c_int, [_p, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _i32,
                                              _i32, _f32, _p, _p, _p, _sz, _p]),
    "mf_quant_e4m3": (ctypes.c_int, [_p, _p, _p, _p, _i32, _i32, _i32, _i32, _p, _p, _p, _p, _p,
                                     _p]),
    "mf_varlen_attn_fwd_noalloc": (ctypes.c_int, [_p, _p, _p, _p, _p, _i32, _i32, _i32, _i32,
                                                  _i32, _f32, _p, _p, _p]),
    "mf_noalloc_get_status": (ctypes.c_int, [_p]),
    "mf_pack3d_size": (ctypes.c_int, [_p, _i32, _p, _p]),
    "mf_pack3d": (ctypes.c_int, [_p, _i32, _p, _p, _p]),
    "mf_rope3d_qk": (ctypes.c_int, [_p, _p, _p, _p, _p, _i32, _i32, _i32, _p]),
    "mf_varlen_attn_fwd_3d": (ctypes.c_int, [_p, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _i32,
                                             _f32, _p, _p, _p, _sz, _p]),
    "mf_varlen_attn_bwd_3d": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _p, _p, _i32, _i32, _i32,
                                             _i32, _i32, _f32, _p, _p, _p, _p, _sz, _p]),
    "mf_cfg_euler_step": (ctypes.c_int, [_p, _p, _i32, _i32, _f32, _f32, _p, _p]),
    "mf_adaln_modulate": (ctypes.c_int, [_p, _p, _i32, _i32, _i32, _p, _p, _f32, _p, _p]),
    "mf_gated_residual": (ctypes.c_int, [_p, _p, _p, _i32, _i32, _i32, _p, _p, _p]),
    "mf_get_status": (ctypes.c_int, [_p, _p]),
    "mf_test_varlen_attn_fwd_stalled": (ctypes.c_int, [_p, _p, _p, _p, _p, _i32, _i32, _i32,
                                                       _i32, _i32, _f32, _p, _p, _p, _sz, _i32,
                                                       _p]),
    "mf_test_varlen_attn_bwd_stalled": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _p, _p, _i32,
                                                       _i32, _i32, _i32, _i32, _f32, _p, _p, _p,
                                                       _p, _sz, _i32, _p]),
    "mf_timing_enable": (ctypes.c_int, [_i32]),
    "mf_timing_reset": (ctypes.c_int, []),
    "mf_timing_read": (ctypes.c_int, [_i32, _p, _p]),
}

# kernel ids of the opt-in timing (mf.h MF_K_*)
KERNELS = ["pack", "rope", "schedule", "attn_fwd", "bwd_pre", "attn_bwd", "attn_bwd_q", "cfg_euler",
           "adaln", "gated_residual", "f8_amax", "f8_quant", "attn_fwd_f8", "rope_table",
           "attn_fwd_rot", "attn_bwd_dq"]


class MFError(RuntimeError):
    def __init__(self, what: str, status: int):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")
        self.status = status


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_stale: bool = True):
    """Load libmf.so, rebuilding it first if a source is newer (nvcc must exist)."""
    global _lib
    if _lib is None:
        if build_if_stale and not _build.up_to_date():
            _build.build()
        if not os.path.exists(_build.LIB):
            raise MFError(f"CUDA library missing at {_build.LIB}", 4)
        lib = ctypes.CDLL(_build.LIB)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def check(status: int, what: str) -> None:
    if status != 0:
        raise MFError(what, status)
