"""ctypes declarations of the C ABI in include/usp.h (loading only)."""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libusp.so")

_c = ctypes
_vp, _i, _f, _sz, _u = _c.c_void_p, _c.c_int, _c.c_float, _c.c_size_t, _c.c_uint
_i64, _u64 = _c.c_int64, _c.c_uint64

SIGNATURES = {
    "usp_attn_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i,
                          _i, _i, _vp, _i, _i, _i, _i, _u, _vp, _sz, _vp]),
    "usp_attn_fwd_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i, _u]),
    "usp_attn_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i,
                          _i, _i, _i, _f, _i, _i, _i, _vp, _i, _i, _i, _i, _u,
                          _vp, _sz, _vp]),
    "usp_attn_bwd_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i, _u]),
    "usp_attn_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i,
                                  _i, _i, _i, _i, _f, _i, _i, _i, _vp, _i, _i, _i,
                                  _i, _u, _vp]),
    "usp_merge_partials": (_i, [_vp, _vp, _i, _i64, _i, _i, _vp, _i, _vp, _vp]),
    "usp_attn_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i,
                             _i, _i, _i, _vp, _sz, _vp]),
    "usp_attn_decode_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "usp_selftest_wait_timeout": (_i, [_u, _vp]),
    "usp_attn_fwd_qkvpacked": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _i, _vp, _i,
                                    _i, _i, _i, _u, _vp, _sz, _vp]),
    "usp_attn_bwd_qkvpacked": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _i,
                                    _vp, _i, _i, _i, _i, _u, _vp, _sz, _vp]),
    "usp_attn_fwd_fp8": (_i, [_vp, _vp, _vp, _f, _f, _f, _vp, _vp, _i, _i, _i, _i, _i, _f,
                              _i, _i, _i, _vp, _i, _i, _i, _u, _vp, _sz, _vp]),
    "usp_attn_fwd_fp8_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i]),
    "usp_quantize_e4m3": (_i, [_vp, _vp, _i64, _f, _vp]),
    "usp_permute": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _vp]),
    "usp_status_string": (_c.c_char_p, [_i]),
    "usp_launch_count": (_u64, []),
    "usp_profile_enable": (_i, [_i]),
    "usp_profile_read": (_i, [_vp, _i]),
    "usp_device_status": (_i, []),
    "usp_last_error_detail": (_c.c_char_p, []),
    "usp_check_cu_seqlens": (_i, [_vp, _i, _i]),
}


class KernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_uint64),
                ("total_ms", ctypes.c_double)]

_lib = None


def load(path: str = LIB_PATH):
    """Load libusp.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -m sequence_long_context_gb300.build)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def exported_symbols():
    return sorted(SIGNATURES)
