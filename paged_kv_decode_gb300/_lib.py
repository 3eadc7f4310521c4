"""ctypes declarations of libpkv's C ABI (include/pkv.h). No computation here."""
from __future__ import annotations

import ctypes
import os
import re
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "pkv.h")

_lock = threading.Lock()
_lib = None


class CacheDesc(ctypes.Structure):
    _fields_ = [
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
    ]


_vp, _i32, _sz, _f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
_dp = ctypes.POINTER(CacheDesc)

# name -> (restype, argtypes), in the order of include/pkv.h
PROTOTYPES = {
    "pkv_workspace_init": (ctypes.c_int, [_vp, _sz, _vp]),
    "pkv_read_status": (ctypes.c_int, [_vp, _vp]),
    "pkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pkv_append": (ctypes.c_int, [_vp, _vp, _vp, _i32, _vp, _vp, _dp, _vp, _vp, _sz]),
    "pkv_decode_workspace_bytes": (_sz, [_dp, _i32, _i32]),
    "pkv_decode_attn": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _f32, _vp, _dp, _i32, _i32, _vp, _sz]),
    "pkv_decode_append_attn": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _f32, _vp, _dp, _i32, _i32,
                                              _vp, _sz, ctypes.c_uint32]),
    "pkv_decode_append_rope_attn": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _f32, _vp, _dp,
                                                   _i32, _i32, _vp, _sz, ctypes.c_uint32]),
    "pkv_rope_table": (ctypes.c_int, [_vp, _i32, _i32, ctypes.c_double, _vp]),
    "pkv_prefill_workspace_bytes": (_sz, [_dp, _i32, _i32]),
    "pkv_prefill_chunk_attn": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _f32, _vp, _dp, _i32,
                                              _i32, _vp, _sz]),
    "pkv_mixed_workspace_bytes": (_sz, [_dp, _i32, _i32, _i32, _i32]),
    "pkv_mixed_step_attn": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _i32, _i32, _vp, _vp, _vp,
                                           _vp, _i32, _i32, _f32, _vp, _dp, _vp, _sz]),
    "pkv_decode_attn_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _f32, _vp, _dp, _i32, _i32]),
    "pkv_selftest_wait_timeout": (ctypes.c_int, [_vp, _sz, ctypes.c_int64, _vp]),
}


def header_functions(path: str = HEADER):
    """Names of the functions include/pkv.h declares."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"\b(pkv_\w+)\s*\(", text)


def load():
    """Load libpkv.so (built by paged_kv_decode_gb300.build). Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libpkv.so not found at {LIB_PATH}; build it with "
                    "`python -m paged_kv_decode_gb300.build` (needs nvcc). There is no CPU fallback."
                )
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in PROTOTYPES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib
