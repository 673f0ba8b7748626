"""ctypes binding of libkdkl.so: the C entry points under their own names.

Argument marshalling only (integers for device pointers and the stream); every
step of the path runs in the library's kernels.  Loading fails loudly when the
library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
# KD_DEBUG=1 in the environment selects the checked build (see build.build_library(debug=True))
LIB_PATH = os.path.join(_HERE, "libkdkl_debug.so" if os.environ.get("KD_DEBUG") == "1" else "libkdkl.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "kdkl.h")

KD_OK = 0
KD_ERR_INVALID_ARG = 1
KD_ERR_UNSUPPORTED = 2
KD_ERR_WORKSPACE = 3
KD_ERR_CUDA = 4
KD_ERR_TIMEOUT = 5
KD_ERR_DEVICE = 6
KD_ERR_IO = 7
KD_MAX_K = 1024
KD_STATIC_SCRATCH_BYTES = 32 * 1024 * 1024

_c_i64 = ctypes.c_int64
_c_ptr = ctypes.c_void_p
_c_int = ctypes.c_int
_c_size = ctypes.c_size_t
_c_float = ctypes.c_float

_SIGNATURES = {
    "kd_status_string": (ctypes.c_char_p, [_c_int]),
    "kd_version": (_c_int, []),
    "kd_topk_cache_workspace": (_c_size, [_c_i64, _c_i64, _c_int]),
    "kd_topk_cache": (_c_int, [_c_ptr, _c_i64, _c_i64, _c_i64, _c_int, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                               _c_size, _c_ptr]),
    "kd_teacher_topk_workspace": (_c_size, [_c_i64, _c_i64, _c_i64, _c_int, _c_i64]),
    "kd_teacher_topk": (_c_int, [_c_ptr, _c_ptr, _c_i64, _c_i64, _c_i64, _c_int, _c_i64, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                 _c_ptr, _c_size, _c_ptr]),
    "kd_fused_kl_workspace": (_c_size, [_c_i64, _c_i64, _c_i64, _c_int, _c_i64]),
    "kd_fused_kl_fwd": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_i64, _c_int, _c_i64,
                                 _c_float, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_size, _c_ptr]),
    "kd_fused_kl_bwd": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_i64, _c_int, _c_i64,
                                 _c_float, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_size, _c_ptr]),
    "kd_chunked_kl_logits_bytes": (_c_size, [_c_i64, _c_i64]),
    "kd_chunked_kl_fwd": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_i64, _c_int, _c_i64,
                                   _c_float, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_size, _c_ptr, _c_size, _c_ptr]),
    "kd_chunked_kl_bwd": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_i64, _c_int, _c_i64,
                                   _c_float, _c_ptr, _c_ptr, _c_ptr, _c_size, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_size,
                                   _c_ptr]),
    "kd_fused_kl_fwd_static": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_i64, _c_int,
                                        _c_i64, _c_float, _c_ptr, _c_ptr, _c_ptr, _c_ptr]),
    "kd_get_device_error": (_c_int, [_c_ptr, _c_ptr, ctypes.POINTER(_c_i64)]),
    "kd_gemm_bf16": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_i64, _c_int, _c_int, _c_int, _c_ptr, _c_size,
                              _c_ptr]),
    "kd_gemm_workspace": (_c_size, []),
    "kd_check_wait_timeout": (_c_int, [_c_ptr, _c_size, _c_i64, _c_ptr]),
    "kd_cache_write": (_c_int, [ctypes.c_char_p, _c_ptr, _c_ptr, _c_ptr, _c_i64, _c_int, _c_i64, _c_i64, _c_int]),
    "kd_cache_info": (_c_int, [ctypes.c_char_p, ctypes.POINTER(_c_i64), ctypes.POINTER(_c_int),
                               ctypes.POINTER(_c_i64), ctypes.POINTER(_c_i64), ctypes.POINTER(_c_int),
                               ctypes.POINTER(_c_int)]),
    "kd_cache_verify": (_c_int, [ctypes.c_char_p]),
    "kd_cache_read": (_c_int, [ctypes.c_char_p, _c_i64, _c_i64, _c_ptr, _c_ptr, _c_ptr]),
    "kd_cache_reader_open": (_c_int, [ctypes.c_char_p, _c_i64, ctypes.POINTER(_c_ptr)]),
    "kd_cache_reader_next": (_c_int, [_c_ptr, _c_ptr, _c_ptr, ctypes.POINTER(_c_i64)]),
    "kd_cache_reader_close": (_c_int, [_c_ptr]),
    "kd_profile_begin": (_c_int, [_c_int]),
    "kd_profile_end": (_c_int, []),
    "kd_profile_read": (_c_int, [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(_c_float), _c_int]),
}

_lib = None


class KDError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def load():
    """Load libkdkl.so and attach argument/return types; raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{os.path.basename(LIB_PATH)} not built at {LIB_PATH}: run "
                               "sparse_teacher_kl_gb300.build.build_library()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def header_functions():
    """Names of the functions include/kdkl.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^KD_API\s+[\w\s\*]+?\b(kd_\w+)\s*\(", text, flags=re.M)))


def status_string(status: int) -> str:
    return load().kd_status_string(int(status)).decode()


def check(status: int, where: str):
    if status != KD_OK:
        raise KDError(status, where)


def _wrap(name):
    def f(*args):
        return getattr(load(), name)(*args)
    f.__name__ = name
    f.__doc__ = f"{name} from include/kdkl.h (raw status return)."
    return f


kd_status_string = _wrap("kd_status_string")
kd_version = _wrap("kd_version")
kd_topk_cache_workspace = _wrap("kd_topk_cache_workspace")
kd_topk_cache = _wrap("kd_topk_cache")
kd_fused_kl_workspace = _wrap("kd_fused_kl_workspace")
kd_teacher_topk_workspace = _wrap("kd_teacher_topk_workspace")
kd_teacher_topk = _wrap("kd_teacher_topk")
kd_fused_kl_fwd = _wrap("kd_fused_kl_fwd")
kd_fused_kl_bwd = _wrap("kd_fused_kl_bwd")
kd_fused_kl_fwd_static = _wrap("kd_fused_kl_fwd_static")
kd_chunked_kl_logits_bytes = _wrap("kd_chunked_kl_logits_bytes")
kd_chunked_kl_fwd = _wrap("kd_chunked_kl_fwd")
kd_chunked_kl_bwd = _wrap("kd_chunked_kl_bwd")
kd_get_device_error = _wrap("kd_get_device_error")
kd_gemm_bf16 = _wrap("kd_gemm_bf16")
kd_gemm_workspace = _wrap("kd_gemm_workspace")
kd_check_wait_timeout = _wrap("kd_check_wait_timeout")
kd_cache_write = _wrap("kd_cache_write")
kd_cache_info = _wrap("kd_cache_info")
kd_cache_verify = _wrap("kd_cache_verify")
kd_cache_read = _wrap("kd_cache_read")
kd_cache_reader_open = _wrap("kd_cache_reader_open")
kd_cache_reader_next = _wrap("kd_cache_reader_next")
kd_cache_reader_close = _wrap("kd_cache_reader_close")
kd_profile_begin = _wrap("kd_profile_begin")
kd_profile_end = _wrap("kd_profile_end")
kd_profile_read = _wrap("kd_profile_read")
