"""ctypes declarations of liboscar.so's C ABI (argument marshalling only; no computation here)."""
from __future__ import annotations

import ctypes as C
import os
import re

from . import build as _build

c_bf16_p = C.POINTER(C.c_uint16)

STATUS = {0: "OSCAR_OK", 1: "OSCAR_ERR_INVALID_ARG", 2: "OSCAR_ERR_UNSUPPORTED", 3: "OSCAR_ERR_WORKSPACE",
          4: "OSCAR_ERR_CUDA", 5: "OSCAR_ERR_NUMERIC"}


class OscarError(RuntimeError):
    def __init__(self, status: int, func: str, msg: str):
        super().__init__(f"{func}: {STATUS.get(status, status)}: {msg}")
        self.status = status


class oscar_pool(C.Structure):
    _fields_ = [("batch", C.c_int32), ("num_q_heads", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("group_size", C.c_int32), ("num_pages", C.c_int32),
                ("max_pages", C.c_int32),
                ("sink_k", C.c_void_p), ("sink_v", C.c_void_p), ("recent_k", C.c_void_p), ("recent_v", C.c_void_p),
                ("codes_k", C.c_void_p), ("codes_v", C.c_void_p), ("scale_k", C.c_void_p), ("zero_k", C.c_void_p),
                ("scale_v", C.c_void_p), ("zero_v", C.c_void_p), ("page_table", C.c_void_p),
                ("sink_len", C.c_void_p), ("hist_len", C.c_void_p), ("recent_start", C.c_void_p),
                ("recent_len", C.c_void_p), ("R_k", C.c_void_p), ("R_v", C.c_void_p), ("clip_k", C.c_void_p),
                ("clip_v", C.c_void_p), ("err", C.c_void_p), ("sync", C.c_void_p),
                ("codebook_k", C.c_void_p), ("codebook_v", C.c_void_p)]


class oscar_bf16_cache(C.Structure):
    _fields_ = [("batch", C.c_int32), ("num_q_heads", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("num_pages", C.c_int32), ("max_pages", C.c_int32),
                ("k_pages", C.c_void_p), ("v_pages", C.c_void_p), ("page_table", C.c_void_p),
                ("seq_len", C.c_void_p), ("err", C.c_void_p)]


P, I32, I64, SZ, F32, F64 = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t, C.c_float, C.c_double
PP = C.POINTER(oscar_pool)
PC = C.POINTER(oscar_bf16_cache)
SIGNATURES = {
    "oscar_last_error_string": ([], C.c_char_p),
    "oscar_version": ([], C.c_char_p),
    "oscar_make_rotation_workspace_size": ([I32], SZ),
    "oscar_make_rotation": ([I32, I32, P, P, P, P, SZ, P], C.c_int),
    "oscar_calib_covariance_k": ([I64, I32, I32, P, P, P], C.c_int),
    "oscar_calib_covariance_v_workspace_size": ([I64, I32, I32], SZ),
    "oscar_calib_covariance_v": ([I64, I32, I32, P, P, P, F64, P, P, SZ, P], C.c_int),
    "oscar_quantize_kv": ([I64, I32, I32, I32, P, P, P, P, P, P, P, P], C.c_int),
    "oscar_quantize_kv_codebook": ([I64, I32, I32, I32, P, P, P, P, P, P, P, P, P], C.c_int),
    "oscar_lloyd_max_workspace_size": ([I64, I32, C.POINTER(C.c_size_t)], C.c_int),
    "oscar_lloyd_max_codebook": ([I64, I32, I32, I32, P, P, P, I32, P, P, C.c_size_t, P], C.c_int),
    "oscar_prefill_pool": ([PP, I32, I64, P, P, P, P], C.c_int),
    "oscar_prefill_pool_shared": ([PP, I32, I64, P, P, I32, P, P], C.c_int),
    "oscar_demote": ([PP, P, P], C.c_int),
    "oscar_append_kv": ([PP, P, P, P], C.c_int),
    "oscar_decode_workspace_size": ([PP, I32, C.POINTER(C.c_size_t)], C.c_int),
    "oscar_decode_attention": ([PP, P, P, F32, I32, P, SZ, P], C.c_int),
    "oscar_profile_events": ([I32, P, P], C.c_int),
    "oscar_decode_attention_noalloc": ([PP, P, P, F32, P], C.c_int),
    "oscar_decode_step": ([PP, P, P, P, P, F32, P, SZ, P], C.c_int),
    "oscar_bf16_prefill": ([PC, I32, I64, P, P, P], C.c_int),
    "oscar_bf16_append_kv": ([PC, P, P, P], C.c_int),
    "oscar_bf16_decode_workspace_size": ([PC, C.POINTER(C.c_size_t)], C.c_int),
    "oscar_bf16_decode_attention": ([PC, P, P, F32, P, SZ, P], C.c_int),
    "oscar_bf16_decode_step": ([PC, P, P, P, P, F32, P, SZ, P], C.c_int),
}

_LIB = None


def header_functions() -> list[str]:
    """Names of every function declared in include/oscar.h."""
    text = open(os.path.join(_build.INCLUDE, "oscar.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(oscar_[a-z0-9_]+)\s*\(", text)))


def load(path: str | None = None) -> C.CDLL:
    """Load liboscar.so (liboscar_debug.so, the build with device-side bounds checks, when the environment
    sets OSCAR_DEBUG=1); raises if it has not been built (there is no fallback implementation)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or (_build.LIB_DEBUG if os.environ.get("OSCAR_DEBUG") == "1" else _build.LIB)
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                           "(the CUDA library is the only implementation; there is no fallback)")
    lib = C.CDLL(path)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes, fn.restype = args, res
    _LIB = lib
    return lib


def check(status: int, func: str) -> None:
    if status != 0:
        raise OscarError(status, func, load().oscar_last_error_string().decode())
