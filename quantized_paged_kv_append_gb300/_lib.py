"""ctypes binding of libqkv.so (include/qkv.h).

Argument marshalling only: torch tensors are passed as device pointers and
every step of the path runs in the library's CUDA kernels. There is no CPU
fallback: if the library cannot be loaded, every call raises.
"""

from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libqkv.so")

QKV_INT8, QKV_K8V4, QKV_ISO3, QKV_ISO4 = 0, 1, 2, 3
QKV_Q4, QKV_K8_VBF16, QKV_KBF16_V8 = 4, 5, 6
FORMATS = {"int8": QKV_INT8, "k8v4": QKV_K8V4, "iso3": QKV_ISO3, "iso4": QKV_ISO4, "q4": QKV_Q4,
           "k8vbf16": QKV_K8_VBF16, "kbf16v8": QKV_KBF16_V8}
QKV_OUT_BF16, QKV_OUT_F32 = 0, 1
ERRORS = {0: "QKV_OK", -1: "QKV_ERR_ARG", -2: "QKV_ERR_HEAD_DIM", -3: "QKV_ERR_GQA", -4: "QKV_ERR_WORKSPACE",
          -5: "QKV_ERR_FORMAT", -6: "QKV_ERR_CUDA", -7: "QKV_ERR_DEVICE", -8: "QKV_ERR_UNSUPPORTED"}

# every symbol include/qkv.h declares
EXPORTS = ["qkv_row_bytes", "qkv_iso_levels", "iso_kv_append", "kv_decode_workspace_size", "kv_decode_attn",
           "kv_extend_workspace_size", "kv_extend_attn", "kv_gather_dequant", "kv_verify_workspace_size", "kv_verify_attn",
           "kv_verify_fixed_workspace_size", "kv_verify_attn_fixed", "kv_decode_attn_noalloc", "qkv_strerror",
           "qkv_last_cuda_error", "qkv_device_error"]


class CacheDesc(C.Structure):
    _fields_ = [("format", C.c_int32), ("num_pages", C.c_int32), ("page_size", C.c_int32),
                ("num_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("reserved0", C.c_int32),
                ("k_codes", C.c_void_p), ("k_scales", C.c_void_p), ("v_codes", C.c_void_p),
                ("v_scales", C.c_void_p), ("quat", C.c_float * 4)]


class QkvError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        msg = f"{what}: {ERRORS.get(code, code)}"
        try:
            msg += f" ({lib().qkv_strerror(code).decode()})"
            if code == -6:
                msg += f", cudaError {lib().qkv_last_cuda_error()}"
        except Exception:
            pass
        super().__init__(msg)


_lib = None


def lib():
    """Load libqkv.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libqkv.so not built ({LIB_PATH}); run quantized_paged_kv_append_gb300.build.build()")
        L = C.CDLL(LIB_PATH)
        P, I, SZ = C.c_void_p, C.c_int, C.c_size_t
        L.qkv_row_bytes.argtypes = [I, I, I, C.POINTER(I), C.POINTER(I)]
        L.qkv_row_bytes.restype = I
        L.qkv_iso_levels.argtypes = [I, P]
        L.qkv_iso_levels.restype = I
        L.iso_kv_append.argtypes = [C.POINTER(CacheDesc), P, P, I, P, P, P, I, I, P]
        L.iso_kv_append.restype = I
        L.kv_decode_workspace_size.argtypes = [C.POINTER(CacheDesc), I, I, I]
        L.kv_decode_workspace_size.restype = SZ
        L.kv_decode_attn.argtypes = [C.POINTER(CacheDesc), P, P, P, I, I, P, I, P, I, C.c_float, P, I, P, SZ, P]
        L.kv_decode_attn.restype = I
        L.kv_extend_workspace_size.argtypes = [C.POINTER(CacheDesc), I, I, I]
        L.kv_extend_workspace_size.restype = SZ
        L.kv_extend_attn.argtypes = [C.POINTER(CacheDesc), P, P, P, I, P, P, I, I, P, I, C.c_float, I, P, I, P, SZ,
                                     P]
        L.kv_extend_attn.restype = I
        L.kv_verify_workspace_size.argtypes = [C.POINTER(CacheDesc), I, I, I]
        L.kv_verify_workspace_size.restype = SZ
        L.kv_verify_attn.argtypes = [C.POINTER(CacheDesc), P, I, I, P, P, I, P, I, I, C.c_float, P, I, P, SZ, P]
        L.kv_verify_attn.restype = I
        L.kv_verify_fixed_workspace_size.argtypes = [C.POINTER(CacheDesc), I, I, I, I]
        L.kv_verify_fixed_workspace_size.restype = SZ
        L.kv_verify_attn_fixed.argtypes = [C.POINTER(CacheDesc), P, I, I, I, P, P, I, I, C.c_float, P, I, P, SZ, P]
        L.kv_verify_attn_fixed.restype = I
        L.kv_gather_dequant.argtypes = [C.POINTER(CacheDesc), P, I, P, P, P]
        L.kv_gather_dequant.restype = I
        L.kv_decode_attn_noalloc.argtypes = [C.POINTER(CacheDesc), P, P, P, I, I, P, I, P, I, C.c_float, P, I, P]
        L.kv_decode_attn_noalloc.restype = I
        L.qkv_strerror.argtypes = [I]
        L.qkv_strerror.restype = C.c_char_p
        L.qkv_last_cuda_error.argtypes = []
        L.qkv_last_cuda_error.restype = I
        L.qkv_device_error.argtypes = [I]
        L.qkv_device_error.restype = I
        _lib = L
    return _lib


def check(rc, what):
    if rc != 0:
        raise QkvError(rc, what)
