"""Thin ctypes binding of libswiftkv.so: the C-ABI calls under the same names,
argument marshalling only. Device memory and streams come from PyTorch; every
step of the computation runs in the library's CUDA kernels. There is no CPU
fallback: loading fails loudly if the library cannot be built or opened.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

from . import build as _build

_lib = None
_lock = threading.Lock()

SWIFTKV_OK = 0
ERRORS = {
    -1: "EINVAL", -2: "EINVAL_L", -3: "EINVAL_GROUP", -4: "EINVAL_SEQLENS", -5: "ENO_PAGES",
    -6: "EOOM", -7: "ECUDA", -8: "EDEVICE", -9: "EUNSUPPORTED", -10: "ESTATE",
}
STATUS_BAD_TOKEN = 1
STATUS_BAD_PAGE = 2
STATUS_TIMEOUT = 4

# every symbol include/swiftkv.h declares
EXPORTS = ("swiftkv_cache_count", "swiftkv_model_create", "swiftkv_load_layer", "swiftkv_load_globals",
           "swiftkv_load_weights", "swiftkv_prefill", "swiftkv_prefill_host", "swiftkv_forward",
           "swiftkv_decode_step",
           "swiftkv_status", "swiftkv_memory", "swiftkv_set_gemm_impl", "swiftkv_set_attention_impl",
           "swiftkv_set_norm_fusion", "swiftkv_set_rows_impl", "swiftkv_gemm_bf16",
           "swiftkv_gemm_skinny_noalloc", "swiftkv_selftest_wait_timeout",
           "swiftkv_profile_begin", "swiftkv_profile_end",
           "swiftkv_last_error", "swiftkv_free")


class SwiftKVError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class ModelConfig(C.Structure):
    _fields_ = [("L", C.c_int), ("d", C.c_int), ("n_q", C.c_int), ("n_kv", C.c_int), ("d_head", C.c_int),
                ("ffn", C.c_int), ("vocab", C.c_int), ("qkv_bias", C.c_int), ("rope_theta", C.c_float),
                ("rms_eps", C.c_float)]


class LayerWeights(C.Structure):
    _fields_ = [("gamma_attn", C.c_void_p), ("wq", C.c_void_p), ("wk", C.c_void_p), ("wv", C.c_void_p),
                ("bq", C.c_void_p), ("bk", C.c_void_p), ("bv", C.c_void_p), ("wo", C.c_void_p),
                ("gamma_mlp", C.c_void_p), ("w_gate", C.c_void_p), ("w_up", C.c_void_p),
                ("w_down", C.c_void_p)]


class HostWeights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("gamma_final", C.c_void_p), ("lm_head", C.c_void_p),
                ("layers", C.POINTER(LayerWeights))]


class KVPages(C.Structure):
    _fields_ = [("k_pool", C.POINTER(C.c_void_p)), ("v_pool", C.POINTER(C.c_void_p)),
                ("num_caches", C.c_int), ("num_pages", C.c_int), ("page_size", C.c_int),
                ("block_table", C.c_void_p), ("max_pages_per_seq", C.c_int), ("kv_dtype", C.c_int),
                ("k_scale", C.POINTER(C.c_void_p)), ("v_scale", C.POINTER(C.c_void_p))]


class ProfileEntry(C.Structure):
    _fields_ = [("name", C.c_char * 32), ("calls", C.c_int), ("kernels", C.c_int), ("ms", C.c_double),
                ("flops", C.c_double), ("bytes", C.c_double)]


def lib(path: str | None = None):
    """Builds (if stale) and opens libswiftkv.so."""
    global _lib
    with _lock:
        if _lib is None:
            so = path or _build.build()
            L = C.CDLL(so)
            vp, i, sz = C.c_void_p, C.c_int, C.c_size_t
            L.swiftkv_cache_count.argtypes = [i, i, i]
            L.swiftkv_model_create.argtypes = [C.POINTER(ModelConfig), i, i, C.POINTER(vp)]
            L.swiftkv_load_layer.argtypes = [vp, i, C.POINTER(LayerWeights), vp]
            L.swiftkv_load_globals.argtypes = [vp, vp, vp, vp, vp]
            L.swiftkv_load_weights.argtypes = [C.POINTER(ModelConfig), C.POINTER(HostWeights), i, i, vp,
                                               C.POINTER(vp)]
            L.swiftkv_prefill.argtypes = [vp, vp, vp, i, i, i, C.POINTER(KVPages), vp, vp]
            L.swiftkv_prefill_host.argtypes = [vp, vp, vp, i, i, i, C.POINTER(KVPages), vp, vp]
            L.swiftkv_forward.argtypes = [vp, vp, vp, vp, i, i, i, C.POINTER(KVPages), vp, vp]
            L.swiftkv_decode_step.argtypes = [vp, vp, vp, i, C.POINTER(KVPages), vp, vp, vp]
            L.swiftkv_status.argtypes = [vp, i]
            L.swiftkv_memory.argtypes = [vp, C.POINTER(sz), C.POINTER(sz)]
            L.swiftkv_set_gemm_impl.argtypes = [vp, i]
            L.swiftkv_set_attention_impl.argtypes = [vp, i]
            L.swiftkv_set_norm_fusion.argtypes = [vp, i]
            L.swiftkv_set_rows_impl.argtypes = [vp, i]
            L.swiftkv_gemm_bf16.argtypes = [vp, vp, vp, i, i, i, i, vp, vp]
            L.swiftkv_gemm_skinny_noalloc.argtypes = [vp, vp, vp, i, i, i, vp]
            L.swiftkv_selftest_wait_timeout.argtypes = [vp, vp, C.c_longlong, vp]
            L.swiftkv_profile_begin.argtypes = [vp]
            L.swiftkv_profile_end.argtypes = [vp, C.POINTER(ProfileEntry), i]
            L.swiftkv_last_error.restype = C.c_char_p
            L.swiftkv_free.argtypes = [vp]
            L.swiftkv_free.restype = None
            _lib = L
    return _lib


def check(code: int) -> int:
    if code < 0:
        raise SwiftKVError(code, lib().swiftkv_last_error().decode())
    return code


def cache_count(L: int, l: int, g: int) -> int:
    return check(lib().swiftkv_cache_count(L, l, g))
