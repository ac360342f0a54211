"""ctypes declarations of the C ABI in include/engram.h.

Loading fails loudly: there is no fallback implementation anywhere.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libengram_gb300.so")

# engram_status_t
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_NOT_MAPPED, ERR_INDEX_RANGE, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE = range(8)
STATUS_NAMES = ["OK", "INVALID_ARG", "UNSUPPORTED", "NOT_MAPPED", "INDEX_RANGE", "CUDA", "TIMEOUT", "WORKSPACE"]

# engram_dtype_t
F32, BF16, I8_ROWSCALE_F16 = 0, 1, 2

EXPORTS = ("engram_status_string", "engram_plan_create", "engram_plan_destroy", "engram_plan_workspace_bytes",
           "engram_hash", "engram_gather", "engram_kv_projection", "engram_stage_b", "engram_forward",
           "engram_get_error", "engram_plan_set_timing", "engram_plan_set_fused_stage_b", "engram_plan_set_cta_pairs",
           "engram_plan_set_fused_decode", "engram_plan_kernel_times",
           "engram_forward_static_scratch", "engram_stage_a", "engram_stage_a_layers", "engram_cache_create", "engram_cache_destroy",
           "engram_cache_observe", "engram_cache_build", "engram_stage_a_cached", "engram_cache_stats",
           "engram_cache_set_dedup", "engram_quantize_fp8", "engram_plan_set_sm_limit", "engram_plan_host_gather_sms", "engram_plan_set_host_gather_sms",
           "engram_sm_split_create", "engram_sm_split_sms", "engram_sm_split_stream", "engram_sm_split_destroy",
           "engram_forward_split", "engram_stage_a_e4m3", "engram_stage_a_layers_e4m3", "engram_stage_b_e4m3")


class Config(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int), ("K", ctypes.c_int), ("row_dim", ctypes.c_int), ("d", ctypes.c_int),
                ("M", ctypes.c_int), ("conv_w", ctypes.c_int), ("conv_dilation", ctypes.c_int),
                ("table_dtype", ctypes.c_int), ("act_dtype", ctypes.c_int), ("eps", ctypes.c_float),
                ("primes", ctypes.POINTER(ctypes.c_uint32)), ("multipliers", ctypes.POINTER(ctypes.c_uint64))]


class Weights(ctypes.Structure):
    _fields_ = [("table", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("w_kv", ctypes.c_void_p),
                ("g_h", ctypes.c_void_p), ("g_k", ctypes.c_void_p), ("g_c", ctypes.c_void_p),
                ("conv", ctypes.c_void_p), ("w_kv_fp8", ctypes.c_void_p), ("w_kv_scale", ctypes.c_void_p)]


class State(ctypes.Structure):
    _fields_ = [("prev_ids", ctypes.c_void_p), ("u_ring", ctypes.c_void_p), ("pos", ctypes.c_void_p)]


class EngramError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        msg = _lib().engram_status_string(status).decode() if _LIB else name
        super().__init__(f"{where}: ENGRAM_ERR_{name} ({msg})")


_LIB = None


def _lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m hashed_gram_embedding_engram_gb300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        lib.engram_status_string.restype = ctypes.c_char_p
        lib.engram_status_string.argtypes = [i32]
        lib.engram_plan_create.argtypes = [ctypes.POINTER(Config), i64, ctypes.POINTER(vp)]
        lib.engram_plan_destroy.argtypes = [vp]
        lib.engram_plan_workspace_bytes.argtypes = [vp, i64, ctypes.POINTER(sz)]
        lib.engram_hash.argtypes = [vp, vp, i32, i32, vp, i32, vp, vp, vp]
        lib.engram_gather.argtypes = [vp, vp, i64, vp, vp, vp, vp]
        lib.engram_kv_projection.argtypes = [vp, vp, i64, vp, vp, vp]
        lib.engram_quantize_fp8.argtypes = [vp, vp, i64, i32, vp, vp, vp]
        lib.engram_stage_a.argtypes = [vp, vp, i32, i32, vp, i32, vp, vp, vp, vp, vp]
        lib.engram_stage_a_layers.argtypes = [i32, vp, vp, i32, i32, vp, i32, vp, vp, vp, vp, vp]
        lib.engram_cache_create.argtypes = [vp, i64, vp, ctypes.POINTER(vp)]
        lib.engram_cache_destroy.argtypes = [vp]
        lib.engram_cache_observe.argtypes = [vp, vp, i32, i32, vp, i32, vp, vp]
        lib.engram_cache_build.argtypes = [vp, i32, vp, ctypes.POINTER(i64)]
        lib.engram_stage_a_cached.argtypes = [vp, vp, i32, i32, vp, i32, vp, vp, vp, vp]
        lib.engram_cache_stats.argtypes = [vp, vp, i32, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64),
                                           ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(i64)]
        lib.engram_cache_set_dedup.argtypes = [vp, i64]
        lib.engram_stage_b.argtypes = [vp, vp, i32, i32, vp, i32, vp, ctypes.POINTER(Weights), vp,
                                       ctypes.POINTER(State), vp, sz, vp]
        lib.engram_forward.argtypes = [vp, vp, i32, i32, vp, i32, ctypes.POINTER(Weights), vp,
                                       ctypes.POINTER(State), vp, sz, vp]
        lib.engram_get_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.engram_forward_static_scratch.argtypes = [vp, vp, i32, i32, vp, i32, ctypes.POINTER(Weights), vp,
                                                      ctypes.POINTER(State), vp]
        lib.engram_plan_set_timing.argtypes = [vp, i32]
        lib.engram_plan_set_fused_stage_b.argtypes = [vp, i32]
        lib.engram_plan_set_cta_pairs.argtypes = [vp, i32]
        lib.engram_plan_set_sm_limit.argtypes = [vp, i32]
        lib.engram_plan_host_gather_sms.argtypes = [vp]
        lib.engram_plan_host_gather_sms.restype = i32
        lib.engram_plan_set_host_gather_sms.argtypes = [vp, i32]
        lib.engram_sm_split_create.argtypes = [i32, i32, ctypes.POINTER(vp)]
        lib.engram_sm_split_sms.argtypes = [vp, i32]
        lib.engram_sm_split_sms.restype = i32
        lib.engram_sm_split_stream.argtypes = [vp, i32]
        lib.engram_sm_split_stream.restype = vp
        lib.engram_sm_split_destroy.argtypes = [vp]
        lib.engram_forward_split.argtypes = [vp, vp, i32, vp, vp, i32, i32, vp, i32, ctypes.POINTER(Weights), vp,
                                             ctypes.POINTER(State), vp, sz, vp]
        lib.engram_stage_a_e4m3.argtypes = [vp, vp, i32, i32, vp, i32, vp, vp, vp, vp, vp]
        lib.engram_stage_a_layers_e4m3.argtypes = [i32, vp, vp, i32, i32, vp, i32, vp, vp, vp, vp, vp]
        lib.engram_stage_b_e4m3.argtypes = [vp, vp, i32, i32, vp, i32, vp, vp, ctypes.POINTER(Weights), vp,
                                            ctypes.POINTER(State), vp, sz, vp]
        lib.engram_plan_set_fused_decode.argtypes = [vp, i32]
        lib.engram_plan_kernel_times.argtypes = [vp, ctypes.POINTER(ctypes.c_float), i32, ctypes.POINTER(i32)]
        for name in EXPORTS:
            if name not in ("engram_status_string", "engram_sm_split_stream"):   # those two return pointers
                getattr(lib, name).restype = i32
        _LIB = lib
    return _LIB


def check(status: int, where: str) -> None:
    if status != OK:
        raise EngramError(status, where)
