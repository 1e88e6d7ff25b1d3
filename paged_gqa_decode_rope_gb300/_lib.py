"""ctypes view of ``libhpc_decode.so`` (declared in include/hpc_decode.h).

Loading fails loudly when the library has not been built: there is no other
implementation to fall back to.
"""

import ctypes
import os

from .build import LIB

HPC_OK = 0
HPC_ERR_INVALID_ARG = -1
HPC_ERR_UNSUPPORTED = -2
HPC_ERR_CUDA = -3
NOALLOC_MAX_ITEMS = 4096
MAX_Q_LEN = 4
Q_BF16, Q_FP8 = 0, 1
OUT_BF16, OUT_FP16, OUT_FP32 = 0, 1, 2

STATUS_BITS = {
    1: "BAD_BLOCK", 2: "BAD_SLOT", 4: "BAD_SEQ_LEN", 8: "BAD_POSITION",
    16: "PLAN_OVERFLOW", 32: "WAIT_TIMEOUT", 64: "BAD_PLAN",
}

_c_i32 = ctypes.c_int32
_c_p = ctypes.c_void_p


class WorkItem(ctypes.Structure):
    _fields_ = [("seq", _c_i32), ("kv_head", _c_i32), ("tile_begin", _c_i32), ("tile_end", _c_i32)]


class Plan(ctypes.Structure):
    _fields_ = [("items", _c_p), ("cta_ptr", _c_p), ("seg_ptr", _c_p), ("home_end", _c_p),
                ("pool", _c_p), ("seg_done", _c_p), ("capacity", _c_i32), ("num_ctas", _c_i32)]


class PlanParams(ctypes.Structure):
    _fields_ = [("min_tiles", _c_i32), ("pool_chunks", _c_i32), ("pool_min_tiles", _c_i32)]


class AttnOptions(ctypes.Structure):
    """hpc_attn_options: new tokens per sequence, q type and scale, output type."""
    _fields_ = [("q_len", ctypes.c_int32), ("q_dtype", ctypes.c_int32),
                ("q_scale", ctypes.c_float), ("out_dtype", ctypes.c_int32)]


# name -> (restype, argtypes); the order follows include/hpc_decode.h
SIGNATURES = {
    "hpc_rope_cos_sin_cache": (ctypes.c_int, [ctypes.c_double, _c_i32, _c_p, _c_p]),
    "hpc_rope_norm_kvwrite": (ctypes.c_int, [
        _c_p, _c_p, _c_p, _c_p, _c_p, _c_i32, _c_p, _c_p, ctypes.c_float,
        _c_p, _c_i32, _c_i32, _c_p, _c_p, _c_p, _c_i32, _c_p, _c_p]),
    "hpc_decode_plan": (ctypes.c_int, [_c_p, _c_i32, _c_i32, ctypes.POINTER(PlanParams),
                                       ctypes.POINTER(Plan), _c_p, _c_p]),
    "hpc_decode_plan_static": (ctypes.c_int, [_c_p, _c_i32, _c_i32, _c_i32, ctypes.POINTER(Plan), _c_p, _c_p]),
    "hpc_decode_attn": (ctypes.c_int, [
        _c_p, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, ctypes.POINTER(Plan),
        _c_p, _c_p, ctypes.c_float, _c_p, _c_p]),
    "hpc_decode_attn_merge": (ctypes.c_int, [
        _c_p, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, ctypes.POINTER(Plan),
        _c_p, _c_p, _c_p, ctypes.c_float, _c_p, _c_p]),
    "hpc_decode_attn_profiled": (ctypes.c_int, [
        _c_p, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, ctypes.POINTER(Plan),
        _c_p, _c_p, ctypes.c_float, _c_p, _c_p, _c_p]),
    "hpc_merge": (ctypes.c_int, [_c_p, _c_p, ctypes.POINTER(Plan), _c_i32, _c_p, _c_p]),
    "hpc_decode_attn_merge_noalloc": (ctypes.c_int, [
        _c_p, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, ctypes.POINTER(Plan),
        _c_p, ctypes.c_float, _c_p, _c_p]),
    "hpc_decode_step": (ctypes.c_int, [
        _c_p, _c_p, _c_p, _c_p, _c_p, _c_i32, _c_p, _c_p, ctypes.c_float, _c_p, _c_i32, _c_i32,
        _c_p, _c_p, _c_p, _c_i32, _c_p, _c_i32, ctypes.POINTER(PlanParams), ctypes.POINTER(Plan),
        _c_p, _c_p, _c_p, _c_p, ctypes.c_float, _c_p, _c_p]),
    "hpc_decode_num_ctas": (ctypes.c_int, [_c_i32, ctypes.POINTER(_c_i32)]),
    "hpc_decode_num_queues": (ctypes.c_int, [_c_i32, _c_i32, _c_i32, ctypes.POINTER(_c_i32)]),
    "hpc_plan_capacity": (_c_i32, [_c_i32, _c_i32, _c_i32]),
    "hpc_decode_attn_mt": (ctypes.c_int, [
        _c_p, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, _c_i32, ctypes.POINTER(Plan),
        _c_p, _c_p, ctypes.c_float, _c_p, _c_p]),
    "hpc_decode_attn_merge_mt": (ctypes.c_int, [
        _c_p, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, _c_i32, ctypes.POINTER(Plan),
        _c_p, _c_p, _c_p, ctypes.c_float, _c_p, _c_p]),
    "hpc_merge_mt": (ctypes.c_int, [_c_p, _c_p, ctypes.POINTER(Plan), _c_i32, _c_i32, _c_p, _c_p]),
    "hpc_rope_norm_kvwrite_ex": (ctypes.c_int, [
        _c_p, _c_p, _c_p, _c_p, _c_p, _c_i32, _c_p, _c_p, ctypes.c_float,
        _c_p, _c_i32, _c_i32, _c_p, _c_p, _c_i32, ctypes.c_float, _c_p, _c_i32, _c_p, _c_p]),
    "hpc_decode_attn_ex": (ctypes.c_int, [
        _c_p, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, ctypes.POINTER(AttnOptions),
        ctypes.POINTER(Plan), _c_p, _c_p, ctypes.c_float, _c_p, _c_p]),
    "hpc_decode_attn_merge_ex": (ctypes.c_int, [
        _c_p, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, ctypes.POINTER(AttnOptions),
        ctypes.POINTER(Plan), _c_p, _c_p, _c_p, ctypes.c_float, _c_p, _c_p]),
    "hpc_merge_ex": (ctypes.c_int, [_c_p, _c_p, ctypes.POINTER(Plan), _c_i32,
                                    ctypes.POINTER(AttnOptions), _c_p, _c_p]),
    "hpc_prefill_plan": (ctypes.c_int, [_c_p, _c_i32, _c_p, _c_p, _c_p, _c_p]),
    "hpc_prefill_attn": (ctypes.c_int, [
        _c_p, _c_i32, _c_p, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_p, _c_p,
        _c_i32, ctypes.c_float, _c_p, _c_p]),
    "hpc_prefill_attn_staged": (ctypes.c_int, [
        _c_p, _c_i32, _c_p, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_p, _c_p,
        _c_i32, ctypes.c_float, _c_p, _c_i32, _c_p, _c_p, _c_p]),
    "hpc_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint64, _c_p, _c_p, _c_p]),
    "hpc_selftest_poll_timeout": (ctypes.c_int, [ctypes.c_uint64, _c_p, _c_p, _c_p]),
}

_lib = None


def lib():
    """The loaded library with typed entry points."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(
                "libhpc_decode.so is not built (expected at %s); build it with "
                "`python -m paged_gqa_decode_rope_gb300.build` or __graft_entry__.build()" % LIB)
        handle = ctypes.CDLL(LIB)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


class HpcError(RuntimeError):
    def __init__(self, call, code):
        names = {HPC_ERR_INVALID_ARG: "HPC_ERR_INVALID_ARG", HPC_ERR_UNSUPPORTED: "HPC_ERR_UNSUPPORTED",
                 HPC_ERR_CUDA: "HPC_ERR_CUDA"}
        super().__init__("%s returned %s" % (call, names.get(code, code)))
        self.code = code


def check(call, code):
    if code != HPC_OK:
        raise HpcError(call, code)


def status_names(status):
    return [name for bit, name in STATUS_BITS.items() if status & bit]
