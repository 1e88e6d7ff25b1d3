"""Python binding of the decode-step C ABI: torch tensors in, C pointers out.

Each function checks dtypes, shapes, devices and contiguity, then calls the
entry point of the same name in libhpc_decode.so on the current CUDA stream.
No step of the computation runs here; torch only provides device memory and
the stream.
"""

import ctypes
import math

import torch

from . import _lib
from ._lib import Plan, check

KV_BF16 = 0
KV_FP8 = 1
HQ, HKV, D, PAGE = 64, 8, 128, 64
THETA = 1.0e6
EPS = 1.0e-6


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _want(t, name, dtypes, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype not in dtypes:
        raise TypeError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtypes))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))


_BF16 = (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (torch.bfloat16, torch.int16)
_FP8 = (torch.uint8, torch.float8_e4m3fn)


def _cache_dtypes(kv_dtype):
    if kv_dtype == KV_BF16:
        return _BF16
    if kv_dtype == KV_FP8:
        return _FP8
    raise ValueError("kv_dtype must be KV_BF16 (0) or KV_FP8 (1)")


def num_ctas(kv_dtype=KV_BF16):
    """Persistent grid of the attention kernel on the current device."""
    n = ctypes.c_int32(0)
    check("hpc_decode_num_ctas", _lib.lib().hpc_decode_num_ctas(kv_dtype, ctypes.byref(n)))
    return n.value


class DecodePlan:
    """Device buffers of a split-KV plan plus the C struct that points at them."""

    def __init__(self, batch, n_ctas, capacity, device):
        self.batch, self.num_ctas, self.capacity = batch, n_ctas, capacity
        self.items = torch.empty((max(capacity, 1), 4), dtype=torch.int32, device=device)
        self.cta_ptr = torch.empty(n_ctas + 1, dtype=torch.int32, device=device)
        self.seg_ptr = torch.empty(batch * HKV + 1, dtype=torch.int32, device=device)
        self.c = Plan(self.items.data_ptr(), self.cta_ptr.data_ptr(), self.seg_ptr.data_ptr(),
                      capacity, n_ctas)

    @classmethod
    def dynamic(cls, batch, device="cuda", n_ctas=None, kv_dtype=KV_BF16):
        n_ctas = num_ctas(kv_dtype) if n_ctas is None else n_ctas
        return cls(batch, n_ctas, _lib.lib().hpc_plan_capacity(batch, n_ctas), device)

    @classmethod
    def static(cls, batch, splits, device="cuda"):
        n = batch * HKV * splits
        return cls(batch, n, n, device)


def rope_cos_sin_cache(max_pos, theta=THETA, device="cuda"):
    out = torch.empty((max_pos, D), dtype=torch.float32, device=device)
    check("hpc_rope_cos_sin_cache",
          _lib.lib().hpc_rope_cos_sin_cache(float(theta), int(max_pos), _p(out), _stream()))
    return out


def rope_norm_kvwrite(q, k, v, positions, cos_sin, q_norm_w, k_norm_w, kv_cache, kv_dtype,
                      slot_mapping, kv_scale, q_out, status, eps=EPS):
    B = q.shape[0]
    _want(q, "q", _BF16, (B, HQ, D))
    _want(k, "k", _BF16, (B, HKV, D))
    _want(v, "v", _BF16, (B, HKV, D))
    _want(positions, "positions", (torch.int32,), (B,))
    _want(cos_sin, "cos_sin", (torch.float32,))
    if cos_sin.dim() != 2 or cos_sin.shape[1] != D:
        raise ValueError("cos_sin must be [max_pos, 128]")
    _want(q_norm_w, "q_norm_w", _BF16, (D,))
    _want(k_norm_w, "k_norm_w", _BF16, (D,))
    _want(kv_cache, "kv_cache", _cache_dtypes(kv_dtype))
    if kv_cache.dim() != 5 or tuple(kv_cache.shape[1:]) != (2, HKV, PAGE, D):
        raise ValueError("kv_cache must be [num_blocks, 2, 8, 64, 128]")
    _want(slot_mapping, "slot_mapping", (torch.int64,), (B,))
    if kv_dtype == KV_FP8:
        _want(kv_scale, "kv_scale", (torch.float32,), (2,))
    _want(q_out, "q_out", _BF16, (B, HQ, D))
    _want(status, "status", (torch.int32,), (1,))
    check("hpc_rope_norm_kvwrite", _lib.lib().hpc_rope_norm_kvwrite(
        _p(q), _p(k), _p(v), _p(positions), _p(cos_sin), cos_sin.shape[0], _p(q_norm_w),
        _p(k_norm_w), float(eps), _p(kv_cache), kv_dtype, kv_cache.shape[0], _p(slot_mapping),
        _p(kv_scale if kv_dtype == KV_FP8 else None), _p(q_out), B, _p(status), _stream()))


def decode_plan(seq_lens, max_blocks, plan, status, min_tiles=1):
    _want(seq_lens, "seq_lens", (torch.int32,), (plan.batch,))
    _want(status, "status", (torch.int32,), (1,))
    check("hpc_decode_plan", _lib.lib().hpc_decode_plan(
        _p(seq_lens), plan.batch, int(max_blocks), int(min_tiles), ctypes.byref(plan.c),
        _p(status), _stream()))


def decode_plan_static(seq_lens, max_blocks, splits, plan, status):
    _want(seq_lens, "seq_lens", (torch.int32,), (plan.batch,))
    _want(status, "status", (torch.int32,), (1,))
    check("hpc_decode_plan_static", _lib.lib().hpc_decode_plan_static(
        _p(seq_lens), plan.batch, int(max_blocks), int(splits), ctypes.byref(plan.c),
        _p(status), _stream()))


def decode_attn(q, kv_cache, kv_dtype, kv_scale, block_table, seq_lens, plan, partial_o,
                partial_lse, status, sm_scale=None):
    B = q.shape[0]
    _want(q, "q", _BF16, (B, HQ, D))
    _want(kv_cache, "kv_cache", _cache_dtypes(kv_dtype))
    if kv_cache.dim() != 5 or tuple(kv_cache.shape[1:]) != (2, HKV, PAGE, D):
        raise ValueError("kv_cache must be [num_blocks, 2, 8, 64, 128]")
    if kv_dtype == KV_FP8:
        _want(kv_scale, "kv_scale", (torch.float32,), (2,))
    _want(block_table, "block_table", (torch.int32,))
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [batch, max_blocks]")
    _want(seq_lens, "seq_lens", (torch.int32,), (B,))
    if plan.batch != B:
        raise ValueError("plan was made for batch %d, not %d" % (plan.batch, B))
    _want(partial_o, "partial_o", (torch.float32,))
    _want(partial_lse, "partial_lse", (torch.float32,))
    if partial_o.numel() < plan.capacity * HKV * D or partial_lse.numel() < plan.capacity * HKV:
        raise ValueError("partial buffers are smaller than the plan capacity")
    _want(status, "status", (torch.int32,), (1,))
    scale = 1.0 / math.sqrt(D) if sm_scale is None else float(sm_scale)
    check("hpc_decode_attn", _lib.lib().hpc_decode_attn(
        _p(q), _p(kv_cache), kv_dtype, _p(kv_scale if kv_dtype == KV_FP8 else None),
        kv_cache.shape[0], _p(block_table), block_table.shape[1], _p(seq_lens), B,
        ctypes.byref(plan.c), _p(partial_o), _p(partial_lse), scale, _p(status), _stream()))


def merge(partial_o, partial_lse, plan, out):
    B = plan.batch
    _want(partial_o, "partial_o", (torch.float32,))
    _want(partial_lse, "partial_lse", (torch.float32,))
    _want(out, "out", _BF16, (B, HQ, D))
    check("hpc_merge", _lib.lib().hpc_merge(
        _p(partial_o), _p(partial_lse), ctypes.byref(plan.c), B, _p(out), _stream()))


class DecodeStep:
    """All four calls of one decode step, with the plan and partial buffers
    allocated once for a batch size (so the step can be graph-captured).

    ``schedule`` is "dynamic" (length-proportional, the default) or
    ("static", splits) for the equal-split comparator.
    """

    def __init__(self, batch, kv_dtype, max_blocks, device="cuda", schedule="dynamic",
                 min_tiles=1, n_ctas=None):
        self.batch, self.kv_dtype, self.max_blocks = batch, kv_dtype, max_blocks
        self.min_tiles = min_tiles
        if schedule == "dynamic":
            self.plan = DecodePlan.dynamic(batch, device, n_ctas, kv_dtype)
            self.splits = None
        else:
            self.splits = int(schedule[1])
            self.plan = DecodePlan.static(batch, self.splits, device)
        cap = max(self.plan.capacity, 1)
        self.partial_o = torch.empty((cap, HKV, D), dtype=torch.float32, device=device)
        self.partial_lse = torch.empty((cap, HKV), dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.q_out = torch.empty((batch, HQ, D), dtype=torch.bfloat16, device=device)
        self.out = torch.empty((batch, HQ, D), dtype=torch.bfloat16, device=device)

    def plan_step(self, seq_lens):
        if self.splits is None:
            decode_plan(seq_lens, self.max_blocks, self.plan, self.status, self.min_tiles)
        else:
            decode_plan_static(seq_lens, self.max_blocks, self.splits, self.plan, self.status)

    def attend(self, q, kv_cache, kv_scale, block_table, seq_lens):
        decode_attn(q, kv_cache, self.kv_dtype, kv_scale, block_table, seq_lens, self.plan,
                    self.partial_o, self.partial_lse, self.status)
        merge(self.partial_o, self.partial_lse, self.plan, self.out)
        return self.out

    def __call__(self, q, k, v, positions, cos_sin, q_norm_w, k_norm_w, kv_cache, slot_mapping,
                 kv_scale, block_table, seq_lens):
        rope_norm_kvwrite(q, k, v, positions, cos_sin, q_norm_w, k_norm_w, kv_cache, self.kv_dtype,
                          slot_mapping, kv_scale, self.q_out, self.status)
        self.plan_step(seq_lens)
        return self.attend(self.q_out, kv_cache, kv_scale, block_table, seq_lens)
