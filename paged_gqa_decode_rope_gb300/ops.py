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
from ._lib import Plan, PlanParams, check

KV_BF16 = 0
KV_FP8 = 1
HQ, HKV, D, PAGE = 64, 8, 128, 64
THETA = 1.0e6
EPS = 1.0e-6
POOL_CHUNKS = 4          # tail chunks per CTA range dealt at run time
POOL_MIN_TILES = 16      # shorter chunks are not worth dealing: no pool then


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


def num_ctas(kv_dtype=KV_BF16, q_len=1, q_dtype=None):
    """Work queues of the persistent attention grid on the current device for
    the KV dtype, the new tokens per sequence and the q dtype: the plan's
    num_ctas."""
    n = ctypes.c_int32(0)
    qd = Q_BF16 if q_dtype is None else int(q_dtype)
    if q_len == 1 and qd == Q_BF16:
        check("hpc_decode_num_ctas", _lib.lib().hpc_decode_num_ctas(kv_dtype, ctypes.byref(n)))
    else:
        check("hpc_decode_num_queues",
              _lib.lib().hpc_decode_num_queues(kv_dtype, int(q_len), qd, ctypes.byref(n)))
    return n.value


class DecodePlan:
    """Device buffers of a split-KV plan plus the C struct that points at them."""

    def __init__(self, batch, n_ctas, capacity, device, pool_chunks=0, pool_min_tiles=POOL_MIN_TILES):
        self.batch, self.num_ctas, self.capacity = batch, n_ctas, capacity
        self.pool_chunks, self.pool_min_tiles = pool_chunks, pool_min_tiles
        self.items = torch.empty((max(capacity, 1), 4), dtype=torch.int32, device=device)
        self.cta_ptr = torch.empty(n_ctas + 1, dtype=torch.int32, device=device)
        self.seg_ptr = torch.empty(batch * HKV + 1, dtype=torch.int32, device=device)
        self.home_end = torch.empty(n_ctas, dtype=torch.int32, device=device)
        self.pool = torch.zeros(3 + max(capacity, 1), dtype=torch.int32, device=device)
        self.seg_done = torch.zeros(max(batch * HKV, 1), dtype=torch.int32, device=device)
        self.c = Plan(self.items.data_ptr(), self.cta_ptr.data_ptr(), self.seg_ptr.data_ptr(),
                      self.home_end.data_ptr(), self.pool.data_ptr(), self.seg_done.data_ptr(),
                      capacity, n_ctas)

    @classmethod
    def dynamic(cls, batch, device="cuda", n_ctas=None, kv_dtype=KV_BF16, pool_chunks=POOL_CHUNKS,
                pool_min_tiles=POOL_MIN_TILES, q_len=1, q_dtype=None):
        n_ctas = num_ctas(kv_dtype, q_len, q_dtype) if n_ctas is None else n_ctas
        cap = _lib.lib().hpc_plan_capacity(batch, n_ctas, pool_chunks)
        return cls(batch, n_ctas, cap, device, pool_chunks, pool_min_tiles)

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
    params = PlanParams(int(min_tiles), int(plan.pool_chunks), int(plan.pool_min_tiles))
    check("hpc_decode_plan", _lib.lib().hpc_decode_plan(
        _p(seq_lens), plan.batch, int(max_blocks), ctypes.byref(params), ctypes.byref(plan.c),
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


def decode_attn_profiled(q, kv_cache, kv_dtype, kv_scale, block_table, seq_lens, plan, partial_o,
                         partial_lse, status, cta_clock, sm_scale=None):
    """hpc_decode_attn that also records [start ns, end ns, SM id] per CTA."""
    B = q.shape[0]
    _want(cta_clock, "cta_clock", (torch.int64,), (plan.num_ctas, 3))
    _want(q, "q", _BF16, (B, HQ, D))
    _want(kv_cache, "kv_cache", _cache_dtypes(kv_dtype))
    _want(block_table, "block_table", (torch.int32,))
    _want(seq_lens, "seq_lens", (torch.int32,), (B,))
    _want(status, "status", (torch.int32,), (1,))
    if partial_o.numel() < plan.capacity * HKV * D or partial_lse.numel() < plan.capacity * HKV:
        raise ValueError("partial buffers are smaller than the plan capacity")
    scale = 1.0 / math.sqrt(D) if sm_scale is None else float(sm_scale)
    check("hpc_decode_attn_profiled", _lib.lib().hpc_decode_attn_profiled(
        _p(q), _p(kv_cache), kv_dtype, _p(kv_scale if kv_dtype == KV_FP8 else None),
        kv_cache.shape[0], _p(block_table), block_table.shape[1], _p(seq_lens), B,
        ctypes.byref(plan.c), _p(partial_o), _p(partial_lse), scale, _p(status), _p(cta_clock),
        _stream()))


def cta_occupancy(cta_clock):
    """SM occupancy and tail idle of one profiled launch.

    From per-CTA [start, end, sm] records: span = last end - first start;
    occupancy = sum of CTA busy time / (SMs used x span); tail idle = mean
    over SMs of (last end overall - that SM's last end)."""
    rec = cta_clock.cpu().numpy()
    rec = rec[rec[:, 1] > 0]
    t0, t1 = rec[:, 0].min(), rec[:, 1].max()
    span = float(t1 - t0)
    sms = {}
    for st, en, sm in rec.tolist():
        b = sms.setdefault(sm, [0, 0])
        b[0] += en - st
        b[1] = max(b[1], en)
    busy = sum(v[0] for v in sms.values())
    tail = sum(t1 - v[1] for v in sms.values()) / len(sms)
    return {"span_us": round(span / 1e3, 2), "sms": len(sms),
            "occupancy": round(busy / (len(sms) * span), 4), "tail_idle_us": round(tail / 1e3, 2),
            "ctas": int(len(rec))}


def decode_attn_merge(q, kv_cache, kv_dtype, kv_scale, block_table, seq_lens, plan, partial_o,
                      partial_lse, out, status, sm_scale=None):
    """Attention with the log-sum-exp merge fused in: writes ``out`` directly."""
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
    if partial_o.numel() < plan.capacity * HKV * D or partial_lse.numel() < plan.capacity * HKV:
        raise ValueError("partial buffers are smaller than the plan capacity")
    _want(out, "out", _BF16, (B, HQ, D))
    _want(status, "status", (torch.int32,), (1,))
    scale = 1.0 / math.sqrt(D) if sm_scale is None else float(sm_scale)
    check("hpc_decode_attn_merge", _lib.lib().hpc_decode_attn_merge(
        _p(q), _p(kv_cache), kv_dtype, _p(kv_scale if kv_dtype == KV_FP8 else None),
        kv_cache.shape[0], _p(block_table), block_table.shape[1], _p(seq_lens), B,
        ctypes.byref(plan.c), _p(partial_o), _p(partial_lse), _p(out), scale, _p(status),
        _stream()))


def merge(partial_o, partial_lse, plan, out):
    B = plan.batch
    _want(partial_o, "partial_o", (torch.float32,))
    _want(partial_lse, "partial_lse", (torch.float32,))
    _want(out, "out", _BF16, (B, HQ, D))
    check("hpc_merge", _lib.lib().hpc_merge(
        _p(partial_o), _p(partial_lse), ctypes.byref(plan.c), B, _p(out), _stream()))


def selftest_wait_timeout(limit_ns, status, waited_ns=None):
    """Run the pipeline's bounded wait on a phase that never completes (see
    hpc_selftest_wait_timeout): sets HPC_STATUS_WAIT_TIMEOUT in ``status``."""
    _want(status, "status", (torch.int32,), (1,))
    if waited_ns is not None:
        _want(waited_ns, "waited_ns", (torch.int64,), (1,))
    check("hpc_selftest_wait_timeout", _lib.lib().hpc_selftest_wait_timeout(
        int(limit_ns), _p(status), _p(waited_ns), _stream()))


def selftest_poll_timeout(limit_ns, status, waited_ns=None):
    """Run the pipeline's bounded polling wait over phases that never complete
    (see hpc_selftest_poll_timeout): sets HPC_STATUS_WAIT_TIMEOUT in ``status``."""
    _want(status, "status", (torch.int32,), (1,))
    if waited_ns is not None:
        _want(waited_ns, "waited_ns", (torch.int64,), (1,))
    check("hpc_selftest_poll_timeout", _lib.lib().hpc_selftest_poll_timeout(
        int(limit_ns), _p(status), _p(waited_ns), _stream()))


def decode_step(q, k, v, positions, cos_sin, q_norm_w, k_norm_w, kv_cache, kv_dtype, slot_mapping,
                kv_scale, block_table, seq_lens, plan, partial_o, partial_lse, q_out, out, status,
                min_tiles=1, eps=EPS, sm_scale=None):
    """The whole step in two launches (hpc_decode_step)."""
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
    _want(block_table, "block_table", (torch.int32,))
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [batch, max_blocks]")
    _want(seq_lens, "seq_lens", (torch.int32,), (B,))
    if plan.batch != B:
        raise ValueError("plan was made for batch %d, not %d" % (plan.batch, B))
    if partial_o.numel() < plan.capacity * HKV * D or partial_lse.numel() < plan.capacity * HKV:
        raise ValueError("partial buffers are smaller than the plan capacity")
    _want(q_out, "q_out", _BF16, (B, HQ, D))
    _want(out, "out", _BF16, (B, HQ, D))
    _want(status, "status", (torch.int32,), (1,))
    params = PlanParams(int(min_tiles), int(plan.pool_chunks), int(plan.pool_min_tiles))
    scale = 1.0 / math.sqrt(D) if sm_scale is None else float(sm_scale)
    check("hpc_decode_step", _lib.lib().hpc_decode_step(
        _p(q), _p(k), _p(v), _p(positions), _p(cos_sin), cos_sin.shape[0], _p(q_norm_w),
        _p(k_norm_w), float(eps), _p(kv_cache), kv_dtype, kv_cache.shape[0], _p(slot_mapping),
        _p(kv_scale if kv_dtype == KV_FP8 else None), _p(block_table), block_table.shape[1],
        _p(seq_lens), B, ctypes.byref(params), ctypes.byref(plan.c), _p(partial_o),
        _p(partial_lse), _p(q_out), _p(out), scale, _p(status), _stream()))


class DecodeStep:
    """All four calls of one decode step, with the plan and partial buffers
    allocated once for a batch size (so the step can be graph-captured).

    ``schedule`` is "dynamic" (length-proportional, the default, with
    ``pool_chunks`` tail chunks per CTA dealt at run time; 0 = none) or
    ("static", splits) for the equal-split comparator.  ``fused`` runs the
    merge inside the attention kernel (hpc_decode_attn_merge) instead of the
    separate hpc_decode_attn + hpc_merge pair.
    """

    def __init__(self, batch, kv_dtype, max_blocks, device="cuda", schedule="dynamic",
                 min_tiles=1, n_ctas=None, pool_chunks=POOL_CHUNKS, fused=True,
                 pool_min_tiles=POOL_MIN_TILES):
        self.batch, self.kv_dtype, self.max_blocks = batch, kv_dtype, max_blocks
        self.min_tiles = min_tiles
        self.fused = fused
        if schedule == "dynamic":
            self.plan = DecodePlan.dynamic(batch, device, n_ctas, kv_dtype, pool_chunks,
                                           pool_min_tiles)
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
        if self.fused:
            decode_attn_merge(q, kv_cache, self.kv_dtype, kv_scale, block_table, seq_lens,
                              self.plan, self.partial_o, self.partial_lse, self.out, self.status)
        else:
            decode_attn(q, kv_cache, self.kv_dtype, kv_scale, block_table, seq_lens, self.plan,
                        self.partial_o, self.partial_lse, self.status)
            merge(self.partial_o, self.partial_lse, self.plan, self.out)
        return self.out

    def __call__(self, q, k, v, positions, cos_sin, q_norm_w, k_norm_w, kv_cache, slot_mapping,
                 kv_scale, block_table, seq_lens, two_launch=True):
        """One step.  With the dynamic plan and the fused merge the step runs
        as two launches (hpc_decode_step) unless ``two_launch`` is False; the
        other configurations make the four calls in order."""
        if two_launch and self.fused and self.splits is None:
            decode_step(q, k, v, positions, cos_sin, q_norm_w, k_norm_w, kv_cache, self.kv_dtype,
                        slot_mapping, kv_scale, block_table, seq_lens, self.plan, self.partial_o,
                        self.partial_lse, self.q_out, self.out, self.status, self.min_tiles)
            return self.out
        rope_norm_kvwrite(q, k, v, positions, cos_sin, q_norm_w, k_norm_w, kv_cache, self.kv_dtype,
                          slot_mapping, kv_scale, self.q_out, self.status)
        self.plan_step(seq_lens)
        return self.attend(self.q_out, kv_cache, kv_scale, block_table, seq_lens)


# ------------------------------------------------------------ multi-token decode

def _check_attn_mt(q, kv_cache, kv_dtype, kv_scale, block_table, seq_lens, plan, partial_o,
                   partial_lse, status):
    if q.dim() != 4:
        raise ValueError("q must be [batch, q_len, 64, 128]")
    B, qn = q.shape[0], q.shape[1]
    if not 1 <= qn <= _lib.MAX_Q_LEN:
        raise ValueError("q_len must be 1 .. %d" % _lib.MAX_Q_LEN)
    _want(q, "q", _BF16, (B, qn, HQ, D))
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
    if (partial_o.numel() < plan.capacity * qn * HKV * D or
            partial_lse.numel() < plan.capacity * qn * HKV):
        raise ValueError("partial buffers are smaller than capacity x q_len rows")
    _want(status, "status", (torch.int32,), (1,))
    return B, qn


def decode_attn_mt(q, kv_cache, kv_dtype, kv_scale, block_table, seq_lens, plan, partial_o,
                   partial_lse, status, sm_scale=None):
    """Multi-token decode attention (q [B, q_len, 64, 128]): partials per item and new token."""
    B, qn = _check_attn_mt(q, kv_cache, kv_dtype, kv_scale, block_table, seq_lens, plan,
                           partial_o, partial_lse, status)
    scale = 1.0 / math.sqrt(D) if sm_scale is None else float(sm_scale)
    check("hpc_decode_attn_mt", _lib.lib().hpc_decode_attn_mt(
        _p(q), _p(kv_cache), kv_dtype, _p(kv_scale if kv_dtype == KV_FP8 else None),
        kv_cache.shape[0], _p(block_table), block_table.shape[1], _p(seq_lens), B, qn,
        ctypes.byref(plan.c), _p(partial_o), _p(partial_lse), scale, _p(status), _stream()))


def decode_attn_merge_mt(q, kv_cache, kv_dtype, kv_scale, block_table, seq_lens, plan, partial_o,
                         partial_lse, out, status, sm_scale=None):
    """Multi-token decode attention with the merge fused in: writes out [B, q_len, 64, 128]."""
    B, qn = _check_attn_mt(q, kv_cache, kv_dtype, kv_scale, block_table, seq_lens, plan,
                           partial_o, partial_lse, status)
    _want(out, "out", _BF16, (B, qn, HQ, D))
    scale = 1.0 / math.sqrt(D) if sm_scale is None else float(sm_scale)
    check("hpc_decode_attn_merge_mt", _lib.lib().hpc_decode_attn_merge_mt(
        _p(q), _p(kv_cache), kv_dtype, _p(kv_scale if kv_dtype == KV_FP8 else None),
        kv_cache.shape[0], _p(block_table), block_table.shape[1], _p(seq_lens), B, qn,
        ctypes.byref(plan.c), _p(partial_o), _p(partial_lse), _p(out), scale, _p(status),
        _stream()))


def merge_mt(partial_o, partial_lse, plan, out):
    """Log-sum-exp merge of multi-token partials into out [B, q_len, 64, 128]."""
    B, qn = plan.batch, out.shape[1]
    _want(partial_o, "partial_o", (torch.float32,))
    _want(partial_lse, "partial_lse", (torch.float32,))
    _want(out, "out", _BF16, (B, qn, HQ, D))
    check("hpc_merge_mt", _lib.lib().hpc_merge_mt(
        _p(partial_o), _p(partial_lse), ctypes.byref(plan.c), B, qn, _p(out), _stream()))


class DecodeStepMT:
    """Multi-token decode of q_len new tokens per sequence: the prologue of all
    B * q_len tokens, the plan, and the attention (merge fused or separate),
    with buffers allocated once for a batch size and q_len."""

    def __init__(self, batch, q_len, kv_dtype, max_blocks, device="cuda", n_ctas=None,
                 pool_chunks=POOL_CHUNKS, pool_min_tiles=POOL_MIN_TILES, fused=True, min_tiles=1):
        self.batch, self.q_len, self.kv_dtype, self.max_blocks = batch, q_len, kv_dtype, max_blocks
        self.fused, self.min_tiles = fused, min_tiles
        self.plan = DecodePlan.dynamic(batch, device, n_ctas, kv_dtype, pool_chunks, pool_min_tiles,
                                       q_len)
        cap = max(self.plan.capacity, 1)
        self.partial_o = torch.empty((cap, q_len, HKV, D), dtype=torch.float32, device=device)
        self.partial_lse = torch.empty((cap, q_len, HKV), dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.q_out = torch.empty((batch, q_len, HQ, D), dtype=torch.bfloat16, device=device)
        self.out = torch.empty((batch, q_len, HQ, D), dtype=torch.bfloat16, device=device)

    def plan_step(self, seq_lens):
        decode_plan(seq_lens, self.max_blocks, self.plan, self.status, self.min_tiles)

    def attend(self, q, kv_cache, kv_scale, block_table, seq_lens):
        if self.fused:
            decode_attn_merge_mt(q, kv_cache, self.kv_dtype, kv_scale, block_table, seq_lens,
                                 self.plan, self.partial_o, self.partial_lse, self.out, self.status)
        else:
            decode_attn_mt(q, kv_cache, self.kv_dtype, kv_scale, block_table, seq_lens, self.plan,
                           self.partial_o, self.partial_lse, self.status)
            merge_mt(self.partial_o, self.partial_lse, self.plan, self.out)
        return self.out

    def __call__(self, q, k, v, positions, cos_sin, q_norm_w, k_norm_w, kv_cache, slot_mapping,
                 kv_scale, block_table, seq_lens):
        """q [B,q_len,64,128], k and v [B,q_len,8,128], positions and
        slot_mapping [B,q_len]; seq_lens counts the new tokens."""
        B, qn = self.batch, self.q_len
        rope_norm_kvwrite(q.reshape(B * qn, HQ, D), k.reshape(B * qn, HKV, D),
                          v.reshape(B * qn, HKV, D), positions.reshape(B * qn), cos_sin, q_norm_w,
                          k_norm_w, kv_cache, self.kv_dtype, slot_mapping.reshape(B * qn), kv_scale,
                          self.q_out.view(B * qn, HQ, D), self.status)
        self.plan_step(seq_lens)
        return self.attend(self.q_out, kv_cache, kv_scale, block_table, seq_lens)



# ------------------------------------------------------------ general (_ex) forms

Q_BF16, Q_FP8 = _lib.Q_BF16, _lib.Q_FP8
OUT_BF16, OUT_FP16, OUT_FP32 = _lib.OUT_BF16, _lib.OUT_FP16, _lib.OUT_FP32
_OUT_TORCH = {OUT_BF16: torch.bfloat16, OUT_FP16: torch.float16, OUT_FP32: torch.float32}


def rope_norm_kvwrite_ex(q, k, v, positions, cos_sin, q_norm_w, k_norm_w, kv_cache, kv_dtype,
                         slot_mapping, kv_scale, q_out, status, q_dtype=Q_BF16, q_scale=1.0, eps=EPS):
    """The prologue with the q output type chosen: q_out is BF16 [T,64,128], or
    uint8 E4M3 codes of q / q_scale [T,64,128] with q_dtype = Q_FP8."""
    T = q.shape[0]
    _want(q, "q", _BF16, (T, HQ, D))
    _want(k, "k", _BF16, (T, HKV, D))
    _want(v, "v", _BF16, (T, HKV, D))
    _want(positions, "positions", (torch.int32,), (T,))
    _want(cos_sin, "cos_sin", (torch.float32,))
    _want(kv_cache, "kv_cache", _cache_dtypes(kv_dtype))
    _want(slot_mapping, "slot_mapping", (torch.int64,), (T,))
    if kv_dtype == KV_FP8:
        _want(kv_scale, "kv_scale", (torch.float32,), (2,))
    _want(q_out, "q_out", (torch.uint8,) if q_dtype == Q_FP8 else _BF16, (T, HQ, D))
    _want(status, "status", (torch.int32,), (1,))
    check("hpc_rope_norm_kvwrite_ex", _lib.lib().hpc_rope_norm_kvwrite_ex(
        _p(q), _p(k), _p(v), _p(positions), _p(cos_sin), cos_sin.shape[0], _p(q_norm_w),
        _p(k_norm_w), float(eps), _p(kv_cache), kv_dtype, kv_cache.shape[0], _p(slot_mapping),
        _p(kv_scale if kv_dtype == KV_FP8 else None), int(q_dtype), float(q_scale), _p(q_out), T,
        _p(status), _stream()))


def _opts(q_len, q_dtype, q_scale, out_dtype):
    return _lib.AttnOptions(int(q_len), int(q_dtype), float(q_scale), int(out_dtype))


def decode_attn_ex(q, kv_cache, kv_dtype, kv_scale, block_table, seq_lens, plan, partial_o,
                   partial_lse, status, q_dtype=Q_BF16, q_scale=1.0, out=None, out_dtype=OUT_BF16,
                   sm_scale=None):
    """The attention with options: q [B, q_len, 64, 128] (BF16, or uint8 E4M3
    codes with q_dtype = Q_FP8); with ``out`` given the merge is fused in and
    out [B, q_len, 64, 128] of ``out_dtype`` is written, else partials."""
    B, qn = q.shape[0], q.shape[1]
    if q.dim() != 4 or not 1 <= qn <= _lib.MAX_Q_LEN:
        raise ValueError("q must be [batch, q_len <= %d, 64, 128]" % _lib.MAX_Q_LEN)
    _want(q, "q", (torch.uint8,) if q_dtype == Q_FP8 else _BF16, (B, qn, HQ, D))
    _want(kv_cache, "kv_cache", _cache_dtypes(kv_dtype))
    _want(block_table, "block_table", (torch.int32,))
    _want(seq_lens, "seq_lens", (torch.int32,), (B,))
    if plan.batch != B:
        raise ValueError("plan was made for batch %d, not %d" % (plan.batch, B))
    if (partial_o.numel() < plan.capacity * qn * HKV * D or
            partial_lse.numel() < plan.capacity * qn * HKV):
        raise ValueError("partial buffers are smaller than capacity x q_len rows")
    _want(status, "status", (torch.int32,), (1,))
    o = _opts(qn, q_dtype, q_scale, out_dtype)
    scale = 1.0 / math.sqrt(D) if sm_scale is None else float(sm_scale)
    ks = _p(kv_scale if kv_dtype == KV_FP8 else None)
    if out is None:
        check("hpc_decode_attn_ex", _lib.lib().hpc_decode_attn_ex(
            _p(q), _p(kv_cache), kv_dtype, ks, kv_cache.shape[0], _p(block_table),
            block_table.shape[1], _p(seq_lens), B, ctypes.byref(o), ctypes.byref(plan.c),
            _p(partial_o), _p(partial_lse), scale, _p(status), _stream()))
    else:
        _want(out, "out", (_OUT_TORCH[out_dtype],), (B, qn, HQ, D))
        check("hpc_decode_attn_merge_ex", _lib.lib().hpc_decode_attn_merge_ex(
            _p(q), _p(kv_cache), kv_dtype, ks, kv_cache.shape[0], _p(block_table),
            block_table.shape[1], _p(seq_lens), B, ctypes.byref(o), ctypes.byref(plan.c),
            _p(partial_o), _p(partial_lse), _p(out), scale, _p(status), _stream()))


def merge_ex(partial_o, partial_lse, plan, out, out_dtype=OUT_BF16):
    B, qn = plan.batch, out.shape[1]
    _want(out, "out", (_OUT_TORCH[out_dtype],), (B, qn, HQ, D))
    o = _opts(qn, Q_BF16, 1.0, out_dtype)
    check("hpc_merge_ex", _lib.lib().hpc_merge_ex(
        _p(partial_o), _p(partial_lse), ctypes.byref(plan.c), B, ctypes.byref(o), _p(out),
        _stream()))


class DecodeStepEx:
    """The step in its general form: q_len new tokens per sequence, q stored as
    BF16 or E4M3 (q_dtype, q_scale; E4M3 needs an FP8 cache), output of
    out_dtype; prologue of the B * q_len tokens, plan, attention (merge fused
    or separate)."""

    def __init__(self, batch, kv_dtype, max_blocks, q_len=1, q_dtype=Q_BF16, q_scale=1.0,
                 out_dtype=OUT_BF16, device="cuda", n_ctas=None, pool_chunks=POOL_CHUNKS,
                 pool_min_tiles=POOL_MIN_TILES, fused=True, min_tiles=1):
        self.batch, self.kv_dtype, self.max_blocks = batch, kv_dtype, max_blocks
        self.q_len, self.q_dtype, self.q_scale, self.out_dtype = q_len, q_dtype, q_scale, out_dtype
        self.fused, self.min_tiles = fused, min_tiles
        self.plan = DecodePlan.dynamic(batch, device, n_ctas, kv_dtype, pool_chunks, pool_min_tiles,
                                       q_len, q_dtype)
        cap = max(self.plan.capacity, 1)
        self.partial_o = torch.empty((cap, q_len, HKV, D), dtype=torch.float32, device=device)
        self.partial_lse = torch.empty((cap, q_len, HKV), dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.q_out = torch.empty((batch, q_len, HQ, D),
                                 dtype=torch.uint8 if q_dtype == Q_FP8 else torch.bfloat16,
                                 device=device)
        self.out = torch.empty((batch, q_len, HQ, D), dtype=_OUT_TORCH[out_dtype], device=device)

    def plan_step(self, seq_lens):
        decode_plan(seq_lens, self.max_blocks, self.plan, self.status, self.min_tiles)

    def attend(self, q, kv_cache, kv_scale, block_table, seq_lens):
        if self.fused:
            decode_attn_ex(q, kv_cache, self.kv_dtype, kv_scale, block_table, seq_lens, self.plan,
                           self.partial_o, self.partial_lse, self.status, self.q_dtype,
                           self.q_scale, self.out, self.out_dtype)
        else:
            decode_attn_ex(q, kv_cache, self.kv_dtype, kv_scale, block_table, seq_lens, self.plan,
                           self.partial_o, self.partial_lse, self.status, self.q_dtype,
                           self.q_scale)
            merge_ex(self.partial_o, self.partial_lse, self.plan, self.out, self.out_dtype)
        return self.out

    def __call__(self, q, k, v, positions, cos_sin, q_norm_w, k_norm_w, kv_cache, slot_mapping,
                 kv_scale, block_table, seq_lens):
        """q [B,q_len,64,128], k and v [B,q_len,8,128], positions and
        slot_mapping [B,q_len]; seq_lens counts the new tokens."""
        B, qn = self.batch, self.q_len
        rope_norm_kvwrite_ex(q.reshape(B * qn, HQ, D), k.reshape(B * qn, HKV, D),
                             v.reshape(B * qn, HKV, D), positions.reshape(B * qn), cos_sin,
                             q_norm_w, k_norm_w, kv_cache, self.kv_dtype,
                             slot_mapping.reshape(B * qn), kv_scale,
                             self.q_out.view(B * qn, HQ, D), self.status, self.q_dtype,
                             self.q_scale)
        self.plan_step(seq_lens)
        return self.attend(self.q_out, kv_cache, kv_scale, block_table, seq_lens)



# ------------------------------------------------------------ prefill / mixed batches

class PrefillAttention:
    """Attention of packed new tokens (prompt chunks, prompts or decode
    tokens) over the paged cache: sequence b owns rows query_start[b] ..
    query_start[b+1]-1 of q and out and sees its history plus its new tokens
    up to each one.  The unit plan and counters are allocated once."""

    def __init__(self, batch, device="cuda", out_dtype=OUT_BF16, staging_pages=0):
        """``staging_pages`` > 0: E4M3 caches go through hpc_prefill_attn_staged
        with a BF16 staging buffer of that many pages (it needs the sum over
        sequences of ceil(seq_len / 64); see ``pages_for``)."""
        self.batch, self.out_dtype = batch, out_dtype
        self.unit_ptr = torch.zeros(batch + 1, dtype=torch.int32, device=device)
        self.counters = torch.zeros(2, dtype=torch.int32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.staging_pages = int(staging_pages)
        self.staging = self.page_ptr = None
        if self.staging_pages > 0:
            self.staging = torch.empty((self.staging_pages, 2, HKV, PAGE, D), dtype=torch.bfloat16,
                                       device=device)
            self.page_ptr = torch.zeros(batch + 1, dtype=torch.int32, device=device)

    @staticmethod
    def pages_for(seq_lens):
        """Staged pages a batch needs: the sum of ceil(L / 64) over its lengths (host values)."""
        return int(sum((int(L) + PAGE - 1) // PAGE for L in seq_lens))

    def plan(self, query_start):
        _want(query_start, "query_start", (torch.int32,), (self.batch + 1,))
        check("hpc_prefill_plan", _lib.lib().hpc_prefill_plan(
            _p(query_start), self.batch, _p(self.unit_ptr), _p(self.counters), _p(self.status),
            _stream()))

    def __call__(self, q, query_start, kv_cache, kv_dtype, kv_scale, block_table, seq_lens, out,
                 sm_scale=None):
        B = self.batch
        T = q.shape[0]
        _want(q, "q", _BF16, (T, HQ, D))
        _want(query_start, "query_start", (torch.int32,), (B + 1,))
        _want(kv_cache, "kv_cache", _cache_dtypes(kv_dtype))
        _want(block_table, "block_table", (torch.int32,))
        if block_table.dim() != 2 or block_table.shape[0] != B:
            raise ValueError("block_table must be [batch, max_blocks]")
        _want(seq_lens, "seq_lens", (torch.int32,), (B,))
        _want(out, "out", (_OUT_TORCH[self.out_dtype],), (T, HQ, D))
        scale = 1.0 / math.sqrt(D) if sm_scale is None else float(sm_scale)
        if self.staging is not None and kv_dtype == KV_FP8:
            check("hpc_prefill_attn_staged", _lib.lib().hpc_prefill_attn_staged(
                _p(q), T, _p(query_start), _p(kv_cache), kv_dtype, _p(kv_scale),
                kv_cache.shape[0], _p(block_table), block_table.shape[1], _p(seq_lens), B,
                _p(self.unit_ptr), _p(self.counters), _p(out), int(self.out_dtype), scale,
                _p(self.staging), self.staging_pages, _p(self.page_ptr), _p(self.status),
                _stream()))
            return out
        check("hpc_prefill_attn", _lib.lib().hpc_prefill_attn(
            _p(q), T, _p(query_start), _p(kv_cache), kv_dtype,
            _p(kv_scale if kv_dtype == KV_FP8 else None), kv_cache.shape[0], _p(block_table),
            block_table.shape[1], _p(seq_lens), B, _p(self.unit_ptr), _p(self.counters), _p(out),
            int(self.out_dtype), scale, _p(self.status), _stream()))
        return out


class HostInputs:
    """A step's host-side inputs in one pinned buffer, mirrored by one device
    buffer, so that they reach the device in a single copy.

    ``specs`` maps a name to (shape, dtype); each tensor starts on a 256-byte
    boundary of both buffers.  ``host[name]`` is the pinned view to fill,
    ``dev[name]`` the device view to pass to the calls, and ``upload()``
    issues the one host -> device copy on the current stream."""

    def __init__(self, specs, device="cuda"):
        self.offsets, total = {}, 0
        for name, (shape, dtype) in specs.items():
            nbytes = int(math.prod(shape)) * torch.empty((), dtype=dtype).element_size()
            self.offsets[name] = (total, nbytes, tuple(shape), dtype)
            total += (nbytes + 255) // 256 * 256
        self.nbytes = total
        self._host = torch.empty(total, dtype=torch.uint8)
        if torch.device(device).type == "cuda":
            self._host = self._host.pin_memory()
        self._dev = torch.empty(total, dtype=torch.uint8, device=device)
        self.host = {n: self._view(self._host, n) for n in self.offsets}
        self.dev = {n: self._view(self._dev, n) for n in self.offsets}

    def _view(self, buf, name):
        off, nbytes, shape, dtype = self.offsets[name]
        return buf[off:off + nbytes].view(dtype).view(shape)

    def upload(self):
        self._dev.copy_(self._host, non_blocking=True)
        return self.dev
