"""Helpers for the GPU parity tests: build/load the library once, and give
the oracle host copies of just the cache pages it needs."""

import math

import numpy as np
import pytest
import torch

from oracle import decode as od
from paged_gqa_decode_rope_gb300 import workloads

TOL_BF16_MAX = 2e-2
TOL_BF16_MEAN = 2e-3
TOL_FP8_MAX = 3e-2


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("the gpu-marked tests need a CUDA device")
    from paged_gqa_decode_rope_gb300.build import build_library
    build_library()


# host copies of device tensors (shared with the benchmark's CPU leg)
raw_cache_host = workloads.raw_cache_host
seq_view = workloads.host_pages
bf16_host = workloads.host_f64


def oracle_outputs(wl, q_bf16, seqs, heads=None, cache=None, kv_scale=None):
    """Oracle attention outputs [len(seqs), 64, 128] over the current cache for
    the given sequences (q taken from the BF16 q tensor)."""
    cache = wl.cache if cache is None else cache
    scale = wl.kv_scale.cpu().numpy().astype(np.float64) if kv_scale is None else kv_scale
    q = bf16_host(q_bf16)
    outs = []
    for b in seqs:
        L = int(wl.lengths[b])
        if L == 0:
            outs.append(np.zeros((64, 128)))
            continue
        sub, row = seq_view(cache, wl.block_table_np[b], L, wl.kv_dtype)
        outs.append(od.decode_attention(q[b], sub, row, L, wl.kv_dtype, scale[0], scale[1],
                                        heads=heads))
    return np.stack(outs)


def compare(got, want, max_tol, mean_tol=None, label=""):
    """Element-wise comparison over the finite (computed) oracle entries."""
    m = np.isfinite(want)
    assert m.any()
    err = np.abs(got[m] - want[m])
    assert np.all(np.isfinite(got[m])), "%s: non-finite outputs" % label
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= max_tol, "%s: max-abs %.3e > %.1e" % (label, mx, max_tol)
    if mean_tol is not None:
        assert mean <= mean_tol, "%s: mean-abs %.3e > %.1e" % (label, mean, mean_tol)
    return mx, mean


def sm_scale():
    return 1.0 / math.sqrt(128)
