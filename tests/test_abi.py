"""The C-ABI library loads and exports every symbol include/hpc_decode.h
declares; host-side argument checks work without a GPU (no kernel runs)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hpc_decode.h")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:int|int32_t)\s+(hpc_\w+)\s*\(", text, flags=re.M)


@pytest.fixture(scope="module")
def lib():
    from paged_gqa_decode_rope_gb300.build import build_library
    build_library()
    from paged_gqa_decode_rope_gb300 import _lib
    return _lib.lib()


def test_header_declares_the_four_calls():
    names = header_functions()
    for n in ("hpc_rope_norm_kvwrite", "hpc_decode_plan", "hpc_decode_attn", "hpc_merge"):
        assert n in names


def test_binding_covers_the_header():
    from paged_gqa_decode_rope_gb300 import _lib
    assert set(header_functions()) == set(_lib.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_host_argument_checks(lib):
    from paged_gqa_decode_rope_gb300._lib import (Plan, PlanParams, HPC_ERR_INVALID_ARG,
                                                  HPC_ERR_UNSUPPORTED)
    NULL = None
    fake = ctypes.c_void_p(4096)       # never dereferenced on the host
    assert lib.hpc_plan_capacity(32, 152, 0) == 152 + 256
    assert lib.hpc_plan_capacity(32, 152, 6) == 152 * 7 + 256
    assert lib.hpc_rope_cos_sin_cache(1e6, 0, fake, NULL) == HPC_ERR_INVALID_ARG
    assert lib.hpc_rope_cos_sin_cache(1e6, 10, NULL, NULL) == HPC_ERR_INVALID_ARG
    # unknown KV dtype, null pointers, negative batch
    args = [fake] * 5 + [16, fake, fake, 1e-6, fake, 7, 4, fake, fake, fake, 1, fake, NULL]
    assert lib.hpc_rope_norm_kvwrite(*args) == HPC_ERR_UNSUPPORTED
    args[10] = 0
    args[0] = NULL
    assert lib.hpc_rope_norm_kvwrite(*args) == HPC_ERR_INVALID_ARG
    args[0] = fake
    args[15] = -1
    assert lib.hpc_rope_norm_kvwrite(*args) == HPC_ERR_INVALID_ARG
    args[15] = 0
    assert lib.hpc_rope_norm_kvwrite(*args) == 0          # empty batch: nothing to launch
    plan = Plan(4096, 4096, 4096, 4096, 4096, 4096, 100, 10)
    st = fake
    P = lambda a, b, c: ctypes.byref(PlanParams(a, b, c))
    assert lib.hpc_decode_plan(fake, 4, 8, P(0, 0, 1), ctypes.byref(plan), st, NULL) == HPC_ERR_INVALID_ARG
    assert lib.hpc_decode_plan(fake, 4, 8, P(1, 65, 1), ctypes.byref(plan), st, NULL) == HPC_ERR_INVALID_ARG
    assert lib.hpc_decode_plan(fake, 4, 8, P(1, 4, 0), ctypes.byref(plan), st, NULL) == HPC_ERR_INVALID_ARG
    assert lib.hpc_decode_plan(fake, 9000, 8, None, ctypes.byref(plan), st, NULL) == HPC_ERR_UNSUPPORTED
    assert lib.hpc_decode_plan(NULL, 4, 8, None, ctypes.byref(plan), st, NULL) == HPC_ERR_INVALID_ARG
    wide = Plan(4096, 4096, 4096, 4096, 4096, 4096, 100, 16385)   # above HPC_MAX_PLAN_CTAS
    assert lib.hpc_decode_plan(fake, 4, 8, None, ctypes.byref(wide), st, NULL) == HPC_ERR_UNSUPPORTED
    bad = Plan(4096, 4096, 4096, 0, 4096, 4096, 100, 10)  # no home_end array
    assert lib.hpc_decode_plan(fake, 4, 8, None, ctypes.byref(bad), st, NULL) == HPC_ERR_INVALID_ARG
    # static plan: num_ctas must be batch * 8 * splits
    assert lib.hpc_decode_plan_static(fake, 4, 8, 2, ctypes.byref(plan), st, NULL) == HPC_ERR_INVALID_ARG
    # attention: misaligned cache, too many blocks, unknown dtype
    a = [fake, ctypes.c_void_p(4097), 0, fake, 100, fake, 8, fake, 4, ctypes.byref(plan),
         fake, fake, 0.088, st, NULL]
    assert lib.hpc_decode_attn(*a) == HPC_ERR_INVALID_ARG
    a[1] = fake
    a[4] = 1 << 22
    assert lib.hpc_decode_attn(*a) == HPC_ERR_UNSUPPORTED
    a[4] = 100
    a[2] = 3
    assert lib.hpc_decode_attn(*a) == HPC_ERR_UNSUPPORTED
    # partial buffers not 16-byte aligned (they are written and read 16 bytes at a time)
    a[2] = 0
    for k in (10, 11):
        b = list(a)
        b[k] = ctypes.c_void_p(fake.value + 4)
        assert lib.hpc_decode_attn(*b) == HPC_ERR_INVALID_ARG
    assert lib.hpc_merge(ctypes.c_void_p(fake.value + 4), fake, ctypes.byref(plan), 4, fake,
                         NULL) == HPC_ERR_INVALID_ARG
    assert lib.hpc_merge(NULL, fake, ctypes.byref(plan), 4, fake, NULL) == HPC_ERR_INVALID_ARG
    assert lib.hpc_merge(fake, fake, ctypes.byref(plan), 0, fake, NULL) == 0
    # the wait self-test: limit outside 1 us .. 1 s, or no status word
    assert lib.hpc_selftest_wait_timeout(10, fake, NULL, NULL) == HPC_ERR_INVALID_ARG
    assert lib.hpc_selftest_wait_timeout(2 * 10 ** 9, fake, NULL, NULL) == HPC_ERR_INVALID_ARG
    assert lib.hpc_selftest_wait_timeout(10 ** 6, NULL, NULL, NULL) == HPC_ERR_INVALID_ARG
    # the queue count for multi-token decode: q_len 1 .. 4, a q dtype it knows, a result slot
    n = ctypes.c_int32(0)
    assert lib.hpc_decode_num_queues(1, 0, 0, ctypes.byref(n)) == HPC_ERR_INVALID_ARG
    assert lib.hpc_decode_num_queues(1, 5, 0, ctypes.byref(n)) == HPC_ERR_INVALID_ARG
    assert lib.hpc_decode_num_queues(1, 2, 7, ctypes.byref(n)) == HPC_ERR_INVALID_ARG
    assert lib.hpc_decode_num_queues(1, 2, 1, NULL) == HPC_ERR_INVALID_ARG
