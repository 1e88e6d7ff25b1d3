"""Plain, slow float64 CPU oracle for the paged GQA decode step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``paged_gqa_decode_rope_gb300``) never imports it, and the oracle shares no
code, constants or helpers with the CUDA kernels.

What it follows (all sources are public web pages about vLLM's HPC_ATTN
backend; every function cites the passage it restates):

* page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA Hopper"
  (24-ai.news, 2026-07-06):
  - intro of "Two new HPC backends in the vLLM ecosystem": model shape, 64 query
    heads, 8 KV heads, head_dim 128, 256K context;
  - "Why does dynamic scheduling matter for attention?": static split-KV
    schedules, the per-step length-proportional dealing of 64-token tiles, the
    fused RoPE -> QK-Norm -> KV-write prologue, BF16 and FP8 support.
* page "[vllm] Introducing the HPC-Ops attention backend" (analysis of vLLM PR
  #46020), "Code analysis" section 2 (the fused RoPE + QK-Norm + KV-cache-write
  custom op that mutates a caller-provided output) and "General lessons" item 1.

Modules:

* ``numerics``  -- BF16 round-to-nearest-even and the OCP FP8 E4M3 codec.
* ``decode``    -- RoPE (NeoX half rotation), RMSNorm, the paged cache write,
                   exact-softmax GQA decode attention, split partials and the
                   log-sum-exp merge, and the end-to-end decode step.
* ``plan``      -- the length-proportional split-KV planner and the static
                   equal-split comparator, plus a coverage checker.

Parity pins (tests/test_oracle_*.py) tie each function to something other than
itself: closed forms, invariants, library special cases (torch SDPA, torch
rms_norm, torch float8/bfloat16 casts), brute force on tiny inputs, and
hand-derived fixtures under tests/golden/.
"""

from . import numerics, decode, plan  # noqa: F401
