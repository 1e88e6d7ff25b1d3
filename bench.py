"""Benchmark of the GB300 paged GQA decode step.

One step = the whole hot path on one batch: fused RoPE/RMSNorm/KV-write
prologue -> length-proportional split-KV plan -> paged GQA decode attention
-> log-sum-exp merge.  The workload is the mixed-length decode batch
(1 x 131072 + 31 x 4096 tokens, 64 q heads / 8 KV heads, head_dim 128, BF16
KV in 64-token pages), whose KV (1.06 GB) is larger than L2, so no flush is
needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload tiny|uniform|mixed|mixed_fp8|heavy_tail] [--seed S]
                    [--no-static] [--no-cpu] [--cpu-seconds T] [--no-multi-token]
                    [--no-prefill] [--no-configs]
    python bench.py --prefill-only
    python bench.py --attn-only dynamic|static:S [--workload W] [--steps K] [--warmup W]

The JSON line also carries the roofline of the dominant kernel (the attention
with the merge fused in), the end-to-end rate through the public API with
host buffers, the CPU oracle baseline, the SM clocks seen while timing, the
dynamic-vs-static schedule comparison, the multi-token and prefill timings,
and every listed decode configuration (tiny, uniform, mixed, mixed FP8, heavy
tail) timed as a whole step, as a graph-replayed step and as the attention
alone (each section can be skipped with its flag).

Prints ONE JSON line on rank 0.  ``value`` is the KV+Q+O bytes of all ranks'
batches divided by the max-over-ranks device time of K steps (TB/s);
``ms_per_step`` is that time per step.  Under torchrun every rank runs its own
batch (weak scaling: the path shards by sequence with no collective).
``--impl reference`` times the float64 CPU oracle on a bounded sample of the
same workload (the slow baseline), on rank 0 only.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attn µs/layer-step & KV-read TB/s vs HBM peak on mixed-length batches"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "attn_traffic.json")
# the sources of the attention kernel; the committed traffic record holds their hash
ATTN_SRCS = [os.path.join(ROOT, "paged_gqa_decode_rope_gb300", "csrc", f)
             for f in ("attn.cu", "attn_kernel.cuh", "common.cuh")]


def _parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="mixed")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-static", action="store_true", help="skip the static-schedule comparison")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    p.add_argument("--no-multi-token", action="store_true", help="skip the multi-token decode timings")
    p.add_argument("--no-prefill", action="store_true", help="skip the prefill timings")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the timings of every listed decode configuration")
    p.add_argument("--prefill-only", action="store_true",
                   help="run only the prefill timings and print them as one JSON line")
    p.add_argument("--attn-only", default=None, metavar="SCHEDULE",
                   help="plan once under SCHEDULE ('dynamic' or 'static:S'), then time only the "
                        "attention launch (merge fused in) on the workload; one JSON line "
                        "(the form profiles are captured with)")
    p.add_argument("--q-len", type=int, default=1,
                   help="--attn-only: new tokens per sequence (multi-token decode, 1 .. 4)")
    p.add_argument("--q-dtype", default="bf16", choices=["bf16", "e4m3"],
                   help="--attn-only: the stored q (e4m3 needs an FP8 cache)")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--cpu-worker", default=None, help=argparse.SUPPRESS)
    return p.parse_args()


# ------------------------------------------------------------ clocks ---------

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1] or rows[-3:]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


# ------------------------------------------------------------ CPU oracle -----

def host_cores():
    """Host CPU cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _cpu_worker(spec_path):
    """Run the float64 oracle (prologue + attention) on this worker's units,
    one BLAS thread.  A unit is one (sequence, KV head): the prologue of the
    sequence and the attention of that KV head's 8 query heads.  The cache
    pages of every sequence sit in one shared-memory block written by the
    parent.  spec["steps"][s] lists this worker's units of step s; a step
    stops early once spec["seconds"] (if > 0) of its work is done.  Prints
    per-step bytes, seconds, tokens and unit counts as JSON."""
    import pickle
    from multiprocessing import shared_memory
    from oracle import decode as od
    with open(spec_path, "rb") as f:
        spec = pickle.load(f)
    shm = shared_memory.SharedMemory(name=spec["shm"])
    # the parent owns the block: attaching must not make this process's
    # resource tracker unlink it at exit
    from multiprocessing import resource_tracker
    resource_tracker.unregister(shm._name, "shared_memory")
    try:
        elem = 2 if spec["kv_dtype"] == 0 else 1
        dt = np.uint16 if spec["kv_dtype"] == 0 else np.uint8
        seqs = {}
        for b, (off, shape) in spec["pages"].items():
            seqs[b] = np.ndarray(shape, dtype=dt, buffer=shm.buf, offset=off)
        res = []
        for units in spec["steps"]:
            done_bytes = done_tok = n = 0
            t_total = 0.0
            for b, h in units:
                it = spec["seqs"][b]
                L = it["L"]
                cache = seqs[b]
                t0 = time.perf_counter()
                od.decode_step(it["q"], it["k"], it["v"], [L - 1], spec["qw"], spec["kw"], cache,
                               np.arange(cache.shape[0])[None, :], [L], [L - 1], spec["kv_dtype"],
                               spec["scale"], heads=range(8 * h, 8 * h + 8))
                t_total += time.perf_counter() - t0
                done_tok += L
                done_bytes += L * 128 * 2 * elem           # one KV head's K and V
                n += 1
                if 0 < spec["seconds"] <= t_total:
                    break
            res.append({"bytes": done_bytes, "seconds": t_total, "tokens": done_tok, "units": n})
        print(json.dumps(res))
    finally:
        del seqs
        shm.close()


def run_oracle_steps(wl, steps, seconds, workers=None):
    """Time the oracle on the host cores over ``steps`` (lists of sequence ids).

    Every sequence of a step is cut into its 8 KV heads; the units are dealt,
    longest first, to the least-loaded of ``workers`` processes (default: all
    host cores), each with one BLAS thread, which run concurrently.  A step's
    time is its slowest worker's time; its bytes, tokens and units are summed.
    Returns one dict per step and the number of workers used."""
    import pickle
    import tempfile
    from multiprocessing import shared_memory
    from paged_gqa_decode_rope_gb300.workloads import host_f64, host_pages
    workers = max(1, workers or host_cores())
    q, k, v = host_f64(wl.q), host_f64(wl.k), host_f64(wl.v)
    ids = sorted({b for ids in steps for b in ids if int(wl.lengths[b]) > 0})
    raw = {b: host_pages(wl.cache, wl.block_table_np[b], int(wl.lengths[b]), wl.kv_dtype)[0]
           for b in ids}
    total = sum(r.nbytes for r in raw.values())
    shm = shared_memory.SharedMemory(create=True, size=max(total, 1))
    paths, procs = [], []
    try:
        pages, off = {}, 0
        for b in ids:
            dst = np.ndarray(raw[b].shape, dtype=raw[b].dtype, buffer=shm.buf, offset=off)
            dst[...] = raw[b]
            pages[b] = (off, raw[b].shape)
            off += raw[b].nbytes
            del dst
        del raw
        per_worker = [[[] for _ in steps] for _ in range(workers)]
        for s, step_ids in enumerate(steps):
            load = [0] * workers
            units = sorted(((b, h) for b in step_ids if b in pages for h in range(8)),
                           key=lambda u: -int(wl.lengths[u[0]]))
            for b, h in units:
                w = load.index(min(load))
                per_worker[w][s].append((b, h))
                load[w] += int(wl.lengths[b])
        common = {"kv_dtype": wl.kv_dtype, "seconds": seconds, "shm": shm.name,
                  "scale": wl.kv_scale.cpu().numpy().astype(np.float64),
                  "qw": host_f64(wl.q_norm_w), "kw": host_f64(wl.k_norm_w)}
        env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
        for w in range(workers):
            mine = sorted({b for st in per_worker[w] for b, _ in st})
            spec = dict(common, steps=per_worker[w], pages={b: pages[b] for b in mine},
                        seqs={b: {"L": int(wl.lengths[b]), "q": q[b:b + 1], "k": k[b:b + 1],
                                  "v": v[b:b + 1]} for b in mine})
            with tempfile.NamedTemporaryFile(suffix=".pkl", delete=False) as f:
                pickle.dump(spec, f)
                paths.append(f.name)
            procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__), "--cpu-worker",
                                           f.name], stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                          text=True, env=env))
        outs = []
        for p in procs:
            o, e = p.communicate(timeout=900)
            if p.returncode != 0:
                raise RuntimeError("oracle worker failed: " + e[-2000:])
            outs.append(json.loads(o.strip().splitlines()[-1]))
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
        for path in paths:
            os.unlink(path)
        shm.close()
        shm.unlink()
    res = []
    for s in range(len(steps)):
        rows = [o[s] for o in outs]
        res.append({"bytes": sum(r["bytes"] for r in rows), "seconds": max(r["seconds"] for r in rows),
                    "tokens": sum(r["tokens"] for r in rows) // 8, "units": sum(r["units"] for r in rows)})
    return res, workers


def cpu_baseline(wl, seconds):
    """The oracle on a bounded, seeded random sample of the workload's
    sequences, on all host cores (about ``seconds`` of work per core at most)."""
    order = np.random.default_rng(123).permutation(wl.batch).tolist()
    picked, est = [], 0
    for b in order:                  # enough sequences for the time budget
        picked.append(b)
        est += int(wl.lengths[b])
        if est > 400000 * host_cores():
            break
    res, workers = run_oracle_steps(wl, [picked], seconds)
    return dict(res[0], workers=workers, seqs=len(picked))


# ------------------------------------------------------------ helpers --------

def _load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def attn_src_sha256():
    """One hash over the attention kernel's sources (in a fixed order)."""
    h = hashlib.sha256()
    for p in ATTN_SRCS:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _traffic_record():
    """Per-launch DRAM bytes of the attention kernel from the committed ncu
    summary, if it was taken on the current kernel sources; else None."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as f:
        rec = json.load(f)
    if rec.get("attn_src_sha256") != attn_src_sha256():
        return None
    return rec


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, ws, device):
    """The largest of x over the ranks of the job (x itself on one rank)."""
    if ws == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(seed, rank):
    """Every rank draws its own batch of the workload (weak scaling)."""
    return seed + rank


def whole_job_tbps(ws, bytes_per_rank_step, steps, elapsed_ms):
    """Bytes of all ranks' batches over the slowest rank's time, in TB/s."""
    return ws * bytes_per_rank_step * steps / (elapsed_ms * 1e-3) / 1e12


# ------------------------------------------------------------ reference ------

def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import torch
    from paged_gqa_decode_rope_gb300.workloads import Workload
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = Workload(args.workload, seed=args.seed, device=dev)
    # each step: the oracle on one bounded slice of the workload, one sequence
    # of at most 8192 tokens, round-robin (float64, one thread)
    short = [b for b in range(wl.batch) if 0 < wl.lengths[b] <= 8192] or [int(np.argmin(wl.lengths))]
    steps = [[short[s % len(short)]] for s in range(args.warmup + args.steps)]
    res, workers = run_oracle_steps(wl, steps, 0.0, workers=min(8, host_cores()))
    res = res[args.warmup:]
    t = sum(r["seconds"] for r in res)
    value = sum(r["bytes"] for r in res) / t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": args.workload + ": " + _describe(wl),
                       "sample": "one sequence of <= 8192 tokens per step"},
            "cpu_baseline": {"value": value, "unit": "TB/s", "cores": workers, "host_cores": host_cores(),
                             "kind": "oracle",
                             "sample": "one <=8192-token sequence per step, prologue + attention, its 8 "
                                       "KV heads on %d processes (one BLAS thread each)" % workers},
            "e2e": {"value": value, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ------------------------------------------------------------ ours -----------

def run_ours(args):
    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    from paged_gqa_decode_rope_gb300.build import build_library
    build_library()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload

    wl = Workload(args.workload, seed=rank_seed(args.seed, rank))
    cos_sin = ops.rope_cos_sin_cache(wl.max_pos + 1)
    step = ops.DecodeStep(wl.batch, wl.kv_dtype, wl.max_blocks)
    stream = torch.cuda.current_stream()
    algo_bytes = wl.kv_bytes() + wl.qo_bytes()

    def one_step():
        # the whole path in two launches: prologue + plan, then attention with
        # the merge fused in (a programmatic dependent of the first)
        step(wl.q, wl.k, wl.v, wl.positions, cos_sin, wl.q_norm_w, wl.k_norm_w, wl.cache,
             wl.slot_mapping, wl.kv_scale, wl.block_table, wl.seq_lens)

    # the clock sampler starts before the warm-up, so that the timed steps
    # follow warm steps directly (no idle gap in which the clocks could drop)
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    for _ in range(max(3, args.warmup)):
        one_step()
    torch.cuda.synchronize()
    if int(step.status.item()) != 0:
        raise RuntimeError("device status %d during warm-up" % int(step.status.item()))
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    t_start.record(stream)
    for s in range(args.steps):
        one_step()
    t_end.record(stream)
    torch.cuda.synchronize()
    # the dominant kernel alone (attention + fused merge), same stream and
    # inputs, K launches back to back: its mean duration per launch
    a_start, a_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_start.record(stream)
    for s in range(args.steps):
        step.attend(step.q_out, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)
    a_end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    if ws > 1:
        torch.distributed.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    attn_ms = a_start.elapsed_time(a_end) / args.steps
    if int(step.status.item()) != 0:
        raise RuntimeError("device status %d during timing" % int(step.status.item()))
    if sampler:
        sampler.stop()
        clocks = sampler.summary(wall0, wall1)
    elapsed_ms = max_over_ranks(elapsed_ms, ws, "cuda")
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_tbps(ws, algo_bytes, args.steps, elapsed_ms)

    # end to end through the public API with host buffers: H2D of the step's
    # inputs from pinned memory, the four calls, D2H of the output
    # (the inputs sit back to back in one pinned buffer: one copy per step)
    names = ("q", "k", "v", "positions", "slot_mapping", "seq_lens", "block_table")
    staged = ops.HostInputs({n: (tuple(getattr(wl, n).shape), getattr(wl, n).dtype) for n in names})
    for n in names:
        staged.host[n].copy_(getattr(wl, n).cpu())
    h2d = sum(staged.host[n].numel() * staged.host[n].element_size() for n in names)
    out_host = torch.empty_like(step.out, device="cpu").pin_memory()
    d2h = out_host.numel() * out_host.element_size()
    e2e_steps = max(10, min(args.steps, 500))

    def e2e_step():
        d = staged.upload()
        out = step(d["q"], d["k"], d["v"], d["positions"], cos_sin, wl.q_norm_w, wl.k_norm_w,
                   wl.cache, d["slot_mapping"], wl.kv_scale, d["block_table"], d["seq_lens"])
        out_host.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, ws, "cuda")
    e2e_value = whole_job_tbps(ws, algo_bytes, 1, e2e_ms)

    # dynamic vs static equal split on the same kernels (attention + merge)
    sched = None
    if rank == 0 and not args.no_static:
        sched = schedule_comparison(ops, wl, stream)
    mt = None
    if rank == 0 and not args.no_multi_token:
        mt = multi_token_times(ops, wl, stream)
        if wl.kv_dtype == 0 and args.workload == "mixed":
            # the same mix over an E4M3 cache, so that both cache types are in the line
            wl8 = Workload("mixed_fp8", seed=rank_seed(args.seed, rank))
            mt = {"mixed BF16": mt, "mixed FP8": multi_token_times(ops, wl8, stream)}
            del wl8
            torch.cuda.empty_cache()
    pre = prefill_times(ops, stream) if rank == 0 and not args.no_prefill else None
    cfgs = config_times(ops, stream) if rank == 0 and not args.no_configs else None

    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return

    peak_gbs, peak_kind = _load_peaks()
    achieved_gbs = algo_bytes / (attn_ms * 1e-3) / 1e9
    rec = _traffic_record()
    roofline = {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": peak_gbs, "unit": "GB/s",
                "frac": round(achieved_gbs / peak_gbs, 4),
                "traffic": rec["bytes_per_launch"] if rec else None,
                "peak_kind": peak_kind,
                "kernel": "decode_attn_kernel<%s> (merge fused)" % ("bf16" if wl.kv_dtype == 0 else "fp8"),
                "algorithmic_bytes_per_launch": algo_bytes, "attn_us": round(attn_ms * 1e3, 2),
                "frac_of_8TBps": round(achieved_gbs / 8000.0, 4)}
    cpu = None
    if ws == 1 and not args.no_cpu:
        r = cpu_baseline(wl, args.cpu_seconds)
        cpu_tbps = r["bytes"] / r["seconds"] / 1e12
        cpu = {"value": cpu_tbps, "unit": "TB/s", "cores": r["workers"], "host_cores": host_cores(),
               "kind": "oracle",
               "sample": "%d of %d sequences (%d tokens), float64 prologue + attention, (sequence, "
                         "KV head) units on %d processes of one BLAS thread each"
                         % (r["seqs"], wl.batch, r["tokens"], r["workers"]),
               "seconds": round(r["seconds"], 2),
               "us_per_layer_step_extrapolated": round(wl.kv_bytes() / (r["bytes"] / r["seconds"]) * 1e6, 1)}
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "TB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "us_per_layer_step": round(ms_per_step * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.kv_dtype == 0 else "fp8_e4m3",
        "data": "synthetic (seeded N(0,1) q/k/v and history, random page permutation, NaN-filled unused slots)",
        "config": {"workload": args.workload + ": " + _describe(wl), "global_batch": wl.batch * ws,
                   "tokens": wl.tokens, "kv_bytes": wl.kv_bytes(), "l2": "inputs larger than L2 (no flush)",
                   "step": "prologue + plan (one launch) -> attention + merge (PDL launch)",
                   "parallelism": "dp%d (sequences per GPU)" % ws},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 4), "unit": "TB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5)},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "schedules": sched,
        "multi_token": mt,
        "prefill": pre,
        "configs": cfgs,
    }
    print(json.dumps(line))


def _describe(wl):
    L = wl.lengths
    kv = "BF16" if wl.kv_dtype == 0 else "FP8-E4M3"
    if len(set(L.tolist())) <= 2:
        parts = []
        for x in sorted(set(L.tolist()), reverse=True):
            parts.append("%dx%d" % (int((L == x).sum()), x))
        return " + ".join(parts) + " tokens, 64q/8kv, d128, %s KV, 64-token pages" % kv
    return "%d seqs, %d tokens, 64q/8kv, d128, %s KV, 64-token pages" % (wl.batch, wl.tokens, kv)


def prefill_times(ops, stream, reps=10):
    """Prefill attention: 4 whole prompts of 4096 tokens and 8 chunks of 512
    new tokens after 7680-token histories on a BF16 cache, and the prompts on
    an E4M3 cache, directly and with the pages staged to BF16 first (the
    staging launches timed with the attention); CUDA events over ``reps``
    calls.  Flops 4 * 64 * 128 per query token and visible key (the causal
    triangle counted exactly)."""
    import torch
    from paged_gqa_decode_rope_gb300.workloads import Workload
    res = {}
    peaks = _load_peak_tflops()
    for name, lengths, q_lens, kvd, staged in (
            ("4 prompts x 4096", [4096] * 4, [4096] * 4, 0, False),
            ("8 chunks of 512 after 7680", [8192] * 8, [512] * 8, 0, False),
            ("4 prompts x 4096, E4M3 cache", [4096] * 4, [4096] * 4, 1, False),
            ("4 prompts x 4096, E4M3 cache staged to BF16", [4096] * 4, [4096] * 4, 1, True)):
        wl = Workload("custom", seed=21, lengths=lengths, kv_dtype=kvd, include_new_token=True)
        qs = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
        g = torch.Generator(device="cuda").manual_seed(1)
        q = torch.randn((int(qs[-1]), 64, 128), generator=g, device="cuda").to(torch.bfloat16)
        qst = torch.as_tensor(qs, device="cuda")
        out = torch.empty_like(q)
        pf = ops.PrefillAttention(wl.batch, staging_pages=ops.PrefillAttention.pages_for(lengths)
                                  if staged else 0)
        pf.plan(qst)
        for _ in range(2):
            pf(q, qst, wl.cache, kvd, wl.kv_scale, wl.block_table, wl.seq_lens, out)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            pf(q, qst, wl.cache, kvd, wl.kv_scale, wl.block_table, wl.seq_lens, out)
        b.record(stream)
        torch.cuda.synchronize()
        if int(pf.status.item()) != 0:
            raise RuntimeError("device status %d in the prefill run" % int(pf.status.item()))
        us = a.elapsed_time(b) / reps * 1e3
        keys = sum(sum(L - n + i + 1 for i in range(n)) for L, n in zip(lengths, q_lens))
        flops = 4.0 * 64 * 128 * keys
        tf = flops / us / 1e6
        res[name] = {"us": round(us, 1), "TFLOP/s": round(tf, 1),
                     "frac_of_bf16_peak": round(tf / peaks, 4) if peaks else None}
    return res


def run_prefill_only():
    """The prefill timings alone (one GPU), as one JSON line."""
    import torch
    sys.path.insert(0, ROOT)
    import __graft_entry__
    __graft_entry__.build()
    from paged_gqa_decode_rope_gb300 import ops
    torch.cuda.set_device(0)
    print(json.dumps({"prefill": prefill_times(ops, torch.cuda.current_stream())}))


def run_attn_only(args):
    """One workload, one plan, W + K attention launches (merge fused in):
    the launches a profile of one schedule captures."""
    import torch
    sys.path.insert(0, ROOT)
    import __graft_entry__
    __graft_entry__.build()
    from paged_gqa_decode_rope_gb300 import ops
    from paged_gqa_decode_rope_gb300.workloads import Workload
    torch.cuda.set_device(0)
    sched = args.attn_only
    if sched.startswith("static:"):
        schedule = ("static", int(sched.split(":", 1)[1]))
    elif sched == "dynamic":
        schedule = "dynamic"
    else:
        raise SystemExit("--attn-only takes 'dynamic' or 'static:S'")
    wl = Workload(args.workload, seed=args.seed, include_new_token=True)
    qn = args.q_len
    if qn == 1 and args.q_dtype == "bf16":
        step = ops.DecodeStep(wl.batch, wl.kv_dtype, wl.max_blocks, schedule=schedule)
        q = wl.q
    else:
        if schedule != "dynamic":
            raise SystemExit("multi-token and E4M3-q runs take the dynamic plan")
        # random q of the multi-token layout (E4M3: codes of q / (max|q| / 448))
        g = torch.Generator(device="cuda").manual_seed(qn)
        q = torch.randn((wl.batch, qn, 64, 128), generator=g, device="cuda")
        qs = float(q.abs().max()) / 448.0
        qd = ops.Q_FP8 if args.q_dtype == "e4m3" else ops.Q_BF16
        q = (q / qs).to(torch.float8_e4m3fn).view(torch.uint8) if qd == ops.Q_FP8 else q.to(torch.bfloat16)
        step = ops.DecodeStepEx(wl.batch, wl.kv_dtype, wl.max_blocks, q_len=qn, q_dtype=qd, q_scale=qs)
    step.plan_step(wl.seq_lens)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)
    b.record(stream)
    torch.cuda.synchronize()
    st = int(step.status.item())
    if st != 0:
        raise RuntimeError("device status %d" % st)
    us = a.elapsed_time(b) / args.steps * 1e3
    nbytes = wl.kv_bytes() + qn * wl.qo_bytes()
    print(json.dumps({"attn_only": sched, "q_len": qn, "q_dtype": args.q_dtype,
                      "workload": args.workload + ": " + _describe(wl),
                      "queues": step.plan.num_ctas, "attn_us": round(us, 2),
                      "TBps": round(nbytes / us / 1e6, 4), "launches": args.warmup + args.steps}))


def _load_peak_tflops():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for k in ("bf16_tflops", "bf16_tflops_burst"):
            if k in d:
                return float(d[k])
    except (OSError, ValueError):
        pass
    return None


def multi_token_times(ops, wl, stream, reps=200):
    """Multi-token decode on the same batch: the attention with the merge fused
    in for q_len = 2 and 4 new tokens per sequence (the cache and lengths of
    the workload, random BF16 q), and on an FP8 cache also with an E4M3 q
    (q_len 1, 2, 4; q quantised with scale max|q|/448 as input synthesis),
    CUDA events over ``reps`` launches.  Bytes
    are the KV bytes plus q_len times the Q + O bytes; flops 4 * 64 * 128 per
    query token and key."""
    import torch
    out = {}
    peak_gbs, _ = _load_peaks()
    runs = [(qn, ops.Q_BF16) for qn in (2, 4)]
    if wl.kv_dtype == 1:                       # an FP8 cache also takes an E4M3 q
        runs += [(qn, ops.Q_FP8) for qn in (1, 2, 4)]
    for qn, qd in runs:
        g = torch.Generator(device="cuda").manual_seed(qn)
        q = torch.randn((wl.batch, qn, 64, 128), generator=g, device="cuda")
        qs = float(q.abs().max()) / 448.0
        q = (q / qs).to(torch.float8_e4m3fn).view(torch.uint8) if qd == ops.Q_FP8 else q.to(torch.bfloat16)
        step = ops.DecodeStepEx(wl.batch, wl.kv_dtype, wl.max_blocks, q_len=qn, q_dtype=qd, q_scale=qs)
        step.plan_step(wl.seq_lens)
        for _ in range(5):
            step.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            step.attend(q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)
        b.record(stream)
        torch.cuda.synchronize()
        if int(step.status.item()) != 0:
            raise RuntimeError("device status %d in the multi-token run" % int(step.status.item()))
        us = a.elapsed_time(b) / reps * 1e3
        nbytes = wl.kv_bytes() + qn * wl.qo_bytes()
        flops = 4.0 * 64 * 128 * qn * wl.tokens
        out["q_len=%d%s" % (qn, ", E4M3 q" if qd == ops.Q_FP8 else "")] = {
                                "attn_us": round(us, 2), "GB/s": round(nbytes / us / 1e3, 1),
                                "frac": round(nbytes / us / 1e3 / peak_gbs, 4),
                                "TFLOP/s": round(flops / us / 1e6, 2)}
    return out


CONFIGS = ("tiny", "uniform", "mixed", "mixed_fp8", "heavy_tail")
L2_BYTES = 129 * 1024 * 1024


def config_times(ops, stream, seed=0, reps=100):
    """Every listed decode configuration at its full size, in the launch
    configuration of the headline: the whole step (prologue + plan in one
    launch, attention with the merge fused in as its programmatic dependent),
    eagerly and replayed from a CUDA graph, and the attention launch alone;
    CUDA events over ``reps`` back-to-back calls each.  A batch whose bytes
    fit twice in L2 (the tiny one) is timed call by call with a write of
    twice the L2 size between calls, outside the events.  Bytes are the
    KV + Q + O bytes of the batch; ``frac`` is the attention's rate over the
    measured copy bandwidth."""
    import torch
    from paged_gqa_decode_rope_gb300.workloads import Workload
    peak_gbs, peak_kind = _load_peaks()
    res = {}
    for name in CONFIGS:
        wl = Workload(name, seed=seed)
        cos_sin = ops.rope_cos_sin_cache(wl.max_pos + 1)
        step = ops.DecodeStep(wl.batch, wl.kv_dtype, wl.max_blocks)
        nbytes = wl.kv_bytes() + wl.qo_bytes()
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda") \
            if nbytes < 2 * L2_BYTES else None

        def one_step():
            step(wl.q, wl.k, wl.v, wl.positions, cos_sin, wl.q_norm_w, wl.k_norm_w, wl.cache,
                 wl.slot_mapping, wl.kv_scale, wl.block_table, wl.seq_lens)

        def attend():
            step.attend(step.q_out, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)

        def timed(fn):
            """Mean µs per call of fn over ``reps`` calls."""
            if flush is None:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(reps):
                    fn()
                b.record(stream)
                torch.cuda.synchronize()
                return a.elapsed_time(b) / reps * 1e3
            total = 0.0
            for _ in range(reps):
                flush.fill_(1.0)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                torch.cuda.synchronize()
                total += a.elapsed_time(b)
            return total / reps * 1e3

        for _ in range(3):
            one_step()
        torch.cuda.synchronize()
        step_us = timed(one_step)
        attn_us = timed(attend)
        # the same step captured once in a CUDA graph and replayed
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream()
        cs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cs):
            one_step()
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=cs):
                one_step()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        graph_us = timed(g.replay)
        st = int(step.status.item())
        if st != 0:
            raise RuntimeError("device status %d in config %s" % (st, name))
        res[name] = {
            "workload": _describe(wl), "tokens": wl.tokens, "bytes": nbytes,
            "step_us": round(step_us, 2), "step_graph_us": round(graph_us, 2),
            "attn_us": round(attn_us, 2),
            "step_TBps": round(nbytes / step_us / 1e6, 4),
            "attn_TBps": round(nbytes / attn_us / 1e6, 4),
            "frac": round(nbytes / attn_us / 1e3 / peak_gbs, 4),
            "step_frac": round(nbytes / step_us / 1e3 / peak_gbs, 4),
            "frac_of_8TBps": round(nbytes / attn_us / 8e6, 4),
            "l2": "flushed between calls" if flush is not None else "inputs larger than L2",
        }
        del g, step, wl, cos_sin, flush
        torch.cuda.empty_cache()
    return {"unit": "us", "peak_GBps": peak_gbs, "peak_kind": peak_kind, "reps": reps, "seed": seed,
            "step": "prologue + plan (one launch) -> attention + merge (PDL launch)", "by_config": res}


def schedule_comparison(ops, wl, stream):
    """Attention + merge under the dynamic plan and static equal splits."""
    import torch

    def time_step(step, reps=30):
        step.plan_step(wl.seq_lens)
        for _ in range(5):
            step.attend(step_q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            step.attend(step_q, wl.cache, wl.kv_scale, wl.block_table, wl.seq_lens)
        b.record(stream)
        torch.cuda.synchronize()
        assert int(step.status.item()) == 0
        return a.elapsed_time(b) / reps * 1e3

    def occupancy(step):
        clock = torch.zeros((step.plan.num_ctas, 3), dtype=torch.int64, device="cuda")
        ops.decode_attn_profiled(step_q, wl.cache, wl.kv_dtype, wl.kv_scale, wl.block_table,
                                 wl.seq_lens, step.plan, step.partial_o, step.partial_lse,
                                 step.status, clock)
        torch.cuda.synchronize()
        return ops.cta_occupancy(clock)

    step_q = wl.q
    dyn = ops.DecodeStep(wl.batch, wl.kv_dtype, wl.max_blocks)
    t_dyn = time_step(dyn)
    occ = {"dynamic": occupancy(dyn)}
    nopool = ops.DecodeStep(wl.batch, wl.kv_dtype, wl.max_blocks, pool_chunks=0)
    t_nopool = time_step(nopool)
    occ["dynamic, no pool"] = occupancy(nopool)
    del nopool
    n_ctas = ops.num_ctas(wl.kv_dtype)
    heuristic = max(1, -(-n_ctas // (wl.batch * 8)))
    sweep = {}
    for S in sorted({1, 2, 4, 8, 16, 32, 64, heuristic}):
        st = ops.DecodeStep(wl.batch, wl.kv_dtype, wl.max_blocks, schedule=("static", S))
        sweep[S] = round(time_step(st), 2)
        occ["static S=%d" % S] = occupancy(st)
        del st
    best_S = min(sweep, key=sweep.get)
    occ = {k: v for k, v in occ.items()
           if k in ("dynamic", "dynamic, no pool", "static S=%d" % heuristic, "static S=%d" % best_S)}
    return {"unit": "us (attn + merge)", "dynamic": round(t_dyn, 2),
            "dynamic_no_pool": round(t_nopool, 2), "pool_chunks": ops.POOL_CHUNKS,
            "static_heuristic_splits": heuristic, "static_heuristic": sweep[heuristic],
            "static_best_splits": best_S, "static_best": sweep[best_S],
            "speedup_vs_heuristic": round(sweep[heuristic] / t_dyn, 3),
            "speedup_vs_best_static": round(sweep[best_S] / t_dyn, 3),
            "static_sweep": {str(k): v for k, v in sweep.items()},
            "occupancy": occ}


def main():
    args = _parse()
    if args.cpu_worker:
        _cpu_worker(args.cpu_worker)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    if args.prefill_only:
        run_prefill_only()
        return
    if args.attn_only:
        run_attn_only(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
