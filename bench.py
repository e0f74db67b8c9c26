#!/usr/bin/env python
"""Benchmark of the paged decode hot path on GB300.

One step = one decode step of the whole hot path over one batch: the host
block manager appends one token to every sequence (slots, copy-on-write pairs,
block tables) and plans the attention's work list, then pk_copy_blocks (when
pairs exist) and pk_paged_attention_decode_append -- the attention with the
slot scatter of the step's new K/V fused into the same launch (and its
log-sum-exp merge when it splits). --no-fuse runs pk_reshape_and_cache as its
own kernel; --grid / --no-order launch the (sequence, partition) grid.

Device timing (``value``): the host side of a window of steps is prepared and
uploaded before the timed region, so inputs are resident in HBM; each timed
step is bracketed by CUDA events on the launching stream, and the L2 is
flushed (a write of twice its size) between steps, outside the events.
``e2e`` times the same steps through the public API from pinned host buffers:
the host block-manager append, the launch, the kernels reading the step's
inputs from host memory and writing the output back across the host link,
and the synchronise are all inside the timer.
``swap`` (after the steps) times preemption by swapping: half the batch's
blocks to a pinned host pool and back, one pk_swap_blocks launch per
direction, beside a contiguous copy-engine copy of the same bytes.
``allocator_sim`` (host) is the allocator policy table on the seeded traces.
``configs`` (a default single-GPU run of the default workload) times the
other target configurations the same way, each with its own roofline
fraction: the 8B-like GQA batch, the 32K-context batch (the planner's
partitions and the 512-token partitions), and the shared-prefix batch at
block sizes 8 / 16 / 32, per sequence and as cascade attention.

Metric: algorithmic K/V bytes read per step (sum over sequences of
context_len * Hk * head_dim * 2 bytes * 2 for K and V) per second.

``--impl reference`` times the CPU oracle on the host cores instead (a
bounded sample of each step's attention rows).

Multi-GPU: every rank runs an independent replica of the workload (the path
shards by sequence with no exchange); ranks meet only at the barriers, and
the slowest rank's time sets the throughput.
"""
from __future__ import annotations

import argparse
import hashlib
import gc
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-decode K/V read GB/s (% of GB300 HBM peak); decode steps/s per batch"
FALLBACK_HBM_GBS = 6800.0
SRC_FOR_TRAFFIC = ["paged_kv_cache_113_gb300/csrc/attention.cu", "paged_kv_cache_113_gb300/csrc/pk_device.cuh"]


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="mha7b", choices=["tiny", "mha7b", "gqa8b", "long", "prefix", "chat", "mixed"])
    p.add_argument("--block-size", type=int, default=None, help="prefix workload only: 8, 16 or 32")
    p.add_argument("--partition", type=int, default=-1, help="0 = no split, -1 = auto, >0 tokens")
    p.add_argument("--attn-impl", default="auto", choices=["auto", "simt", "mma"])
    p.add_argument("--window", type=int, default=32, help="distinct decode steps prepared ahead and cycled")
    p.add_argument("--e2e-steps", type=int, default=30)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--no-graphs", action="store_true", help="launch the timed steps eagerly, not as CUDA graphs")
    p.add_argument("--no-order", action="store_true", help="launch sequences in index order, not longest first")
    p.add_argument("--no-fuse", action="store_true",
                   help="run the slot scatter as its own kernel instead of inside the attention launch")
    p.add_argument("--grid", action="store_true",
                   help="launch the (sequence, partition) grid in longest-first sequence order instead of the "
                        "planned work list")
    p.add_argument("--cascade", action="store_true",
                   help="cascade attention: each shared prefix read once per group (prefix workload)")
    p.add_argument("--no-swap", action="store_true", help="skip the swap-out / swap-in bandwidth measurement")
    p.add_argument("--no-allocator-sim", action="store_true", help="skip the allocator policy table")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the target configurations timed beside the default workload (gqa8b, long, prefix)")
    p.add_argument("--config-steps", type=int, default=100, help="timed steps of each extra configuration")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline time budget")
    p.add_argument("--reference-seconds", type=float, default=90.0, help="reference arm time budget")
    a = p.parse_args(argv)
    if a.warmup < 3:
        p.error("--warmup must be at least 3")
    return a


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def reduce_max(values):
    """Element-wise maximum over ranks (identity without a process group).

    The slowest rank's time sets the whole job's throughput. Works on the
    gloo (CPU tensors) and nccl (CUDA tensors) backends."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_throughput(world: int, bytes_per_rank: float, seconds_max: float) -> float:
    """Whole-job GB/s: every rank processes the same replica, so the job moves
    world * bytes_per_rank in the slowest rank's time."""
    return world * bytes_per_rank / seconds_max / 1e9


def measured_hbm_peak():
    for path in (os.path.join(ROOT, "MEASURED_PEAKS.json"),):
        try:
            with open(path) as f:
                v = float(json.load(f)["hbm_gbs"])
            return v, "measured"
        except (OSError, KeyError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal


def read_stream_peak(dev, gib: int = 4, reps: int = 5) -> dict:
    """A read-only bandwidth reference measured in this run: the library's
    pure read stream (pk_read_stream) over a buffer far larger than L2,
    against the copy benchmark's read + write."""
    import torch
    import paged_kv_cache_113_gb300 as pk
    x = torch.ones(gib << 28, dtype=torch.float32, device=dev)   # gib GiB
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    nbytes = x.numel() * 4
    st = torch.cuda.current_stream(dev).cuda_stream

    def run():
        rc = pk.lib().pk_read_stream(ctypes_ptr(x), nbytes, ctypes_ptr(sink), st)
        if rc != 0:
            raise RuntimeError(f"pk_read_stream: status {rc}")
    for _ in range(2):
        run()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        run()
    e1.record()
    torch.cuda.synchronize()
    gbs = reps * nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9
    del x, sink
    torch.cuda.empty_cache()
    return {"value": gbs, "unit": "GB/s", "kernel": f"read_stream_kernel over {gib} GiB (each 16-byte vector once)"}


def ctypes_ptr(t):
    import ctypes
    return ctypes.c_void_p(t.data_ptr())


def source_hash():
    """Hash of the attention kernels' source with // comments and blank lines
    removed, so that comment edits do not retire the recorded traffic."""
    h = hashlib.sha256()
    for rel in SRC_FOR_TRAFFIC:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            for line in f:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()


def ncu_traffic(workload: str):
    """DRAM bytes per attention launch from the committed ncu summary, if the
    kernel source is unchanged since it was taken (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
        e = table[workload]
        if e.get("source_sha256") == source_hash():
            return int(e["dram_bytes_per_step"])
    except (OSError, KeyError, ValueError):
        pass
    return None


# ---------------------------------------------------------------------------
# Clocks sampler (nvidia-smi during the timed region)
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, uuid: str = None):
        self.dev = uuid or str(device_index)
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="pk_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.dev, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self, t_begin: float, t_end: float):
        """Summary of the samples taken between wall-clock times t_begin and t_end."""
        import datetime
        if self.proc is None:
            return {"samples": 0, "note": "nvidia-smi unavailable"}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if t_begin <= r[0] <= t_end]
        used = inside or [r for r in rows if r[0] >= t_begin][:1]
        if not used:
            return {"samples": 0, "samples_in_region": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, _, flags in used for i, fl in enumerate(flags)
                          if fl.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in used), "sm_max_mhz": max(r[2] for r in used),
                "reasons": reasons, "samples_in_region": len(inside), "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def oracle_state(wl):
    import oracle
    return oracle.run_workload(wl, attention=False)


def host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def host_cpu_model() -> str:
    """The host CPU's model name (x86 `model name`, or the Arm implementer/part pair)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model name"):
        for line in info.splitlines():
            if line.startswith(key):
                return line.split(":", 1)[1].strip()
    fields = {}
    for line in info.splitlines():
        if ":" in line:
            k, v = line.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    if "CPU part" in fields:
        return f"arm implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    return "unknown"


_POOLS = {}


def _oracle_pool(threads: int):
    """One thread pool per size, created once (not inside a timed call)."""
    from concurrent.futures import ThreadPoolExecutor
    if threads not in _POOLS:
        _POOLS[threads] = ThreadPoolExecutor(max_workers=threads)
    return _POOLS[threads]


def oracle_threads(threads: int, n_rows: int) -> int:
    """Host threads the oracle timing uses for n_rows rows: at least four rows each."""
    return max(1, min(threads, n_rows // 4))


def time_oracle_rows(wl, ref, rows: np.ndarray, threads: int = 1):
    """Times the oracle's attention over the given (seq, head) rows; returns (seconds, kv bytes).

    With ``threads`` > 1 the rows are dealt round-robin (longest first) to
    that many host threads, each calling the oracle on its share; the C
    oracle is reentrant and ctypes releases the interpreter lock for the
    call, so the threads run on separate cores."""
    import oracle
    ctx = ref["ctx_lens"]
    args = (ref["q"], ref["k_cache"], ref["v_cache"], ref["tables"], ref["ctx_lens"], wl.scale, wl.dtype)
    threads = oracle_threads(threads, len(rows))
    if threads == 1:
        t0 = time.perf_counter()
        oracle.paged_attention(*args, select=rows)
        dt = time.perf_counter() - t0
    else:
        order = np.argsort(-ctx[rows[:, 0]], kind="stable")
        shares = [np.ascontiguousarray(rows[order[i::threads]]) for i in range(threads)]
        ex = _oracle_pool(threads)
        t0 = time.perf_counter()
        list(ex.map(lambda sel: oracle.paged_attention(*args, select=sel), shares))
        dt = time.perf_counter() - t0
    # The step's algorithmic K/V bytes counted per query-head row: a KV head's
    # bytes are shared by its group of Hq / Hk query heads, so each row counts
    # 1 / group of them (a whole step sums to the same bytes as the GPU arm).
    group = wl.num_q_heads // wl.num_kv_heads
    nbytes = int(sum(int(ctx[s]) for s, _ in rows)) * wl.head_dim * wl.esz * 2 // group
    return dt, nbytes


def unique_kv_bytes(wl, si) -> int:
    """K/V bytes of the distinct physical slots a step reads (shared prefix
    blocks count once); equals the algorithmic bytes without sharing."""
    B = wl.block_size
    ctx = si.ctx_lens.astype(np.int64)
    slots = []
    for s in range(len(ctx)):
        n = int(ctx[s])
        nb = -(-n // B)
        blocks = si.tables[s, :nb].astype(np.int64)
        sl = (blocks[:, None] * B + np.arange(B)[None, :]).reshape(-1)[:n]
        slots.append(sl)
    return int(np.unique(np.concatenate(slots)).size) * wl.num_kv_heads * wl.head_dim * wl.esz * 2


def all_rows(wl):
    return np.array([(s, h) for s in range(wl.num_seqs) for h in range(wl.num_q_heads)], dtype=np.int32)


def cpu_baseline(wl, ref, seconds: float):
    """The oracle on the host cores: whole decode steps (every row) on all
    host threads, repeated until half the time budget is used (at least
    once), then a random sample of rows on one thread for the other half."""
    rows = all_rows(wl)
    threads = oracle_threads(host_threads(), len(rows))
    total_t, total_b, reps = 0.0, 0, 0
    while reps == 0 or total_t < seconds / 2:
        dt, nb = time_oracle_rows(wl, ref, rows, threads)
        total_t += dt
        total_b += nb
        reps += 1
        if total_t > 2 * seconds:
            break
    # One thread: the same per-row work on a sample sized from the all-core rate.
    rng = np.random.default_rng(1)
    n1 = int(min(len(rows), max(1, len(rows) * reps * (seconds / 2) / max(total_t * threads, 1e-9))))
    dt1, nb1 = time_oracle_rows(wl, ref, rows[rng.choice(len(rows), size=n1, replace=False)], 1)
    return {"value": total_b / total_t / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "cpu": host_cpu_model(),
            "single_thread": {"value": nb1 / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"{n1} random attention rows of one step"},
            "sample": f"{reps} full decode step(s) of attention ({len(rows)} rows each), C, fp64, "
                      f"rows dealt to {threads} host threads"}


def workload_config(wl, args, extra=None):
    c = {"workload": wl.name, "num_seqs": wl.num_seqs, "num_q_heads": wl.num_q_heads,
         "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "block_size": wl.block_size,
         "num_blocks": wl.num_blocks, "kv_dtype": wl.dtype, "ctx_mean": round(float(np.mean(wl.ctx_lens)), 1),
         "ctx_max": int(np.max(wl.ctx_lens)), "seed": wl.seed, "parallelism": f"replicas{args.gpus}"}
    if extra:
        c.update(extra)
    return c


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from workloads import make_workload
    wl = make_workload(args.workload, block_size=args.block_size)
    ref = oracle_state(wl)
    rows = all_rows(wl)
    rng = np.random.default_rng(0)
    # Calibrate the per-row cost on a few rows, then size each step's sample
    # so that warm-up plus timed steps fit the time budget.
    threads = oracle_threads(host_threads(), len(rows))
    probe = rows[rng.choice(len(rows), size=min(4 * threads, len(rows)), replace=False)]
    dt, _ = time_oracle_rows(wl, ref, probe, threads)
    per_row = dt / len(probe)
    budget = args.reference_seconds / (args.steps + args.warmup)
    n = int(max(1, min(len(rows), budget / max(per_row, 1e-9))))
    samples = [rows[rng.choice(len(rows), size=n, replace=False)] for _ in range(args.steps + args.warmup)]
    for i in range(args.warmup):
        time_oracle_rows(wl, ref, samples[i], threads)
    tt, tb = 0.0, 0
    for i in range(args.steps):
        dt, nb = time_oracle_rows(wl, ref, samples[args.warmup + i], threads)
        tt += dt
        tb += nb
    gbs = tb / tt / 1e9
    frac = n / len(rows)
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tt / args.steps / frac,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, args, {"sample_rows_per_step": n, "rows_per_step": len(rows)}),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": oracle_threads(threads, n), "kind": "oracle",
                         "cpu": host_cpu_model(),
                         "sample": f"{n} of {len(rows)} attention rows per step (random), C, fp64, dealt to "
                                   f"{oracle_threads(threads, n)} host threads; ms_per_step scaled to all rows"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------
class StepOptions:
    """How a decode step is launched (the bench flags that shape the step)."""

    def __init__(self, partition=-1, attn_impl="auto", cascade=False, grid=False, no_order=False, no_fuse=False,
                 no_graphs=False):
        self.partition, self.attn_impl, self.cascade = partition, attn_impl, cascade
        self.grid, self.no_order, self.no_fuse, self.no_graphs = grid, no_order, no_fuse, no_graphs

    @classmethod
    def from_args(cls, args):
        return cls(args.partition, args.attn_impl, args.cascade, args.grid, args.no_order, args.no_fuse,
                   args.no_graphs)


class L2Flush:
    """Evicts L2 between steps: writes 2x L2, then reads 2x L2 so that the
    next step starts on a cold and clean L2 (no dirty lines to write back)."""

    def __init__(self, dev):
        import torch
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.buf = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.buf.zero_()
        self.buf.sum()


def time_device_steps(st, wl, dev, opt: StepOptions, steps: int, warmup: int, window: int, reserve: int,
                      flush: L2Flush, world: int = 1, sampler=None):
    """Device time of ``steps`` decode steps of the state ``st``.

    The host side of a window of steps is prepared and uploaded first; each
    window step is captured as CUDA graphs (copy_blocks when pairs exist; the
    attention, with the step's scatter fused in by default) and the timed
    steps cycle through the window. Each step is bracketed by CUDA events on
    the launching stream, L2 flushed between steps outside the events.
    ``reserve`` is the number of tokens later phases may still append (it
    sizes the workspace). Returns the raw sums; the caller reduces over ranks.
    """
    import torch
    import paged_kv_cache_113_gb300 as pk

    R = max(1, min(window, steps + warmup))
    host_steps = [st.prepare_step() for _ in range(R)]
    dsteps = [st.upload(si) for si in host_steps]
    planned = not (opt.cascade or opt.grid or opt.no_order)
    # The default step: copy-on-write copies (if any), then one attention
    # launch that also writes the step's new K/V (the scatter fused in).
    fused = planned and not opt.no_fuse and opt.attn_impl == "auto"
    if planned:
        # The default schedule: each step's work list from the host planner
        # (pk_attention_plan), longest item first.
        for si, d in zip(host_steps, dsteps):
            d["partition"], d["items"] = st.plan(si, opt.partition)
    step_bytes = [wl.kv_bytes(si.ctx_lens) for si in host_steps]
    step_unique = [unique_kv_bytes(wl, si) for si in host_steps]
    max_ctx = max(si.max_context_len for si in host_steps) + reserve
    if planned:
        ws_bytes = max(st.workspace_bytes(max_ctx, d["partition"]) for d in dsteps)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev) if ws_bytes else None
    else:
        ws = st.alloc_workspace(max_ctx, opt.partition)
    out = st.new_out()
    simt = opt.attn_impl == "simt" or wl.dtype == "f32"
    groups = st.cascade_groups() if opt.cascade else None
    if groups is not None:
        ws = st.alloc_cascade_workspace(max_ctx, groups, opt.partition)

    # Kernels one step launches: copy_blocks (if pairs), the scatter (unless
    # fused into the attention), the attention kernel, and the split-K merge
    # when the step splits (the cascade kernel's parts always merge).
    def launches(si, d):
        if groups is not None and groups["num_groups"]:
            return (1 if len(si.pairs) else 0) + 3  # scatter, cascade kernel (prefix and suffix CTAs), merge
        part = d["partition"] if "partition" in d else st.resolve_partition(si.max_context_len, opt.partition)
        split = part > 0 and math.ceil(si.max_context_len / part) > 1
        scatter = 0 if fused and not simt else 1
        return (1 if len(si.pairs) else 0) + scatter + 1 + (1 if split else 0)

    def cache_writes(d):
        if d["pairs"].shape[0]:
            pk.pk_copy_blocks(st.k_cache, st.v_cache, d["pairs"])
        if not fused:
            pk.pk_reshape_and_cache(d["k"], d["v"], d["slots"], st.k_cache, st.v_cache)

    def attend(d):
        if groups is not None:
            st.attention_cascade(d, out, groups, ws, opt.partition, ordered=not opt.no_order)
        elif fused:
            pk.pk_paged_attention_decode_append(out, d["q"], d["k"], d["v"], d["slots"], st.k_cache, st.v_cache,
                                                d["tables"], d["ctx_lens"], wl.scale, d["max_context_len"],
                                                d["partition"], d["items"], ws)
        else:
            st.attention(d, out, ws, opt.partition, opt.attn_impl, ordered=not opt.no_order)

    # warm-up (eager; also performs the library's one-time set-up)
    for i in range(warmup):
        flush()
        cache_writes(dsteps[i % R])
        attend(dsteps[i % R])
    torch.cuda.synchronize()
    kind, _ = pk.pk_get_device_error()
    if kind:
        raise RuntimeError(f"device error during warm-up: {pk.DEVERR_NAMES.get(kind)}")

    # Each window step as two CUDA graphs (cache writes; attention + merge), so
    # the timed region holds GPU work only, as a decode loop would run it.
    graphs = None
    if not opt.no_graphs:
        graphs = []
        for d in dsteps:
            g_w, g_a = None, torch.cuda.CUDAGraph()
            if d["pairs"].shape[0] or not fused:  # nothing to capture when the scatter is fused
                g_w = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g_w):
                    cache_writes(d)
            with torch.cuda.graph(g_a):
                attend(d)
            graphs.append((g_w, g_a))
        torch.cuda.synchronize()

    if sampler is not None:
        sampler.start()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    n_launch = 0
    total_bytes = 0
    total_unique = 0
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    clock0 = time.time()
    # A timed event record takes ~2 us of GPU time (measured on GB300), so the
    # step's middle event is recorded only when cache writes precede the
    # attention; otherwise the attention is timed from the step's first event.
    has_writes = [bool(d["pairs"].shape[0]) or not fused for d in dsteps]
    for i in range(steps):
        flush()
        j = (warmup + i) % R
        d = dsteps[j]
        e0, e1, e2 = ev[i]
        e0.record()
        if not has_writes[j]:
            ev[i][1] = e0
        elif graphs:
            graphs[j][0].replay()
            e1.record()
        else:
            cache_writes(d)
            e1.record()
        if graphs:
            graphs[j][1].replay()
        else:
            attend(d)
        e2.record()
        n_launch += launches(host_steps[j], d)
        total_bytes += step_bytes[j]
        total_unique += step_unique[j]
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop(clock0, time.time()) if sampler is not None else None
    t_step = sum(a.elapsed_time(c) for a, _, c in ev) / 1e3
    t_attn = sum(b.elapsed_time(c) for _, b, c in ev) / 1e3
    kind, idx = pk.pk_get_device_error()
    if kind:
        raise RuntimeError(f"device error in the timed steps: {pk.DEVERR_NAMES.get(kind)} at {idx}")
    part = st.resolve_partition(max(si.max_context_len for si in host_steps), opt.partition)
    if planned:
        parts = sorted({d["partition"] for d in dsteps})
        part = parts[0] if len(parts) == 1 else parts
    if groups is not None:
        part = opt.partition if opt.partition >= 0 else "auto (cascade)"
    del graphs
    return {"t_step": t_step, "t_attn": t_attn, "bytes": total_bytes, "unique": total_unique,
            "launches": n_launch, "wall": wall, "clocks": clocks, "window": R, "partition": part,
            "fused": fused, "planned": planned, "simt": simt, "graphs": not opt.no_graphs,
            "groups": None if groups is None else int(groups["num_groups"]),
            "kernel": ("attn_cascade_kernel + attn_lse_merge_kernel" if groups is not None else
                       "attn_mma_kernel (+ attn_lse_merge_kernel when split)" if not simt
                       else "attn_simt_kernel (+ attn_merge_kernel when split)")}


def traffic_key(wl, cascade: bool, partition: int) -> str:
    """Key of a workload's entry in the committed ncu traffic table."""
    k = wl.name if wl.name != "prefix" else f"prefix{wl.block_size}"
    if partition > 0:
        k += f"_p{partition}"
    return k + ("_cascade" if cascade else "")


# The target configurations measured beside the headline workload on a
# default single-GPU run: (workload, block size, partition, cascade).
EXTRA_CONFIGS = [("gqa8b", None, -1, False), ("long", None, -1, False), ("long", None, 512, False),
                 ("prefix", 8, -1, False), ("prefix", 8, -1, True), ("prefix", 16, -1, False),
                 ("prefix", 16, -1, True), ("prefix", 32, -1, False), ("prefix", 32, -1, True)]


def run_configs(args, dev, flush, peak: float, peak_kind: str) -> dict:
    """The target configurations, each a short device-timed run of its own
    (the headline's step, L2 flushing and events; no e2e, swap or CPU legs),
    under one clock sampler."""
    import torch
    from paged_kv_cache_113_gb300.harness import DecodeState
    from workloads import make_workload

    sampler = None
    if not args.no_clocks:
        sampler = ClockSampler(torch.cuda.current_device(), gpu_uuid(dev))
        sampler.start()
    t0, c0 = time.perf_counter(), time.time()
    rows = []
    steps = max(1, min(args.steps, args.config_steps))
    for name, B, part, cascade in EXTRA_CONFIGS:
        wl = make_workload(name, block_size=B)
        wl.enable_memo()
        st = DecodeState(wl, dev, extra_tokens=args.window + 1)
        opt = StepOptions(partition=part, cascade=cascade)
        m = time_device_steps(st, wl, dev, opt, steps, args.warmup, args.window, 1, flush)
        attn_gbs = m["bytes"] / m["t_attn"] / 1e9
        ms = 1e3 * m["t_step"] / steps
        rows.append({
            "workload": name, "block_size": wl.block_size, "num_seqs": wl.num_seqs,
            "num_q_heads": wl.num_q_heads, "num_kv_heads": wl.num_kv_heads,
            "partition": m["partition"], "partition_requested": "auto" if part == -1 else part,
            "attention": f"cascade ({m['groups']} shared-prefix groups)" if cascade else "per sequence",
            "steps": steps, "value": m["bytes"] / m["t_step"] / 1e9, "unit": "GB/s",
            "ms_per_step": ms, "steps_per_s": 1e3 / ms, "attention_gbs": attn_gbs,
            "attention_unique_gbs": m["unique"] / m["t_attn"] / 1e9,
            "kv_bytes_per_step_mean": m["bytes"] / steps, "kv_unique_bytes_per_step_mean": m["unique"] / steps,
            "gpu_launches": m["launches"],
            "roofline": {"bound": "hbm", "kernel": m["kernel"], "achieved": attn_gbs, "peak": peak,
                         "unit": "GB/s", "frac": attn_gbs / peak, "peak_kind": f"{peak_kind} copy bandwidth",
                         "frac_unique": m["unique"] / m["t_attn"] / 1e9 / peak,
                         "traffic": ncu_traffic(traffic_key(wl, cascade, part)),
                         "bytes_per_launch": m["bytes"] / steps, "ms_per_launch": 1e3 * m["t_attn"] / steps},
        })
        del st
        torch.cuda.empty_cache()
    clocks = sampler.stop(c0, time.time()) if sampler is not None else None
    return {"note": "each configuration timed as the headline (planned work list, scatter fused in, CUDA "
                    "graphs, L2 flushed between steps, CUDA events); 'cascade' rows run attn_cascade_kernel "
                    "with a separate scatter; frac_unique counts each shared block once",
            "wall_s": time.perf_counter() - t0, "clocks": clocks, "rows": rows}


def gpu_uuid(dev):
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return None


def run_ours(args):
    import torch
    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import paged_kv_cache_113_gb300 as pk
    from paged_kv_cache_113_gb300.harness import DecodeState
    from workloads import make_workload

    if rank == 0:
        pk.build()
    if world > 1:
        torch.distributed.barrier()
    pk.lib()

    wl = make_workload(args.workload, block_size=args.block_size)
    wl.enable_memo()
    R = max(1, min(args.window, args.steps + args.warmup))
    E = 0 if args.no_e2e else max(1, args.e2e_steps)
    Ew = 0 if args.no_e2e else 8
    st = DecodeState(wl, dev, extra_tokens=R + E + Ew + 1)
    flush = L2Flush(dev)
    sampler = None if args.no_clocks else ClockSampler(local_rank, gpu_uuid(dev))
    opt = StepOptions.from_args(args)
    m = time_device_steps(st, wl, dev, opt, args.steps, args.warmup, args.window, E + Ew + 1, flush,
                          world=world, sampler=sampler)
    total_bytes, total_unique = m["bytes"], m["unique"]
    t_step, t_attn = reduce_max([m["t_step"], m["t_attn"]])
    value = job_throughput(world, total_bytes, t_step)
    attn_gbs = total_bytes / t_attn / 1e9
    peak, peak_kind = measured_hbm_peak()
    read_peak = read_stream_peak(dev) if rank == 0 else None

    e2e = None
    if E:
        # On a fresh copy of the workload's state, so that the e2e steps see
        # the device steps' context lengths rather than ones a window further.
        st_e2e = DecodeState(wl, dev, extra_tokens=E + Ew + 1)
        e2e = run_e2e(st_e2e, wl, E, Ew, args, dev)
        del st_e2e
        torch.cuda.empty_cache()
        e2e["value"] = job_throughput(world, e2e["_bytes"], reduce_max([e2e["_seconds"]])[0])
        e2e.pop("_seconds")
        e2e.pop("_bytes")

    prefix_cache = run_prefix_cache(st, wl) if wl.chat_choice is not None else None
    allocator_sim = None if args.no_allocator_sim else run_allocator_sim()
    swap = None if args.no_swap or m["groups"] is not None else run_swap(st, wl, dev)

    configs = None
    if world == 1 and not args.no_configs and args.workload == "mha7b":
        del st
        torch.cuda.empty_cache()
        configs = run_configs(args, dev, flush, peak, peak_kind)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ref = oracle_state(wl)
        cpu = cpu_baseline(wl, ref, args.cpu_seconds)

    mean_ms = 1e3 * t_step / args.steps
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": mean_ms, "steps_per_s": 1e3 / mean_ms,
            "pct_of_peak": 100.0 * value / world / peak, "peak_kind": peak_kind,
            "pct_of_nominal_hbm": 100.0 * value / world / NOMINAL_HBM_GBS,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32",
            "data": "synthetic",
            "config": workload_config(wl, args, {
                "partition": m["partition"], "attn_impl": args.attn_impl, "window_steps": m["window"],
                "l2": "flushed between steps: 2x L2 written then 2x L2 read (cold, clean L2), outside the step events",
                "kv_bytes_per_step_mean": total_bytes / args.steps,
                "kv_unique_bytes_per_step_mean": total_unique / args.steps,
                "launch": "CUDA graphs per step" if m["graphs"] else "eager",
                "scatter": "fused into the attention launch" if m["fused"] else "own kernel",
                "seq_order": "index" if args.no_order else
                             ("planned work list, longest item first (host)" if m["planned"] else "longest first (host)"),
                "attention": (f"cascade: {m['groups']} shared-prefix groups, prefix read once per group"
                              if m["groups"] is not None else "per sequence")}),
            "roofline": {"bound": "hbm", "kernel": m["kernel"],
                         "achieved": attn_gbs, "peak": peak, "unit": "GB/s", "frac": attn_gbs / peak,
                         "peak_kind": f"{peak_kind} copy bandwidth",
                         "traffic": ncu_traffic(traffic_key(wl, m["groups"] is not None, args.partition)),
                         "bytes_per_launch": total_bytes / args.steps, "ms_per_launch": 1e3 * t_attn / args.steps},
            "attention_gbs": attn_gbs,
            "attention_unique_gbs": total_unique / t_attn / 1e9,
            "read_stream_peak": (dict(read_peak, attention_frac=attn_gbs / read_peak["value"])
                                 if read_peak else None),
            "gpu_launches": m["launches"],
            "wall_s_timed_region": m["wall"],
            "clocks": m["clocks"],
            "e2e": e2e,
            "configs": configs,
            "swap": swap,
            "prefix_cache": prefix_cache,
            "allocator_sim": allocator_sim,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_e2e(st, wl, E, Ew, args, dev):
    """The same decode steps through the public API from pinned host memory:
    per step pk_decode_step_launch of the prepared step (zero-copy: the
    kernels read q, the new K/V and the slots from pinned host memory and
    write the output back to it), pk_decode_step_prepare of the next step
    (host block-manager append, overlapped with the GPU), then a stream
    synchronise."""
    import torch
    import paged_kv_cache_113_gb300 as pk

    def pinned(a):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16) if wl.dtype == "bf16" \
            else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
        return t.pin_memory()

    inputs = [tuple(pinned(x) for x in wl.step_inputs(10_000 + i)) for i in range(E + Ew)]
    max_ctx = int(wl.ctx_lens.max()) + st.steps_done + E + Ew + 1
    # Zero-copy: each step's inputs sit in their own pinned host buffers when
    # the step starts; the launch points the captured kernels at them, and
    # the kernels read them and write the output back across the host link
    # inside the timed step.
    stepper = pk.DecodeStepper(st.bm, range(wl.num_seqs), wl.num_q_heads, wl.scale, st.max_blocks,
                               st.k_cache, st.v_cache, args.partition, max_context_len=max_ctx,
                               zero_copy=True)
    torch.cuda.synchronize()
    stream = stepper.stream
    tot_t, tot_b = 0.0, 0
    per_step, host_launch, host_prepare = [], [], []
    resident = True
    # The overlapped loop of a serving engine: each step's host half (block-
    # manager append, metadata) is prepared while the step before runs on the
    # GPU, so a timed step holds its launch, the next step's host half and
    # the synchronise. Step 0's host half is prepared before the warm-up.
    # Every step appends one token to every sequence, so step i reads the
    # starting lengths + i + 1 tokens; its bytes are counted up front, keeping
    # host work out of the loop.
    lens0 = np.array([st.bm.seq_len(s) for s in range(wl.num_seqs)], dtype=np.int64)
    step_bytes = [wl.kv_bytes(lens0 + i + 1) for i in range(E + Ew)]
    stepper.prepare()
    # No collector pauses inside the timed steps (as timeit does).
    gc_enabled = gc.isenabled()
    gc.disable()
    try:
        for i in range(E + Ew):
            q, k, v = inputs[i]
            stream.synchronize()
            t0 = time.perf_counter()
            stepper.launch_prepared(q_host=q, k_host=k, v_host=v)
            t1 = time.perf_counter()
            stepper.prepare()
            t2 = time.perf_counter()
            stream.synchronize()
            dt = time.perf_counter() - t0
            st.steps_done += 1
            if i >= Ew:
                resident = resident and stepper.graph_count > 0
                tot_t += dt
                tot_b += step_bytes[i]
                per_step.append(dt)
                host_launch.append(t1 - t0)
                host_prepare.append(t2 - t1)
    finally:
        if gc_enabled:
            gc.enable()
    kind, idx = pk.pk_get_device_error()
    if kind:
        raise RuntimeError(f"device error in the e2e steps: {pk.DEVERR_NAMES.get(kind)} at {idx}")
    assert resident, "the timed e2e steps run with resident tables, as captured graphs"
    stepper.release()
    return {"value": tot_b / tot_t / 1e9, "unit": "GB/s", "h2d_bytes_per_step": int(stepper.h2d_bytes_resident),
            "d2h_bytes_per_step": int(stepper.d2h_bytes), "steps": E, "ms_per_step": 1e3 * tot_t / E,
            "ms_per_step_median": 1e3 * float(np.median(per_step)), "ms_per_step_max": 1e3 * max(per_step),
            "host_us_median": {"launch": 1e6 * float(np.median(host_launch)),
                               "prepare_next_overlapped": 1e6 * float(np.median(host_prepare))},
            "host_launch_us_median": 1e6 * float(np.median(host_launch)),
            "host_prepare_us_median": 1e6 * float(np.median(host_prepare)),
            "includes": "pk_decode_step_launch of the prepared step on that step's own pinned input "
                        "buffers (device-resident block tables, its own stream, zero-copy; on steady steps "
                        "one CUDA graph of one kernel, re-pointed at the step's buffers: the scatter reading "
                        "the slots and the new K/V from pinned host memory and advancing the tables, the "
                        "attention reading q from and writing the output to pinned host memory over the "
                        "host link), then pk_decode_step_prepare of the next step (host block-manager "
                        "append, overlapped with the GPU), stream sync",
            "_seconds": tot_t, "_bytes": tot_b}


def run_swap(st, wl, dev, reps: int = 5) -> dict:
    """Preemption by swapping, measured after the decode steps: every other
    sequence of the batch is swapped out to a pinned host pool and back in,
    ``reps`` times. Each direction is one pk_swap_blocks launch timed with
    CUDA events; the host-link peak beside it is a contiguous copy-engine
    copy of the same bytes between pinned host memory and the device."""
    import torch
    import paged_kv_cache_113_gb300 as pk

    victims = list(range(0, wl.num_seqs, 2))
    nblk = sum(len(st.bm.table(s)) for s in victims)
    st.bm.set_swap_space(nblk, np.arange(nblk, dtype=np.int32))
    shape = (nblk,) + tuple(st.k_cache.shape[1:])
    hk = torch.empty(shape, dtype=st.k_cache.dtype).pin_memory()
    hv = torch.empty(shape, dtype=st.k_cache.dtype).pin_memory()
    moved = 2 * hk.numel() * hk.element_size()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    t_out = t_in = 0.0
    for r in range(reps + 1):
        po = torch.from_numpy(np.concatenate([st.bm.swap_out(s) for s in victims])).to(dev)
        torch.cuda.synchronize()
        ev[0].record()
        pk.pk_swap_blocks(st.k_cache, st.v_cache, hk, hv, po, pk.PK_SWAP_OUT)
        ev[1].record()
        pi = torch.from_numpy(np.concatenate([st.bm.swap_in(s) for s in victims])).to(dev)
        torch.cuda.synchronize()
        ev[2].record()
        pk.pk_swap_blocks(st.k_cache, st.v_cache, hk, hv, pi, pk.PK_SWAP_IN)
        ev[3].record()
        torch.cuda.synchronize()
        if r:
            t_out += ev[0].elapsed_time(ev[1]) / 1e3
            t_in += ev[2].elapsed_time(ev[3]) / 1e3
    kind, idx = pk.pk_get_device_error()
    if kind:
        raise RuntimeError(f"device error while swapping: {pk.DEVERR_NAMES.get(kind)} at {idx}")
    st.bm.check_invariants()

    # Copy-engine reference: the same bytes as two contiguous copies per direction.
    scratch = torch.empty(2 * hk.numel(), dtype=hk.dtype, device=dev)
    t_d2h = t_h2d = 0.0
    for r in range(reps + 1):
        torch.cuda.synchronize()
        ev[0].record()
        hk.view(-1).copy_(scratch[:hk.numel()], non_blocking=True)
        hv.view(-1).copy_(scratch[hk.numel():], non_blocking=True)
        ev[1].record()
        scratch[:hk.numel()].copy_(hk.view(-1), non_blocking=True)
        scratch[hk.numel():].copy_(hv.view(-1), non_blocking=True)
        ev[2].record()
        torch.cuda.synchronize()
        if r:
            t_d2h += ev[0].elapsed_time(ev[1]) / 1e3
            t_h2d += ev[1].elapsed_time(ev[2]) / 1e3
    out_gbs, in_gbs = reps * moved / t_out / 1e9, reps * moved / t_in / 1e9
    d2h_gbs, h2d_gbs = reps * moved / t_d2h / 1e9, reps * moved / t_h2d / 1e9
    return {"sequences": len(victims), "blocks": nblk, "bytes_per_direction": moved, "reps": reps,
            "out_gbs": out_gbs, "in_gbs": in_gbs, "out_ms": 1e3 * t_out / reps, "in_ms": 1e3 * t_in / reps,
            "link_copy_d2h_gbs": d2h_gbs, "link_copy_h2d_gbs": h2d_gbs,
            "frac_out": out_gbs / d2h_gbs, "frac_in": in_gbs / h2d_gbs,
            "kernel": "swap_blocks_kernel (one launch per direction, host pool mapped into the device)",
            "peak_kind": "contiguous pinned copy of the same bytes, measured in this run"}


def run_prefix_cache(st, wl, reps: int = 3) -> dict:
    """Prefix caching on the chat workload: how much of the admitted prompts
    the cache served (so prefill never recomputes or rewrites them), and the
    host cost of admission through the public API (add_seq_cached, append of
    the rest, commit), replayed on a fresh block manager, best of ``reps``."""
    import paged_kv_cache_113_gb300 as pk
    from workloads import prefill_plan

    plan = prefill_plan(wl)
    toks = {op[1]: wl.chat_tokens(op[1]) for op in plan if op[0] == "admit"}
    best = None
    for _ in range(reps):
        bm = pk.BlockManager(wl.num_blocks, wl.block_size, wl.alloc_order())
        t0 = time.perf_counter()
        for op in plan:
            r = op[1]
            if op[0] == "admit":
                t = toks[r]
                c = bm.add_seq_cached(r, t)
                if len(t) > c:
                    bm.append(r, len(t) - c)
                bm.commit(r, t)
            else:
                bm.free_seq(r)
        dt = time.perf_counter() - t0
        best = dt if best is None else min(best, dt)
    prompt = sum(len(t) for t in toks.values())
    per_token = wl.num_kv_heads * wl.head_dim * wl.esz * 2
    return {"requests_admitted": len(toks), "prompt_tokens": st.prompt_tokens, "cached_tokens": st.cached_tokens,
            "cached_fraction": st.cached_tokens / max(st.prompt_tokens, 1),
            "prefill_kv_bytes_written": (st.prompt_tokens - st.cached_tokens) * per_token,
            "prefill_kv_bytes_without_cache": st.prompt_tokens * per_token,
            "cache": st.bm.cache_stats(),
            "host_admission_us_per_request": 1e6 * best / len(toks),
            "host_admission_prompt_tokens_per_s": prompt / best,
            "host_admission": "add_seq_cached + append of the uncached rest + commit, Python binding, best of 3"}


def run_allocator_sim(reps: int = 3) -> dict:
    """The allocator policy table ("The KV Cache Is an Allocator Problem",
    "What the trace shows") on the seeded traces, from the library's
    simulator, with its host time per run (best of ``reps``)."""
    import paged_kv_cache_113_gb300 as pk
    from workloads import ALLOCATOR_TRACES, allocator_trace

    out = {"rule": "a failed growth drops the request", "traces": {}}
    for name in ALLOCATOR_TRACES:
        C, trace = allocator_trace(name)
        rows = {}
        for policy, B in (("max_reservation", 0), ("exact_contiguous", 0), ("paged", 4), ("paged", 8),
                          ("paged", 16)):
            best = None
            for _ in range(reps):
                t0 = time.perf_counter()
                r = pk.pk_sim_run(trace, C, policy, B, "drop")
                dt = time.perf_counter() - t0
                best = dt if best is None else min(best, dt)
            s = r["summary"]
            rows[policy if not B else f"paged_b{B}"] = {
                "rejected": s["rejected"], "rejected_despite_free": s["rejected_despite_free"],
                "growth_failures": s["growth_failures"],
                "growth_failures_despite_free": s["growth_failures_despite_free"],
                "peak_reserved": s["peak_reserved"], "peak_waste": s["peak_waste"], "peak_live": s["peak_live"],
                "host_ms": 1e3 * best, "host_us_per_step": 1e6 * best / s["num_steps"]}
        out["traces"][name] = {"capacity_slots": C, "requests": len(trace), "steps": r["summary"]["num_steps"],
                               "policies": rows}
    return out


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
