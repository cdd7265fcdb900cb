"""Benchmark of one paged-attention decode step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 8b_gqa]
                    [--kernel auto|mma|simt|generic|tc] [--impl native|reference]

A step is the whole hot path over one batch: pa_reshape_and_cache (append the
new K/V rows) then pa_decode (attention through the block tables, with the
split-K merge when a sequence spans several 512-row partitions). Inputs are
the seeded synthetic workloads of paged_kv_cache_29_gb300.workloads, resident
in HBM before timing. Between timed steps a 256 MiB buffer is written and a
second 256 MiB buffer is read, so that every timed step starts with an L2 that
holds none of its inputs and no dirty lines left to write back (the attended
K/V bytes are also larger than L2). Timing uses CUDA events on
the launching stream; clocks are sampled with nvidia-smi during the timed
region.

One JSON line is printed by rank 0. `value` is the step's algorithmic bytes
(K/V rows attended, q read, out written, block-table entries and context
lengths used, the append's reads and writes) over the step time, in GB/s.
`roofline` covers the attention call (decode + merge kernels) against the
measured HBM copy bandwidth. `e2e` repeats the measurement through the same
public API with the step's per-step inputs copied from pinned host memory (one
packed buffer, one copy) and the output copied back inside the timed region
(the KV pool stays resident: it is the cache). `cpu_baseline` times the fp64 oracle on a bounded sample of
the same workload on the host's cores.

--impl reference times the oracle itself (the CPU baseline) in the same JSON
format. Under torchrun every rank runs its own batch (weak scaling, no
collective on the data path); only the barrier and the max-over-ranks of the
timings cross ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_cache_29_gb300 import accounting  # noqa: E402
from paged_kv_cache_29_gb300 import workloads as wl  # noqa: E402

METRIC = "paged decode attention: achieved KV GB/s (% of GB300 HBM peak) and seqs/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
COPY_PAIRS = 4096
# Bound on every collective of a multi-rank run (the final barrier and the
# max/sum over ranks): a rank that died makes the others fail, not wait.
PG_TIMEOUT_S = 300
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "pa_decode_8b_gqa_ncu.md")
CSRC = os.path.join(ROOT, "paged_kv_cache_29_gb300", "csrc")


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def measured_hbm_gbs() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C/C++/CUDA source without its comments and blank lines (the kernel
    sources hold no comment markers inside string literals)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(csrc: str = CSRC) -> str:
    """Hash of the kernel sources' code (comments and blank lines left out), so
    that a profile taken on one build stays matched across comment edits."""
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str) -> float | None:
    """DRAM bytes per launch of the attention call from the committed ncu
    summary, if it was taken on the current kernel sources and this workload."""
    try:
        with open(PROFILE_SUMMARY) as f:
            lines = f.read().splitlines()
    except OSError:
        return None
    vals = {}
    for line in lines:
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != kernel_source_hash():
        return None
    if vals.get("workload") != workload or vals.get("kernel") != kernel:
        return None
    try:
        return float(vals["dram_bytes_per_call"])
    except (KeyError, ValueError):
        return None


def packed_buffer(arrays, pin=False, storage=None):
    """numpy arrays back to back in one byte tensor (each region 256-byte
    aligned): returns the byte tensor and a typed view per array. With
    `storage` the views are cut from that tensor (same layout), else a host
    tensor is made (pinned if asked) holding the arrays' bytes."""
    import torch
    offs, off = [], 0
    for a in arrays:
        off = (off + 255) // 256 * 256
        offs.append(off)
        off += a.nbytes
    if storage is None:
        storage = torch.empty(off, dtype=torch.uint8, pin_memory=pin)
        for a, o in zip(arrays, offs):
            raw = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
            storage[o:o + raw.size] = torch.from_numpy(raw)
    views = []
    for a, o in zip(arrays, offs):
        tdt = {np.dtype(np.uint16): torch.bfloat16, np.dtype(np.int64): torch.int64,
               np.dtype(np.int32): torch.int32, np.dtype(np.float32): torch.float32}[a.dtype]
        views.append(storage[o:o + a.nbytes].view(tdt).view(a.shape))
    return storage, views


def _quick_step_seconds(run, flush) -> float:
    """Wall time of one step (for sizing the clock soak)."""
    import torch
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(5):
        run()
    torch.cuda.synchronize()
    return (time.perf_counter() - t0) / 5


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def reduce_over_ranks(timings, counts, device):
    """Whole-job figures: the max of each timing and the sum of each work
    count over all ranks (the inputs unchanged without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(x) for x in timings], [float(x) for x in counts]
    t = torch.tensor([float(x) for x in timings], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    c = torch.tensor([float(x) for x in counts], device=device, dtype=torch.float64)
    dist.all_reduce(c, op=dist.ReduceOp.SUM)
    return t.tolist(), c.tolist()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---------------------------------------------------------------------------
# CPU oracle baseline (the oracle as it stands, on a bounded sample)
# ---------------------------------------------------------------------------

def sample_step(step: wl.DecodeStep, seqs: list[int]) -> wl.DecodeStep:
    idx = np.array(seqs, dtype=np.int64)
    Q = step.num_queries
    tok = (idx[:, None] * Q + np.arange(Q)[None, :]).reshape(-1)
    return wl.DecodeStep(**{**step.__dict__, "q": step.q[idx], "k_new": step.k_new[tok],
                            "v_new": step.v_new[tok], "slot_mapping": step.slot_mapping[tok],
                            "block_tables": step.block_tables[idx],
                            "context_lens": step.context_lens[idx]})


def oracle_decode(step: wl.DecodeStep, sub: wl.DecodeStep, threads: int):
    """The oracle's attention for the sequences of `sub` over `step`'s pool,
    with the oracle function of the step's kind."""
    import oracle
    args = (sub.block_tables, sub.context_lens, step.scale)
    if step.cache_dtype == "int8":
        return oracle.decode_int8(sub.q, step.k_cache, step.v_cache, step.k_row_scales,
                                  step.v_row_scales, *args, num_threads=threads)
    if step.cache_dtype == "fp8":
        return oracle.decode_kv(sub.q, step.k_cache, step.v_cache, *args, step.k_scale,
                                step.v_scale, num_threads=threads)
    if step.num_queries > 1:
        return oracle.decode_multi(sub.q, step.k_cache, step.v_cache, *args, num_threads=threads)
    if step.window > 0:
        return oracle.decode_window(sub.q, step.k_cache, step.v_cache, *args, step.window,
                                    num_threads=threads)
    return oracle.decode(sub.q, step.k_cache, step.v_cache, *args, num_threads=threads)


def oracle_sample_plan(step: wl.DecodeStep, target_s: float, threads: int):
    """Pick a sample of sequences that keeps the oracle busy about target_s
    seconds; the rate is probed on one short sequence first."""
    order = list(np.argsort(step.context_lens, kind="stable"))
    probe = sample_step(step, [order[len(order) // 2]])
    t0 = time.perf_counter()
    oracle_decode(step, probe, 1)
    per_token = (time.perf_counter() - t0) / max(int(probe.context_lens.sum()), 1)
    budget_tokens = target_s * max(threads, 1) / max(per_token, 1e-12)
    chosen, tokens = [], 0
    rng = np.random.default_rng(123)
    for s in rng.permutation(step.num_seqs):
        n = int(step.context_lens[s])
        if chosen and tokens + n > budget_tokens:
            continue
        chosen.append(int(s))
        tokens += n
        if tokens >= budget_tokens:
            break
    return sorted(chosen)


def time_oracle(step: wl.DecodeStep, seqs: list[int], threads: int) -> tuple[float, int]:
    """Seconds for one oracle decode over the sampled sequences, and their
    algorithmic attention bytes."""
    sub = sample_step(step, seqs)
    t0 = time.perf_counter()
    oracle_decode(step, sub, threads)
    dt = time.perf_counter() - t0
    return dt, accounting.step_bytes_for(sub).decode


def cpu_baseline(step: wl.DecodeStep, target_s: float = 12.0) -> dict:
    """The oracle over a bounded sample, repeated until about target_s seconds
    of host time have passed; reports the mean rate."""
    threads = os.cpu_count() or 1
    seqs = oracle_sample_plan(step, target_s, threads)
    total_s, total_bytes, reps = 0.0, 0, 0
    while reps == 0 or (total_s < target_s and reps < 1000):
        dt, nbytes = time_oracle(step, seqs, threads)
        total_s += dt
        total_bytes += nbytes
        reps += 1
    return {"value": round(total_bytes / total_s / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": (f"fp64 C oracle (OpenMP, {threads} threads) attention over {len(seqs)} of "
                       f"{step.num_seqs} sequences ({int(step.context_lens[seqs].sum())} of "
                       f"{int(step.context_lens.sum())} rows) of {step.name}, {reps} passes in "
                       f"{total_s:.1f} s; GB/s of the sample's algorithmic attention bytes"),
            "seconds": round(total_s, 3)}


def oracle_rates(step: wl.DecodeStep, seconds: float) -> dict:
    """The oracle's rate on a bounded sample of the workload at every host
    core and at one thread (about `seconds` of host time each), with the time
    a whole step's attention would take at that rate."""
    full = accounting.step_bytes_for(step).decode
    out = {}
    for key, threads in (("all_cores", os.cpu_count() or 1), ("one_thread", 1)):
        seqs = oracle_sample_plan(step, seconds, threads)
        dt, nbytes, reps = 0.0, 0, 0
        while reps == 0 or (dt < 0.5 * seconds and reps < 1000):   # tiny samples: repeat
            t, b = time_oracle(step, seqs, threads)
            dt, nbytes, reps = dt + t, nbytes + b, reps + 1
        rate = nbytes / dt
        out[key] = {"threads": threads, "gbs": round(rate / 1e9, 4),
                    "step_ms_at_this_rate": round(full / rate * 1e3, 3),
                    "sample": f"{len(seqs)} of {step.num_seqs} sequences, "
                              f"{int(step.context_lens[seqs].sum())} rows, {reps} passes "
                              f"in {dt:.2f} s"}
    return out


# ---------------------------------------------------------------------------
# the native (CUDA) arm
# ---------------------------------------------------------------------------

class DeviceWorkload:
    """One workload resident on the GPU with its step and attention-call
    closures. A step is one fused append + decode call for workloads with one
    query token per sequence and no window (pa_append_decode and its FP8/INT8
    forms: the decode kernel writes, or quantises, the new rows itself), else
    the append call followed by the decode call."""

    def __init__(self, pa, step: wl.DecodeStep, dev, kernel: str = "auto"):
        import torch
        self.step, self.kernel = step, kernel
        cd = step.cache_dtype
        self.fp8, self.int8 = cd == "fp8", cd == "int8"

        def up(a):
            # bf16 arrays are uint16 bit patterns; FP8 pools stay uint8 codes
            t = torch.from_numpy(np.ascontiguousarray(a))
            if a.dtype == np.uint16:
                t = t.view(torch.bfloat16)
            return t.to(dev)

        # A step's inputs (q, the new rows, slots, block tables, lengths) live
        # in one device buffer, 256-byte-aligned regions, so that the
        # end-to-end step moves them from one pinned host buffer with a single
        # copy.
        step_inputs = [step.q, step.k_new, step.v_new, step.slot_mapping, step.block_tables,
                       step.context_lens]
        self.in_host, _ = packed_buffer(step_inputs, pin=True)
        self.in_dev = self.in_host.to(dev)
        _, (self.q, self.k_new, self.v_new, self.slots, self.tables, self.lens) = \
            packed_buffer(step_inputs, storage=self.in_dev)
        self.k_cache, self.v_cache = up(step.k_cache), up(step.v_cache)
        if self.int8:
            self.k_rs, self.v_rs = up(step.k_row_scales), up(step.v_row_scales)
        self.out = torch.empty_like(self.q)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = pa.pa_decode_workspace_size_multi(step.num_seqs, step.num_queries, step.num_heads,
                                               step.head_dim, step.max_context_len)
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        self.pa = pa
        # (the fused calls take no kernel choice: a requested kernel runs the
        # append call, then the decode call with that kernel)
        self.fused = step.num_queries == 1 and step.window == 0 and kernel == "auto"
        # append (not in the fused step), decode, and the split-K merge when a
        # sequence can span more than one partition (at most 4096 sequences:
        # one launch each)
        part = pa.pa_default_partition_size(cd)
        self.launches_per_step = (1 if self.fused else 2) + \
            (1 if math.ceil(step.max_context_len / part) > 1 else 0)

    def append(self, st=None):
        pa, s = self.pa, self.step
        if self.int8:
            pa.pa_reshape_and_cache_int8(self.k_new, self.v_new, self.slots, self.k_cache,
                                         self.v_cache, self.k_rs, self.v_rs,
                                         error_word=self.err, stream=st)
        elif self.fp8:
            pa.pa_reshape_and_cache_fp8(self.k_new, self.v_new, self.slots, self.k_cache,
                                        self.v_cache, s.k_scale, s.v_scale, error_word=self.err,
                                        stream=st)
        else:
            pa.pa_reshape_and_cache(self.k_new, self.v_new, self.slots, self.k_cache,
                                    self.v_cache, error_word=self.err, stream=st)

    def decode(self, st=None):
        pa, s = self.pa, self.step
        common = dict(workspace=self.workspace, error_word=self.err, stream=st)
        mcl = s.max_context_len
        if self.int8:
            pa.pa_decode_int8(self.q, self.k_cache, self.v_cache, self.k_rs, self.v_rs,
                              self.tables, self.lens, s.scale, self.out, mcl, **common)
        elif self.fp8:
            pa.pa_decode_fp8(self.q, self.k_cache, self.v_cache, self.tables, self.lens, s.scale,
                             self.out, mcl, s.k_scale, s.v_scale, kernel=self.kernel, **common)
        elif s.num_queries > 1:
            pa.pa_decode_multi(self.q, self.k_cache, self.v_cache, self.tables, self.lens,
                               s.scale, self.out, mcl, **common)
        elif s.window > 0:
            pa.pa_decode_window(self.q, self.k_cache, self.v_cache, self.tables, self.lens,
                                s.scale, s.window, self.out, mcl, **common)
        else:
            pa.pa_decode(self.q, self.k_cache, self.v_cache, self.tables, self.lens, s.scale,
                         self.out, mcl, kernel=self.kernel, **common)

    def unfused_step(self, st=None):
        self.append(st)
        self.decode(st)

    def run_step(self, st=None):
        pa, s = self.pa, self.step
        if not self.fused:
            return self.unfused_step(st)
        common = dict(workspace=self.workspace, error_word=self.err, stream=st)
        args = (self.k_new, self.v_new, self.slots, self.k_cache, self.v_cache)
        if self.int8:
            pa.pa_append_decode_int8(*args, self.k_rs, self.v_rs, self.q, self.tables, self.lens,
                                     s.scale, self.out, s.max_context_len, **common)
        elif self.fp8:
            pa.pa_append_decode_fp8(*args, self.q, self.tables, self.lens, s.scale, self.out,
                                    s.max_context_len, s.k_scale, s.v_scale, **common)
        else:
            pa.pa_append_decode(*args, self.q, self.tables, self.lens, s.scale, self.out,
                                s.max_context_len, **common)

    def capture(self):
        """CUDA graphs of the step, the attention call alone and the two-call
        step (launches replayed without host gaps, as a serving loop replays a
        decode step); they run the same kernels as the eager calls."""
        import torch
        self.graph_step, self.graph_decode = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        self.graph_unfused = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph_step):
            self.run_step(None)
        with torch.cuda.graph(self.graph_decode):
            self.decode(None)
        with torch.cuda.graph(self.graph_unfused):
            self.unfused_step(None)

    def check_error_word(self, where: str):
        if int(self.err.item()) != 0:
            raise RuntimeError(f"device error word {int(self.err.item()):#x} {where}")


class L2Flusher:
    """Between timed steps: evict the step's data (write a buffer larger than
    L2), then replace the dirty lines with clean ones (read another), so that
    every timed step starts with an L2 holding none of its data and nothing
    to write back."""

    def __init__(self, dev):
        import torch
        self.dirty = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.clean = torch.ones(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev).view(torch.int32)

    def __call__(self, i: int = 1):
        self.dirty.fill_(i & 0xff)
        self.clean.max()


def timed_runs(run, reps, flush, stream) -> list[float]:
    """Milliseconds of `run` per repetition: CUDA events on the launching
    stream around each one, the L2 flushed before each (outside the events)."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for i in range(reps):
        flush(i)
        evs[i][0].record(stream)
        run()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def workload_summary(pa, name: str, args, dev, flush, stream, peak: float,
                     oracle_seconds: float) -> dict:
    """Step and attention-call timings of one more workload (graph replays,
    L2 flushed between them) and the oracle's rate on it."""
    import torch
    step = wl.make(name)
    b = accounting.step_bytes_for(step)
    w = DeviceWorkload(pa, step, dev)
    for _ in range(args.warmup):
        flush()
        w.run_step(stream)
    torch.cuda.synchronize()
    w.check_error_word("during warm-up")
    w.capture()
    step_ms = timed_runs(w.graph_step.replay, args.steps, flush, stream)
    decode_ms = timed_runs(w.graph_decode.replay, args.steps, flush, stream)
    w.check_error_word("in the timed region")
    st, dc = sum(step_ms) / len(step_ms), sum(decode_ms) / len(decode_ms)
    decode_gbs = b.decode / (dc * 1e-3) / 1e9
    res = {
        "cache_dtype": step.cache_dtype, "num_seqs": step.num_seqs,
        "num_queries": step.num_queries, "window": step.window,
        "total_context_rows": int(step.context_lens.sum()),
        "step": "fused append + decode call" if w.fused else "append call + decode call",
        "step_us": round(st * 1e3, 2),
        "decode_call_us": round(dc * 1e3, 2),
        "seqs_per_s": round(step.num_seqs / (st * 1e-3), 1),
        "step_gbs": round(b.total / (st * 1e-3) / 1e9, 2),
        "kv_gbs": round(b.kv / (st * 1e-3) / 1e9, 2),
        "decode_call_gbs": round(decode_gbs, 2),
        "frac_of_measured_hbm": round(decode_gbs / peak, 4),
        "frac_of_nominal_8tbs": round(decode_gbs / NOMINAL_HBM_GBS, 4),
        "algorithmic_bytes_per_call": b.decode,
    }
    if b.kv_unique != b.kv:
        res["kv_unique_gbs"] = round(b.kv_unique / (st * 1e-3) / 1e9, 2)
        res["kv_note"] = "kv_gbs counts each sequence's reads of shared blocks; " \
                         "kv_unique_gbs counts each physical row once"
    del w
    torch.cuda.empty_cache()
    if oracle_seconds > 0:
        res["oracle"] = oracle_rates(step, oracle_seconds)
    return res


def kernel_supported(step: wl.DecodeStep, kernel: str) -> bool:
    """Whether the workload's decode call takes this kernel choice: bf16/fp32
    single-query decode any of mma, simt, generic; FP8 mma or tc; INT8,
    multi-query and window calls only their default."""
    if kernel == "auto":
        return True
    if step.cache_dtype == "fp8":
        return kernel in ("mma", "tc")
    if step.cache_dtype == "int8" or step.num_queries > 1 or step.window > 0:
        return False
    return kernel in ("mma", "simt", "generic")


def run_native(args) -> dict | None:
    import torch
    import paged_kv_cache_29_gb300 as pa

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        import datetime
        dist.init_process_group("nccl", device_id=torch.device("cuda", local),
                                timeout=datetime.timedelta(seconds=PG_TIMEOUT_S))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    step = wl.make(args.workload, seed=wl.WORKLOAD_SEEDS[args.workload] + 1000 * rank)
    if not kernel_supported(step, args.kernel):
        raise SystemExit(f"--kernel {args.kernel} does not apply to workload {args.workload}")
    bytes_ = accounting.step_bytes_for(step)
    cd = step.cache_dtype
    mcl = step.max_context_len
    w = DeviceWorkload(pa, step, dev, args.kernel)
    flush_l2 = L2Flusher(dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        flush_l2()
        w.run_step(stream)
    torch.cuda.synchronize()
    w.check_error_word("during warm-up")
    w.capture()
    for _ in range(args.warmup):
        flush_l2()
        w.graph_step.replay()
    torch.cuda.synchronize()

    K = args.steps
    # Clock soak: untimed back-to-back steps under the clock sampler, so the
    # clocks reported describe this load, then the timed region.
    soak_steps = 0
    if args.clock_soak_s > 0:
        soak_steps = max(1, int(args.clock_soak_s /
                                max(1e-4, _quick_step_seconds(w.graph_step.replay, flush_l2))))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for _ in range(soak_steps):
            w.graph_step.replay()
        # Timed region: K whole steps (append + attention), graph replays.
        step_ms = timed_runs(w.graph_step.replay, K, flush_l2, stream)
    if world > 1:
        torch.distributed.barrier()
    total_ms = sum(step_ms)
    # The attention call alone (roofline of the dominant kernel) and the eager
    # step through the Python binding, for reference.
    decode_ms = timed_runs(w.graph_decode.replay, K, flush_l2, stream)
    decode_avg = sum(decode_ms) / K
    eager_ms = timed_runs(lambda: w.run_step(stream), K, flush_l2, stream)
    unfused_ms = timed_runs(w.graph_unfused.replay, K, flush_l2, stream) if w.fused else step_ms
    append_ms = sum(a - b for a, b in zip(step_ms, decode_ms)) / K
    w.check_error_word("in the timed region")

    # ---- end to end through the public API with host buffers --------------
    # The step's inputs come from one pinned host buffer (the packed layout
    # above), the output goes back to pinned memory.
    out_host = torch.empty(w.out.shape, dtype=w.out.dtype).pin_memory()
    h2d = w.in_host.numel()
    d2h = out_host.numel() * out_host.element_size()

    def e2e_step():
        w.in_dev.copy_(w.in_host, non_blocking=True)
        w.run_step()
        out_host.copy_(w.out, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for i in range(K):
        flush_l2(i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    e2e_total = sum(e2e_ms)

    # Copy-on-write block copies (pa_copy_blocks): COPY_PAIRS random distinct
    # (src, dst) pairs of this pool, after every other measurement (it
    # overwrites pool blocks). INT8 pools carry row scales pa_copy_blocks
    # does not move: not measured there.
    copy_info = None
    if not w.int8:
        pairs = min(COPY_PAIRS, step.num_blocks // 2)
        perm = torch.randperm(step.num_blocks, generator=torch.Generator().manual_seed(7))
        mapping = torch.stack([perm[:pairs], perm[pairs:2 * pairs]], dim=1).to(dev)

        def copy():
            pa.pa_copy_blocks(w.k_cache, w.v_cache, mapping, error_word=w.err, stream=stream)
        for _ in range(args.warmup):
            copy()
        copy_ms = timed_runs(copy, K, flush_l2, stream)
        block_bytes = step.num_kv_heads * step.block_size * step.head_dim * step.elem_bytes
        copy_bytes = pairs * 2 * 2 * block_bytes + pairs * 16   # K and V read + written, pairs
        copy_info = (pairs, copy_bytes, sum(copy_ms) / K)
    torch.cuda.synchronize()
    w.check_error_word("in the timed region")

    (total_ms, e2e_total, decode_avg), (all_bytes, all_seqs) = reduce_over_ranks(
        [total_ms, e2e_total, decode_avg], [float(bytes_.total), float(step.num_seqs)], dev)
    if rank != 0:
        return None

    peak, peak_kind = measured_hbm_gbs()
    ms_per_step = total_ms / K
    value = all_bytes / (ms_per_step * 1e-3) / 1e9
    decode_gbs = bytes_.decode / (decode_avg * 1e-3) / 1e9
    traffic = profiled_traffic(args.workload, args.kernel)
    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8_e4m3" if w.fp8 else ("int8 codes, fp32 row scales" if w.int8 else cd),
        "data": "synthetic (seeded N(0,1) K/V/q; lengths per the workload recipe)",
        "config": {
            "workload": args.workload,
            "num_seqs": step.num_seqs, "num_queries": step.num_queries, "window": step.window,
            "num_heads": step.num_heads,
            "num_kv_heads": step.num_kv_heads, "head_dim": step.head_dim,
            "block_size": step.block_size, "cache_dtype": cd,
            "total_context_rows": int(step.context_lens.sum()),
            "max_context_len": mcl, "partition_size": pa.pa_default_partition_size(cd),
            "kernel": args.kernel,
            "step": ("fused append + decode call (new rows written by the decode kernel)"
                     if w.fused else "append call + decode call"),
            "l2": "between timed steps a 256 MiB buffer is written, then another 256 MiB read (L2 clean, holding none of the step's data); attended K/V also exceed L2",
            "parallelism": f"replicas x{world} (independent batches per GPU)",
        },
        "seqs_per_s": round(all_seqs / (ms_per_step * 1e-3), 1),
        "kv_gbs": round(bytes_.kv * world / (ms_per_step * 1e-3) / 1e9, 2),
        "pct_of_measured_hbm": round(100 * value / peak / world, 2),
        "pct_of_nominal_8tbs": round(100 * value / NOMINAL_HBM_GBS / world, 2),
        "step_breakdown_ms": {"append_and_overlap": round(append_ms, 5),
                              "decode_call": round(decode_avg, 5),
                              "unfused_step": round(sum(unfused_ms) / K, 5)},
        "eager_ms_per_step": round(sum(eager_ms) / K, 5),
        "step_ms_spread": {"median": round(float(np.median(step_ms)), 5),
                           "p10": round(float(np.percentile(step_ms, 10)), 5),
                           "p90": round(float(np.percentile(step_ms, 90)), 5)},
        "timing": "CUDA graph replay of one step per timed iteration; eager_ms_per_step "
                  "is the same step launched through the Python binding",
        "roofline": {
            "bound": "hbm",
            "kernel": "pa_decode call (decode_stream_kernel, combine_kernel)",
            "achieved": round(decode_gbs, 2),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(decode_gbs / peak, 4),
            "frac_of_nominal_8tbs": round(decode_gbs / NOMINAL_HBM_GBS, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_call": bytes_.decode,
            "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)",
        },
        "e2e": {
            "value": round(all_bytes / (e2e_total / K * 1e-3) / 1e9, 2),
            "unit": "GB/s",
            "ms_per_step": round(e2e_total / K, 5),
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "transfers": "inputs: one copy of a packed pinned buffer (q, new K/V rows, slots, "
                         "block tables, lengths); output: one copy to pinned memory",
        },
        "gpu_launches": w.launches_per_step * K,
        "gpu_launches_note": "kernels of this library in the timed graph replays",
        "copy_blocks": None if copy_info is None else {
            "pairs": copy_info[0],
            "bytes_per_call": copy_info[1],
            "ms_per_call": round(copy_info[2], 5),
            "achieved": round(copy_info[1] / (copy_info[2] * 1e-3) / 1e9, 2),
            "unit": "GB/s",
            "frac": round(copy_info[1] / (copy_info[2] * 1e-3) / 1e9 / peak, 4),
            "note": "pa_copy_blocks of random distinct block pairs of this pool (copy-on-write), "
                    "CUDA events per call, L2 flushed between calls",
        },
        "clocks": clocks.summary(),
    }
    if bytes_.kv_unique != bytes_.kv:
        res["kv_unique_gbs"] = round(bytes_.kv_unique / (ms_per_step * 1e-3) / 1e9, 2)
    if world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(step, args.cpu_seconds)
        res["oracle_one_thread"] = oracle_rates(step, args.workload_oracle_seconds)["one_thread"]
    if world == 1 and args.all_workloads:
        del w
        torch.cuda.empty_cache()
        table = {}
        for name in wl.WORKLOADS:
            if name == args.workload:
                continue
            table[name] = workload_summary(
                pa, name, args, dev, flush_l2, stream, peak,
                0.0 if args.no_cpu_baseline else args.workload_oracle_seconds)
        res["workloads"] = table
        res["workloads_note"] = (
            "the other workloads, measured after the headline in the same process the same "
            "way (CUDA-graph replays of the step and of the attention call alone, L2 flushed "
            "between replays); decode_call_gbs = algorithmic attention bytes / attention call "
            "time; oracle: the fp64 C oracle's rate on a bounded sample of each workload at "
            "every host core and at one thread")
    return res


# ---------------------------------------------------------------------------
# the reference arm: the oracle, timed as it stands
# ---------------------------------------------------------------------------

def run_reference(args) -> dict | None:
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    step = wl.make(args.workload)
    threads = os.cpu_count() or 1
    per_step_s = max(1.0, min(args.cpu_seconds, 120.0 / max(args.steps + args.warmup, 1)))
    seqs = oracle_sample_plan(step, per_step_s, threads)
    for _ in range(args.warmup):
        time_oracle(step, seqs, threads)
    times, nbytes = [], 0
    for _ in range(args.steps):
        dt, nbytes = time_oracle(step, seqs, threads)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = nbytes / (ms * 1e-3) / 1e9
    sample = (f"fp64 C oracle (OpenMP, {threads} threads) attention over {len(seqs)} of "
              f"{step.num_seqs} sequences ({int(step.context_lens[seqs].sum())} rows) of "
              f"{step.name} per step")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) K/V/q; lengths per the workload recipe)",
        "config": {"workload": args.workload, "num_seqs": len(seqs),
                   "sampled_from": step.num_seqs, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main() -> None:
    ap = argparse.ArgumentParser(description="paged decode attention benchmark")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="8b_gqa", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--kernel", default="auto", choices=["auto", "mma", "simt", "generic", "tc"],
                    help="decode kernel (bf16/fp32 caches: mma, simt, generic; FP8: mma, tc)")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target oracle time of the CPU baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload-oracle-seconds", type=float, default=1.5,
                    help="host seconds of each per-workload oracle sample (all cores, 1 thread)")
    ap.add_argument("--all-workloads", action=argparse.BooleanOptionalAction, default=True,
                    help="also measure every other workload (N=1 only) into `workloads`")
    ap.add_argument("--clock-soak-s", type=float, default=1.0,
                    help="seconds of untimed back-to-back steps under the clock sampler "
                         "before the timed region (0 = none)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, _, _ = dist_env()
    if args.gpus != world and world > 1:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    res = run_reference(args) if args.impl == "reference" else run_native(args)
    if res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl == "native":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
