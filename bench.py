#!/usr/bin/env python
"""Benchmark of paged decode attention on GB300 (one JSON line on rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--headline-only] [--no-cpu-baseline]

A step is one decode call over one batch of the named workload (all of the
path: the persistent decode kernel, and the LSE-merge kernel where the plan
has split units). The headline workload is the largest single-GPU one, MLA
decode BF16 with B=512, q_len 1, 128 heads and L=4096; every other workload
(tiny, GQA-8, ragged split-KV, FP8 KV, MLA q_len 2, FP8 latent MLA, prefill,
and three appends) gets an entry of its own under "workloads", with its
rooflines and, on a single-GPU run, the FP64 oracle's time on the host cores.
Inputs are seeded synthetic tensors made on the device; the L2 is flushed (a
256 MiB write, then a 256 MiB read of another buffer) between timed calls,
outside the timed events. Device time is taken with CUDA events around
CUDA-graph replays of the call on the stream the kernels run on.

--gpus N runs N independent replicas, one rank per GPU (the path has no
cross-GPU exchange): under torchrun WORLD_SIZE must equal N; outside it the
script starts the N ranks itself. The reported time is the max over ranks
and ``value`` is the whole job's time per call (time / (steps x N)).

``--impl reference`` times the FP64 CPU oracle instead, on bounded samples of
the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention: µs/call and KV GB/s as % of GB300 8 TB/s HBM roofline"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20

WORKLOAD_TEXT = {
    "tiny": "tiny paged GQA decode: B=2, Hq=8, Hkv=1, D=128, P=16, NHD, seq_lens 37/64",
    "gqa8": "GQA-8 decode BF16: B=32, q_len=1, Hq=64, Hkv=8, D=128, HND, P=32, L=4096",
    "ragged": "ragged split-KV decode BF16: B=128, q_len 1/2/4, Hq=32, Hkv=8, D=128, P=64, HND, L log-uniform [1,16384]",
    "fp8": "FP8 KV decode: B=16, q_len=1, Hq=64, Hkv=8, D=128, HND, P=64, L=4096, e4m3 K/V",
    "mla1": "MLA decode BF16: B=512, q_len=1, 128 heads, 576/512, P=64, L=4096",
    "mla2": "MLA decode BF16: B=512, q_len=2, 128 heads, 576/512, P=64, L=4096",
    "mla_fp8": "FP8 latent MLA decode: B=128, q_len=1, 128 heads, E4M3 query and latent cache, 576/512, P=64, L=4096",
    "prefill": "paged prefill BF16: B=4, q_len=511 over L=2047 (causal), Hq=64, Hkv=8, D=128, HND, P=32",
}
# workloads whose bound is the tensor pipe rather than HBM
TENSOR_BOUND = ("prefill",)
# workloads run by the tensor-core prefill kernel (paged_prefill_run)
PREFILL_KERNEL = ("prefill",)


# the paged KV append (the step before decode), timed on its own
APPEND_TEXT = {
    "append_bf16": "paged KV append BF16: 32 requests x 512 new tokens, Hkv 8, D 128, HND, P 32, 4096-page pools",
    "append_e4m3": "paged KV append E4M3 (x / scale, RN-even, saturating): 32 x 512 new tokens, Hkv 8, D 128, HND, P 32",
}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops():
    """Burst cuBLAS bf16 rate (the peak for a kernel timed on its own)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def attention_flops(x):
    """Algorithmic flops of one call: every query row's visible keys, 2 flops
    per multiply-add of Q.K and of P.V (row i of a request with q_len new
    tokens sees keys 0 .. L - q_len + i)."""
    import numpy as np
    seq = x.seq_lens_host().astype(np.int64)
    ql = np.diff(x.q_indptr_host()).astype(np.int64)
    # sum over i of (L - q + i + 1) = q (L - q + 1) + q (q - 1) / 2
    keys = int(np.sum(ql * (seq - ql + 1) + ql * (ql - 1) // 2))
    return 2.0 * keys * x.num_q_heads * (x.head_dim_qk + x.head_dim_v)


# the sources that decide what each kernel reads and writes (kernel, shared
# device helpers, workspace layout, planner, launch code)
_SHARED_SOURCES = ("device_common.cuh", "kernels.h", "ws_layout.h", "plan.cpp", "plan_internal.h", "api.cu")
KERNEL_SOURCES = {"gqa": ("decode_gqa.cu",) + _SHARED_SOURCES, "mla": ("decode_mla.cu",) + _SHARED_SOURCES,
                  "prefill": ("prefill_gqa.cu",) + _SHARED_SOURCES,
                  "append": ("append.cu", "kernels.h")}


def kernel_source_hash(kernel="gqa"):
    """Digest of the sources behind one kernel. A stored DRAM-traffic figure
    is only reported while they still hash to the value it was captured at."""
    import hashlib
    csrc = os.path.join(ROOT, "paged_kv_cache_199_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def dram_traffic(workload, batch=None):
    """Per-launch DRAM bytes (read + write) of the workload's kernel from the
    committed ncu summary, or None when none was recorded, the batch differs
    from the capture, or the kernel's sources changed since."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    w = d.get("workloads", {}).get(workload)
    if w is None or batch is not None or w.get("source_hash") != kernel_source_hash(w.get("kernel", "gqa")):
        return None
    return w.get("bytes_per_launch")


_BYTE_UNITS = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9}
WORKLOAD_KERNEL = {"tiny": "gqa", "gqa8": "gqa", "ragged": "gqa", "fp8": "gqa", "mla1": "mla", "mla2": "mla",
                   "mla_fp8": "mla", "prefill": "prefill", "append_bf16": "append", "append_e4m3": "append"}


def record_traffic(report, workload, scale=1, captured_batch=None):
    """Writes one workload's per-launch DRAM bytes into profiles/dram_traffic.json
    from an ncu report (any capture holding dram__bytes_read.sum and
    dram__bytes_write.sum of the workload's kernel; the mean over its
    launches), stamped with the current source hash of that kernel. `scale`
    multiplies the figure when a smaller batch was captured."""
    import csv
    import io
    import subprocess
    out = subprocess.run(["ncu", "-i", report, "--page", "raw", "--csv"], capture_output=True, text=True, check=True)
    rows = list(csv.reader(io.StringIO(out.stdout)))
    head, units, data = rows[0], rows[1], rows[2:]
    col = {n: i for i, n in enumerate(head)}
    for m in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
        if m not in col:
            raise SystemExit(f"{report}: no {m} (capture with --set full or --metrics {m})")

    def mean_bytes(metric):
        i = col[metric]
        vals = [float(r[i].replace(",", "")) * _BYTE_UNITS[units[i]] for r in data if len(r) > i and r[i]]
        return sum(vals) / len(vals)

    rd, wr = mean_bytes("dram__bytes_read.sum"), mean_bytes("dram__bytes_write.sum")
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    with open(path) as f:
        d = json.load(f)
    kernel = WORKLOAD_KERNEL[workload]
    e = {"kernel": kernel, "source_hash": kernel_source_hash(kernel), "bytes_per_launch": int(round((rd + wr) * scale)),
         "read": int(round(rd * scale)), "write": int(round(wr * scale))}
    if captured_batch is not None:
        e["scaled_from_batch"] = captured_batch
    d.setdefault("workloads", {})[workload] = e
    with open(path, "w") as f:
        json.dump(d, f, indent=1)
        f.write("\n")
    print(json.dumps({workload: e}))
    return 0


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.25)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        med = statistics.median(sm)
        # a run with a throttle reason or SM clocks below 0.7 x max is not a valid measurement
        valid = not (reasons & {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}) and med >= 0.7 * max(mx)
        return {"sm_mhz": med, "sm_max_mhz": max(mx), "reasons": sorted(reasons), "samples": len(sm),
                "valid": valid}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_us_per_call(per_rank_total_us: float, steps: int, world: int) -> float:
    """Whole-job time per call for `world` independent replicas that each ran
    `steps` calls in (at most) `per_rank_total_us`."""
    return per_rank_total_us / (steps * world)


# ---------------------------------------------------------------------------
# reference arm: the FP64 oracle on the host cores
# ---------------------------------------------------------------------------

def host_cpu_info():
    """The host's processor as the oracle timing saw it: logical CPUs, the
    OpenMP thread setting and the CPU model (``model name`` in /proc/cpuinfo;
    Arm hosts print no model line there, so lscpu's is used)."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if not model:
        try:
            outp = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in outp.splitlines():
                if line.strip().lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    import platform
    return {"nproc": os.cpu_count(), "omp_num_threads": os.environ.get("OMP_NUM_THREADS"),
            "cpu_model": model or platform.processor() or platform.machine()}


def oracle_sample_us_per_call(inputs, budget_s: float = 12.0, max_reqs=None, full_tokens=None):
    """Time the oracle on groups of whole requests (as many per call as it has
    threads, longest first, so that every core has work) until ~budget_s of
    host time, and scale by cached tokens to `full_tokens` (default: the
    batch's own). Returns (us_per_call, sample, cores)."""
    import numpy as np

    import oracle
    from tests.helpers import run_oracle, subset  # test-side marshalling of the same arrays
    cores = oracle.max_threads()
    lens = inputs.seq_lens_host().astype(np.int64)
    order = [int(b) for b in np.argsort(-lens, kind="stable")]
    if max_reqs is not None:
        order = order[:max_reqs]
    done, t_total, kv_done = 0, 0.0, 0
    group = max(1, cores)
    for g0 in range(0, len(order), group):
        reqs = order[g0:g0 + group]
        a = subset(inputs, reqs)
        t0 = time.perf_counter()
        run_oracle(inputs, arrays=a)
        t_total += time.perf_counter() - t0
        done += len(reqs)
        kv_done += int(lens[reqs].sum())
        if t_total >= budget_s:
            break
    total_kv = int(lens.sum()) if full_tokens is None else int(full_tokens)
    us = t_total / max(kv_done, 1) * total_kv * 1e6
    sample = (f"{done} of {inputs.batch} requests ({kv_done} of {int(lens.sum())} cached tokens) timed in "
              f"calls of up to {group} requests, scaled by cached tokens to {total_kv}")
    return us, sample, cores


def cpu_baseline_for(name, full_inputs, budget_s, max_batch=32):
    """The oracle, as it stands, on a bounded sample of the workload: a copy
    of at most `max_batch` requests of the same shapes generated on the host,
    timed request by request and scaled to the full workload's cached tokens."""
    from paged_kv_cache_199_gb300 import workloads as W
    batch = full_inputs.batch
    xc = W.workload(name, device="cpu", batch=min(batch, max_batch) if batch > max_batch else None)
    full_tokens = int(full_inputs.seq_lens.to("cpu").long().sum().item())
    us, sample, cores = oracle_sample_us_per_call(xc, budget_s=budget_s, full_tokens=full_tokens)
    if xc.batch != batch:
        sample = f"a {xc.batch}-request copy of the workload's shapes: " + sample
    d = {"value": round(us, 1), "unit": "us/call", "cores": cores, "kind": "oracle", "sample": sample}
    d.update(host_cpu_info())
    return d


def oracle_append_us(e4m3, runs):
    """Median host time (us) of the oracle's append on the shapes of run_append."""
    import numpy as np

    import oracle
    rng = np.random.default_rng(11)
    batch, Hkv, D, P, pages, n_new = 32, 8, 128, 32, 4096, 512
    per_req = pages // batch
    elem = np.uint8 if e4m3 else np.uint16
    k_pool = np.zeros((pages, Hkv, P, D), elem)
    v_pool = np.zeros_like(k_pool)
    table = rng.permutation(pages).astype(np.int32).reshape(batch, per_req)
    seq_lens = np.full(batch, per_req * P, np.int32)
    qi = (np.arange(batch + 1) * n_new).astype(np.int32)
    k_new = rng.integers(0x3000, 0x4000, (batch * n_new, Hkv, D)).astype(np.uint16)
    v_new = rng.integers(0x3000, 0x4000, (batch * n_new, Hkv, D)).astype(np.uint16)
    vals = []
    for _ in range(max(runs, 1)):
        t0 = time.perf_counter()
        oracle.paged_append(k_new, v_new, table, seq_lens, qi, k_pool, v_pool, num_kv_heads=Hkv, head_dim=D,
                            page_size=P, layout=oracle.HND, kv_dtype=oracle.E4M3 if e4m3 else oracle.BF16,
                            k_scale=0.05, v_scale=0.05, zero_tail=True)
        vals.append((time.perf_counter() - t0) * 1e6)
    return statistics.median(vals)


def run_reference_append(args):
    """The oracle's append on the host cores, the same shapes as run_append."""
    e4m3 = args.workload == "append_e4m3"
    v = oracle_append_us(e4m3, args.steps)
    line = {"impl": "reference", "metric": "paged KV append: us/call", "value": round(v, 1), "unit": "us/call",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(v / 1e3, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if e4m3 else "bf16",
            "data": "synthetic", "config": {"workload": APPEND_TEXT[args.workload]},
            "cpu_baseline": {"value": round(v, 1), "unit": "us/call", "cores": 1, "kind": "oracle",
                             "sample": "the whole append (single-threaded C)"},
            "e2e": {"value": round(v, 1), "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    if args.workload in APPEND_TEXT:
        return run_reference_append(args)
    from paged_kv_cache_199_gb300 import workloads as W
    # a copy of at most 32 requests of the workload's shapes, scaled to its cached tokens
    nb = _full_batch(args.workload)
    x = W.workload(args.workload, device="cpu", batch=min(32, nb) if nb > 32 else None)
    full_tokens = _full_tokens(args.workload)
    # every step is a bounded sample, so that the K + W steps end in a couple of minutes
    per_step = max(0.5, min(args.ref_budget, 120.0 / max(args.steps, 1)))
    for _ in range(max(args.warmup, 0)):
        oracle_sample_us_per_call(x, budget_s=min(per_step, 2.0), max_reqs=1, full_tokens=full_tokens)
    vals = []
    sample = cores = None
    for _ in range(args.steps):
        us, sample, cores = oracle_sample_us_per_call(x, budget_s=per_step, full_tokens=full_tokens)
        vals.append(us)
    v = statistics.median(vals)
    cpu = {"value": round(v, 1), "unit": "us/call", "cores": cores, "kind": "oracle", "sample": sample}
    cpu.update(host_cpu_info())
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": "us/call",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(v / 1e3, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD_TEXT[args.workload]},
        "cpu_baseline": cpu,
        "e2e": {"value": round(v, 1), "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _full_batch(name):
    from paged_kv_cache_199_gb300 import workloads as W
    return {"tiny": 2, "gqa8": 32, "ragged": 128, "fp8": 16, "mla1": 512, "mla2": 512, "mla_fp8": 128,
            "prefill": 4}[name] if name in W.WORKLOADS else 1


def _full_tokens(name):
    """Cached tokens of the full workload, from its length recipe (no pools made)."""
    from paged_kv_cache_199_gb300 import workloads as W
    if name == "ragged":
        L, _ = W.ragged_lengths(3, 128, 16384)
        return int(L.sum())
    if name == "tiny":
        return 37 + 64
    per = {"gqa8": 4096, "fp8": 4096, "mla1": 4096, "mla2": 4096, "mla_fp8": 4096, "prefill": 2047}[name]
    return per * _full_batch(name)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def flush_l2(flush):
    """Evict the L2 between timed calls: write a buffer larger than the L2,
    then read another, so that the next call starts on a clean cache (no
    dirty lines of the flush left to be written back during the call)."""
    flush[0].add_(1)
    flush[1].sum(dtype=torch_float32())


def torch_float32():
    import torch
    return torch.float32


def time_device(dec, out, lse, steps, warmup, flush, use_graph=True):
    """Per-call device time (us) with an L2 flush between calls."""
    import torch
    stream = torch.cuda.current_stream()
    graph = None
    if use_graph:
        try:
            dec.run(out, lse)  # warm the launch path outside capture
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                dec.run(out, lse)
            torch.cuda.synchronize()
        except Exception:
            graph = None
    call = graph.replay if graph is not None else (lambda: dec.run(out, lse))
    for _ in range(warmup):
        flush_l2(flush)
        call()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush_l2(flush)
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        call()
        e.record(stream)
        e.synchronize()
        times.append(s.elapsed_time(e) * 1e3)
    return times, graph is not None


def time_e2e(dec, x, steps, warmup):
    """The same call through the public API with host buffers: pinned
    host->device copies of the step's inputs (query, block table, lengths),
    the decode, and a device->host read of the output (+ LSE)."""
    import torch
    stream = torch.cuda.current_stream()
    q_h = x.q.cpu().pin_memory()
    bt_h = x.block_tables.cpu().pin_memory()
    sl_h = x.seq_lens.cpu().pin_memory()
    qi_h = x.q_indptr.cpu().pin_memory()
    q_d = torch.empty_like(x.q)
    bt_d = torch.empty_like(x.block_tables)
    sl_d = torch.empty_like(x.seq_lens)
    qi_d = torch.empty_like(x.q_indptr)
    out, lse = dec.alloc_outputs(True)
    out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    lse_h = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in (q_h, bt_h, sl_h, qi_h))
    d2h = out.numel() * out.element_size() + lse.numel() * lse.element_size()

    def step():
        q_d.copy_(q_h, non_blocking=True)
        bt_d.copy_(bt_h, non_blocking=True)
        sl_d.copy_(sl_h, non_blocking=True)
        qi_d.copy_(qi_h, non_blocking=True)
        dec.run(out, lse, q=q_d, seq_lens=sl_d, block_tables=bt_d, q_indptr=qi_d)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(steps):
        step()
    e.record(stream)
    e.synchronize()
    return s.elapsed_time(e) * 1e3 / steps, h2d, d2h


def time_e2e_pipelined(dec, x, steps, warmup):
    """The same call through the public API with host buffers, as a serving
    loop would run it: two sets of device inputs and outputs, the
    host->device copies of step i+1 and the device->host read of step i-1 on
    copy streams while step i decodes. The decodes stay in order on one
    stream (they share the plan's workspace). Every step still copies its own
    inputs (query, block table, lengths) from pinned host memory and reads
    its own output and LSE back; the timed region ends when the last read is
    done."""
    import torch
    cin, comp, cout = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    host_in = [t.cpu().pin_memory() for t in (x.q, x.block_tables, x.seq_lens, x.q_indptr)]
    dev_in = [[torch.empty_like(t) for t in (x.q, x.block_tables, x.seq_lens, x.q_indptr)] for _ in range(2)]
    outs = [dec.alloc_outputs(True) for _ in range(2)]
    host_out = [(torch.empty(o.shape, dtype=o.dtype, pin_memory=True),
                 torch.empty(l.shape, dtype=l.dtype, pin_memory=True)) for o, l in outs]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    torch.cuda.synchronize()

    def step(i):
        b = i % 2
        q_d, bt_d, sl_d, qi_d = dev_in[b]
        out, lse = outs[b]
        with torch.cuda.stream(cin):
            if i >= 2:
                cin.wait_event(ev_comp[b])   # step i-2's decode is done with these inputs
            for d, h in zip(dev_in[b], host_in):
                d.copy_(h, non_blocking=True)
            ev_in[b].record(cin)
        comp.wait_event(ev_in[b])
        if i >= 2:
            comp.wait_event(ev_out[b])       # step i-2's results have been read out
        dec.run(out, lse, q=q_d, seq_lens=sl_d, block_tables=bt_d, q_indptr=qi_d, stream=comp)
        ev_comp[b].record(comp)
        with torch.cuda.stream(cout):
            cout.wait_event(ev_comp[b])
            host_out[b][0].copy_(out, non_blocking=True)
            host_out[b][1].copy_(lse, non_blocking=True)
            ev_out[b].record(cout)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(cin)
    for i in range(warmup, warmup + steps):
        step(i)
    e.record(cout)
    e.synchronize()
    torch.cuda.synchronize()
    b = (warmup + steps - 1) % 2   # the last step's results reached the host intact
    if not (torch.equal(host_out[b][0], outs[b][0].cpu()) and torch.equal(host_out[b][1], outs[b][1].cpu())):
        raise RuntimeError("end-to-end timing: the read-back differs from the device output")
    return s.elapsed_time(e) * 1e3 / steps


def bench_workload(name, args, world, rank, flush, want_e2e=True):
    import torch

    from paged_kv_cache_199_gb300 import binding as B
    from paged_kv_cache_199_gb300 import workloads as W
    x = W.workload(name, device="cuda", batch=args.batch if name == args.workload else None)
    dec = B.PagedDecode(x, prefill=name in PREFILL_KERNEL and not args.decode_kernel)
    out, lse = dec.alloc_outputs(True)
    dec.run(out, lse)
    torch.cuda.synchronize()
    code, info = dec.read_error()
    if code != 0:
        raise RuntimeError(f"{name}: device error {B.DEVICE_ERRORS.get(code, code)} (request {info})")
    times, graphed = time_device(dec, out, lse, args.steps, args.warmup, flush)
    res = {"times_us": times, "graphed": graphed, "inputs": x, "dec": dec,
           "launches_per_call": dec.info.launches_per_run}
    if want_e2e:
        res["e2e_serial_us"], res["h2d"], res["d2h"] = time_e2e(dec, x, max(args.steps, 3), max(args.warmup, 1))
        res["e2e_us"] = time_e2e_pipelined(dec, x, max(args.steps, 3), max(args.warmup, 2))
    return res


def bench_append(kv_dtype, n_new, steps, warmup, flush, with_e2e=False):
    """Paged KV append of n_new tokens for each of 32 requests into pools of the
    GQA-8 geometry (4096 pages, HND, P=32, Hkv=8, D=128); algorithmic bytes are
    the new bf16 rows read plus the pool rows written (K and V)."""
    import torch

    from paged_kv_cache_199_gb300 import binding as B
    g = torch.Generator(device="cuda").manual_seed(11)
    batch, Hkv, D, P, pages = 32, 8, 128, 32, 4096
    per_req = pages // batch
    L0 = per_req * P - n_new            # cached tokens before the append
    dt = torch.bfloat16 if kv_dtype == B.PD_KV_BF16 else torch.uint8
    k_pool = torch.zeros((pages, Hkv, P, D), dtype=dt, device="cuda")
    v_pool = torch.zeros_like(k_pool)
    table = torch.randperm(pages, device="cuda", generator=g).to(torch.int32).view(batch, per_req)
    seq_lens = torch.full((batch,), L0 + n_new, dtype=torch.int32, device="cuda")
    q_indptr = (torch.arange(batch + 1, device="cuda", dtype=torch.int32) * n_new)
    k_new = torch.randn((batch * n_new, Hkv, D), generator=g, device="cuda").to(torch.bfloat16)
    v_new = torch.randn((batch * n_new, Hkv, D), generator=g, device="cuda").to(torch.bfloat16)
    ks = torch.tensor([0.05], device="cuda")
    vs = torch.tensor([0.05], device="cuda")
    err = torch.zeros(2, dtype=torch.int32, device="cuda")

    def call():
        B.paged_kv_append(k_new, v_new, q_indptr, seq_lens, table, k_pool, v_pool, num_kv_heads=Hkv,
                          head_dim=D, page_size=P, layout=B.PD_LAYOUT_HND, kv_dtype=kv_dtype, k_scale=ks,
                          v_scale=vs, zero_tail=True, error_word=err)
    for _ in range(warmup):
        flush_l2(flush)
        call()
    torch.cuda.synchronize()
    times = []
    stream = torch.cuda.current_stream()
    for _ in range(steps):
        flush_l2(flush)
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        call()
        e.record(stream)
        e.synchronize()
        times.append(s.elapsed_time(e) * 1e3)
    assert err.tolist() == [0, 0]
    us = statistics.fmean(times)    # events step by about 2 us: the mean resolves below a step
    elem = 2 if kv_dtype == B.PD_KV_BF16 else 1
    nbytes = 2 * batch * n_new * Hkv * D * (2 + elem)
    if not with_e2e:
        return us, nbytes
    # end to end: the new rows come from pinned host memory, the error word goes back
    k_host = k_new.cpu().pin_memory()
    v_host = v_new.cpu().pin_memory()
    err_host = torch.zeros(2, dtype=torch.int32).pin_memory()
    e2e = []
    for i in range(steps + 1):
        flush_l2(flush)
        torch.cuda.synchronize()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        k_new.copy_(k_host, non_blocking=True)
        v_new.copy_(v_host, non_blocking=True)
        call()
        err_host.copy_(err, non_blocking=True)
        e.record(stream)
        e.synchronize()
        if i > 0:
            e2e.append(s.elapsed_time(e) * 1e3)
    h2d = k_host.numel() * 2 + v_host.numel() * 2
    return us, nbytes, statistics.fmean(e2e), h2d, 8


def run_append(args, world, rank, local, flush, peak, peak_kind):
    """--workload append_*: the paged KV append alone (one launch per call)."""
    import torch

    from paged_kv_cache_199_gb300 import binding as B
    dtype = B.PD_KV_BF16 if args.workload == "append_bf16" else B.PD_KV_FP8_E4M3
    barrier(world)
    with ClockSampler(local) as clocks:
        us, nbytes, e2e_us, h2d, d2h = bench_append(dtype, 512, args.steps, args.warmup, flush, with_e2e=True)
        barrier(world)
    us = reduce_max(us, world)
    gbs = nbytes / (us * 1e-6) / 1e9
    line = {"metric": "paged KV append: us/call", "value": round(us / world, 2), "unit": "us/call", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 5),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if dtype == B.PD_KV_BF16 else "e4m3", "data": "synthetic",
            "config": {"workload": APPEND_TEXT[args.workload],
                       "l2": "flushed between timed calls (256 MiB write, then 256 MiB read of another buffer)"},
            "clocks": clocks.summary(), "gpu_launches": args.steps,
            "e2e": {"value": round(reduce_max(e2e_us, world) / world, 2), "unit": "us/call",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                         "traffic": dram_traffic(args.workload), "kernel": "paged_append_kernel",
                         "note": "new bf16 rows read + pool rows written (K and V) / mean call time"}}
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        us_cpu = oracle_append_us(args.workload == "append_e4m3", 3)
        line["cpu_baseline"] = {"value": round(us_cpu, 1), "unit": "us/call", "cores": 1, "kind": "oracle",
                                "sample": "the whole append, 3 runs (single-threaded C), median"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def roofline_for(name, x, mean_us, kname, args):
    """HBM and tensor rooflines of one call: algorithmic bytes (visible K/V rows,
    Q, out, LSE, block table) or flops (2 per multiply-add of Q.K and P.V over
    every row's visible keys) per call / mean device time of the call. The
    first is the one that bounds the workload."""
    peak, peak_kind = measured_peaks()
    tpeak, tkind = measured_bf16_tflops()
    kv = x.kv_bytes()
    q_elem = 1 if x.q.dtype.itemsize == 1 else 2
    other = (x.q.numel() * q_elem + x.total_q * x.num_q_heads * (x.head_dim_v * 2 + 4)
             + x.block_tables.numel() * 4)
    gbs = (kv + other) / (mean_us * 1e-6) / 1e9
    tf = attention_flops(x) / (mean_us * 1e-6) / 1e12
    traffic = dram_traffic(name, args.batch if name == args.workload else None)
    hbm = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
           "peak_kind": peak_kind, "traffic": traffic, "kernel": kname,
           "note": "algorithmic bytes (visible K/V rows + Q + out + LSE + table) per call / mean device time "
                   "of the call (the decode launch, plus the merge launch where the plan has one)"}
    tensor = {"bound": "tensor", "achieved": round(tf, 1), "peak": tpeak, "unit": "TFLOP/s",
              "frac": round(tf / tpeak, 4), "peak_kind": tkind, "traffic": traffic, "kernel": kname,
              "note": "algorithmic flops (2 per multiply-add of Q.K and P.V over every row's visible keys) per "
                      "call / mean device time of the call; peak = burst cuBLAS bf16"}
    if name in TENSOR_BOUND:
        return tensor, hbm
    return hbm, tensor


def kernel_name(name, x, args):
    if name in PREFILL_KERNEL and not args.decode_kernel:
        return "gqa_prefill_kernel"
    return "gqa_decode_kernel" if x.kind == "gqa" else "mla_decode_kernel"


def workload_entry(name, r, args, cpu_budget):
    """One workload's figures: device time per call, KV GB/s, rooflines and,
    on a single-GPU run, the oracle's time on the host cores."""
    import numpy as np
    x = r["inputs"]
    times = r["times_us"]
    med = statistics.median(times)
    mean = statistics.fmean(times)
    kv = x.kv_bytes()
    primary, secondary = roofline_for(name, x, mean, kernel_name(name, x, args), args)
    # CUDA events advance in steps of about 2 us on this hardware: the mean of
    # many calls resolves a call's time below one step, the median does not
    e = {"config": WORKLOAD_TEXT[name], "us_per_call": round(mean, 2), "median_us": round(med, 2),
         "p10_us": round(float(np.percentile(times, 10)), 2), "p90_us": round(float(np.percentile(times, 90)), 2),
         "kv_bytes": kv, "kv_gbs": round(kv / (mean * 1e-6) / 1e9, 1),
         "pct_of_8tbs": round(100.0 * kv / (mean * 1e-6) / 1e9 / NOMINAL_HBM_GBS, 1),
         "tflops": round(attention_flops(x) / (mean * 1e-6) / 1e12, 1),
         "launches_per_call": r["launches_per_call"], "roofline": primary,
         "roofline_" + secondary["bound"]: secondary}
    if cpu_budget:
        e["cpu_baseline"] = cpu_baseline_for(name, x, cpu_budget)
    return e


def run_ours(args, world, rank, local):
    import torch

    from paged_kv_cache_199_gb300 import binding as B
    from paged_kv_cache_199_gb300 import build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    build.build()
    B.load()
    flush = (torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda"),
             torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda"))
    peak, peak_kind = measured_peaks()

    if args.workload in APPEND_TEXT:
        return run_append(args, world, rank, local, flush, peak, peak_kind)

    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t0 = time.perf_counter()
        main = bench_workload(args.workload, args, world, rank, flush)
        torch.cuda.synchronize()
        barrier(world)
        wall = time.perf_counter() - t0
    import numpy as np
    x = main["inputs"]
    dev_us = statistics.median(main["times_us"])
    mean_us = statistics.fmean(main["times_us"])
    total_us = reduce_max(sum(main["times_us"]), world)
    value = aggregate_us_per_call(total_us, args.steps, world)
    kv = x.kv_bytes()
    e2e_us = reduce_max(main["e2e_us"], world) / world
    e2e_serial_us = reduce_max(main["e2e_serial_us"], world) / world
    primary, secondary = roofline_for(args.workload, x, mean_us, kernel_name(args.workload, x, args), args)
    single = rank == 0 and world == 1 and not args.no_cpu_baseline

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "us/call", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean_us / 1e3, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": x.kv_dtype,
        "data": "synthetic (seeded, generated on device)",
        "config": {"workload": WORKLOAD_TEXT[args.workload] + (f" (batch overridden to {x.batch})" if args.batch else ""),
                   "batch": x.batch,
                   "kv_bytes": kv, "l2": "flushed between timed calls (256 MiB write, then 256 MiB read of another buffer)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "timing": "CUDA events around CUDA-graph replay" if main["graphed"] else "CUDA events"},
        "kv_gbs": round(kv / (dev_us * 1e-6) / 1e9, 1),
        "pct_of_8tbs": round(100.0 * kv / (dev_us * 1e-6) / 1e9 / NOMINAL_HBM_GBS, 1),
        "median_us": round(dev_us, 2),
        "p10_us": round(float(np.percentile(main["times_us"], 10)), 2),
        "p90_us": round(float(np.percentile(main["times_us"], 90)), 2),
        "samples_us": [round(t, 2) for t in main["times_us"]],
        "clocks": clocks.summary(),
        "e2e": {"value": round(e2e_us, 2), "unit": "us/call", "h2d_bytes_per_step": main["h2d"],
                "d2h_bytes_per_step": main["d2h"],
                "mode": "pipelined: step i+1's host-to-device copies and step i-1's read-back overlap step i's "
                        "decode (two buffer sets); every step copies its inputs and reads its results",
                "serial_value": round(e2e_serial_us, 2)},
        "gpu_launches": main["launches_per_call"] * args.steps,
        "tflops": round(attention_flops(x) / (mean_us * 1e-6) / 1e12, 1),
        "roofline": primary,
        "roofline_" + secondary["bound"]: secondary,
        "wall_s": round(wall, 3),
    }
    if args.all_workloads:
        extra = {args.workload: workload_entry(args.workload, main, args, 0)}
        del main
        torch.cuda.empty_cache()
        for name in WORKLOAD_TEXT:
            if name == args.workload:
                continue
            try:
                r = bench_workload(name, args, world, rank, flush, want_e2e=False)
            except B.PdError as e:
                extra[name] = {"unavailable": str(e)}
                continue
            extra[name] = workload_entry(name, r, args, 0)
            del r
            torch.cuda.empty_cache()
        for label, dtype_code, n_new in (("append_bf16_32x512", B.PD_KV_BF16, 512),
                                         ("append_e4m3_32x512", B.PD_KV_FP8_E4M3, 512),
                                         ("append_bf16_32x1", B.PD_KV_BF16, 1)):
            us, nbytes = bench_append(dtype_code, n_new, args.steps, args.warmup, flush)
            gbs = nbytes / (us * 1e-6) / 1e9
            extra[label] = {"config": f"paged KV append, 32 requests x {n_new} new tokens, Hkv 8, D 128, HND P 32",
                            "us_per_call": round(us, 2), "bytes": nbytes, "gbs": round(gbs, 1),
                            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                                         "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                                         "kernel": "paged_append_kernel",
                                         "traffic": dram_traffic(label.rsplit("_", 1)[0]) if n_new == 512 else None}}
            torch.cuda.empty_cache()
        if single:
            # the oracle on the host cores, beside every GPU figure (bounded samples)
            for name in WORKLOAD_TEXT:
                if "unavailable" in extra.get(name, {}):
                    continue
                budget = args.ref_budget if name == args.workload else args.cpu_budget
                xg = W_workload_shape(name)
                extra[name]["cpu_baseline"] = cpu_baseline_for(name, xg, budget)
        line["workloads"] = extra
    if single:
        line["cpu_baseline"] = (line["workloads"][args.workload]["cpu_baseline"] if args.all_workloads
                                else cpu_baseline_for(args.workload, W_workload_shape(args.workload), args.ref_budget))
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


class _Shape:
    """The batch size and total cached tokens of a workload (what the oracle
    sample is scaled to), without its pools."""

    def __init__(self, name):
        import torch
        self.batch = _full_batch(name)
        self.seq_lens = torch.tensor([_full_tokens(name)], dtype=torch.int64)


def W_workload_shape(name):
    return _Shape(name)


def relaunch_under_torchrun(n, argv):
    """`--gpus N` outside torchrun: start N replica ranks of this script (one
    per GPU, 127.0.0.1 rendezvous) and return rank 0's exit code."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(WORKLOAD_TEXT) + list(APPEND_TEXT), default="mla1")
    ap.add_argument("--all-workloads", dest="all_workloads", action="store_true", default=True,
                    help="also time every other workload (the default)")
    ap.add_argument("--headline-only", dest="all_workloads", action="store_false",
                    help="time the named workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=12.0,
                    help="oracle seconds per reference step, and for the headline's cpu_baseline")
    ap.add_argument("--cpu-budget", type=float, default=3.0,
                    help="oracle seconds for each other workload's cpu_baseline")
    ap.add_argument("--decode-kernel", action="store_true",
                    help="run the prefill workload through paged_decode_run (16-row mma.sync units) "
                         "instead of the tensor-core prefill kernel")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size (profiling a smaller case)")
    ap.add_argument("--record-traffic", metavar="NCU_REPORT", default=None,
                    help="write --workload's per-launch DRAM bytes from this ncu report into "
                         "profiles/dram_traffic.json (no GPU needed) and exit")
    ap.add_argument("--traffic-scale", type=float, default=1.0,
                    help="with --record-traffic: multiply the captured bytes (a capture at a smaller batch)")
    args = ap.parse_args(argv)
    if args.record_traffic:
        return record_traffic(args.record_traffic, args.workload, args.traffic_scale,
                              args.batch if args.traffic_scale != 1.0 else None)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    env_world = os.environ.get("WORLD_SIZE")
    if env_world is None and args.gpus > 1:
        return relaunch_under_torchrun(args.gpus, sys.argv[1:] if argv is None else argv)
    if env_world is not None and int(env_world) != args.gpus:
        raise SystemExit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={env_world}; launch one rank per GPU")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
