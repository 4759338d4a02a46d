#!/usr/bin/env python3
"""Benchmark of the exact per-row top-K path on GB300.

Workload (one step): the prefill top-K of the sparse-attention indexer --
4096 query rows of fp32 N(0,1) logits at each of 8192, 51200 and 102400
columns, K = 512, causal row ends row_end[i] = cols - 4096 + i + 1, output
into a preallocated strided int32 [4096, 640] buffer.  That is 12288 rows
per step and every valid column read once from HBM (2.55 GB per step; the
inputs are far larger than L2, so consecutive steps start cold).

Prints one JSON line: rows/s over the timed steps (device-timed with CUDA
events, inputs resident), the end-to-end figure through the same API with
host buffers, the roofline of the dominant kernel against the measured HBM
copy bandwidth, the CPU oracle timed on a bounded sample, clocks sampled
during the timed region, and per-stage figures of the other workloads
(rank-major pairs merge, one-round decode merge, adversarial bf16 top-K).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With --impl reference the CPU oracle itself is the arm being timed.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_attention_indexer_radix_gb300 import inputs  # noqa: E402

ROWS, K, LD_OUT = inputs.PREFILL_ROWS, inputs.PREFILL_K, inputs.PREFILL_LD_OUT
WIDTHS = inputs.PREFILL_COLS
METRIC = "rows/s and achieved HBM GB/s (% of GB300 peak) for exact per-row top-K"
WORKLOAD = ("prefill top-K: 4096 query rows x {8192, 51200, 102400} cols fp32 ~N(0,1), "
            "K=512, causal row_end[i]=cols-4096+i+1, strided int32 output [4096, 640]")
CPU_SAMPLE_STRIDE = 8  # every 8th row of each width: 512 rows per width
# The prefill page's own times for this workload (vLLM PR #57206, Synthetic
# controls): the native radix selector top_k_per_row_prefill on one GB200,
# per width in microseconds.  Another machine's figure: context for
# vs_baseline, not the target.
PAGES_NATIVE_US = {8192: 80.9, 51200: 321.4, 102400: 688.3}


def algorithmic_bytes(cols: int, rows: int = ROWS, k: int = K, elt: int = 4) -> int:
    """Valid prefixes read once plus the ids written once."""
    ends = np.clip(np.arange(rows) + (cols - rows + 1), 0, cols)
    return int(ends.sum()) * elt + rows * k * 4


def pages_rows_per_s(widths=WIDTHS, rows=ROWS):
    """rows/s of one step at the pages' per-width times, or None when the
    step is not the pages' workload (a profiling subset)."""
    if rows != ROWS or tuple(widths) != tuple(WIDTHS):
        return None
    return rows * len(widths) / (sum(PAGES_NATIVE_US[c] for c in widths) * 1e-6)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "sparse_attention_indexer_radix_gb300", "csrc",
                                           "*"))):
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_tag: str):
    """dram bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_tag)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# clocks-event reason bits of NVML's nvmlDeviceGetCurrentClocksEventReasons
NVML_REASON_BITS = {"gpu_idle": 0x1, "sw_power_cap": 0x4, "hw_slowdown": 0x8,
                    "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40}
NVML_CLOCK_SM = 1


def device_uuid(index: int):
    """NVML-style UUID ("GPU-...") of CUDA device `index`, or None: CUDA and
    NVML may number the GPUs differently, the UUID names the same one."""
    try:
        u = str(torch.cuda.get_device_properties(index).uuid)
    except (AttributeError, RuntimeError):
        return None
    return u if u.startswith("GPU-") else "GPU-" + u


class ClockSampler:
    """SM clock and throttle reasons of the GPU while the timed region runs.

    NVML (through ctypes) is polled about every millisecond from a thread,
    so even a timed region of a few milliseconds gets samples; samples that
    NVML flags as idle are left out.  Without NVML, nvidia-smi polls every
    100 ms instead."""

    SMI_FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.uuid = device_uuid(index)
        self.proc = None
        self.thread = None
        self.samples = []  # (sm MHz, reason bits) from NVML
        self.lines = []    # nvidia-smi CSV lines
        self.max_mhz = None

    def _nvml(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if self.uuid is None or lib.nvmlInit_v2() != 0:
                return None
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) != 0:
                return None
            try:
                reasons = lib.nvmlDeviceGetCurrentClocksEventReasons
            except AttributeError:
                reasons = lib.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            return lib, h, reasons
        except (OSError, AttributeError):
            return None

    def _poll(self, lib, h, reasons):
        import ctypes
        clk, bits = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            if (lib.nvmlDeviceGetClockInfo(h, NVML_CLOCK_SM, ctypes.byref(clk)) == 0 and
                    reasons(h, ctypes.byref(bits)) == 0):
                self.samples.append((float(clk.value), int(bits.value)))
            time.sleep(0.001)

    def __enter__(self):
        import threading
        nv = self._nvml()
        if nv is not None:
            self.stop = threading.Event()
            self.thread = threading.Thread(target=self._poll, args=nv, daemon=True)
            self.thread.start()
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.uuid or str(self.index),
                 f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.thread is not None:
            self.stop.set()
            self.thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        if self.thread is not None:
            busy = [(c, b) for c, b in self.samples if not b & NVML_REASON_BITS["gpu_idle"]]
            for c, b in busy:
                sm.append(c)
                reasons.update(nm for nm in names if b & NVML_REASON_BITS[nm])
            if self.max_mhz is not None:
                mx.append(self.max_mhz)
            source = "nvml"
        else:
            for ln in self.lines:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) < 7:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx.append(float(parts[1]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[3:7]):
                    if v.lower() == "active":
                        reasons.add(nm)
            source = "nvidia-smi"
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": max(mx) if mx else None,
                    "reasons": ["unsampled"], "samples": 0, "source": source}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "source": source}


# --------------------------------------------------------------- workload --

def make_prefill(device, widths=WIDTHS, rows=ROWS):
    data = []
    for cols in widths:
        i = WIDTHS.index(cols)
        x, ends = inputs.prefill(rows=ROWS, cols=cols, seed=1236 + i, device=device)
        if rows != ROWS:  # a smaller case for profiler captures: the last rows
            x, ends = x[-rows:].contiguous(), ends[-rows:].contiguous()
        out = torch.full((rows, LD_OUT), -7, dtype=torch.int32, device=device)
        data.append((cols, x, ends, out))
    return data


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    """The largest of the ranks' values (the job's time is its slowest
    rank's); on the process group's own device (CUDA for NCCL, CPU for
    gloo)."""
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_rows_per_s(rows_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput of `world` replicas, each processing
    rows_per_step rows per step: every rank's rows over the slowest rank's
    time (weak scaling)."""
    return rows_per_step * steps * world / (max_ms * 1e-3)


# ------------------------------------------------------------- CPU oracle --

def cpu_sample_rows():
    return np.arange(0, ROWS, CPU_SAMPLE_STRIDE)


def time_oracle_prefill(host_data, nthreads=0):
    """One bounded sample of the workload through the oracle (the sampled
    rows of each width).  Returns (rows, seconds)."""
    import oracle
    rows = 0
    t0 = time.perf_counter()
    for cols, x, ends in host_data:
        oracle.topk_rows(x, K, row_ends=ends, nthreads=nthreads)
        rows += x.shape[0]
    return rows, time.perf_counter() - t0


def host_prefill_sample(device_data=None):
    """The sampled rows of each width as host arrays: copied from the device
    inputs when given (the very rows the GPU arm processes), else generated
    with the same seeds on the best available device."""
    sel = cpu_sample_rows()
    out = []
    if device_data is None:
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        device_data = [(cols,) + inputs.prefill(rows=ROWS, cols=cols, seed=1236 + i, device=dev)
                       for i, cols in enumerate(WIDTHS)]
    for item in device_data:
        cols, x, ends = item[0], item[1], item[2]
        idx = torch.as_tensor(sel, device=x.device)
        out.append((cols, np.ascontiguousarray(x.index_select(0, idx).cpu().numpy()),
                    np.ascontiguousarray(ends.index_select(0, idx).cpu().numpy())))
    return out, sel


# ---------------------------------------------------------------- stages --

def timed_calls(fn, reps, flush):
    """Median device time (ms) of fn() over reps, L2 flushed before each."""
    times = []
    for _ in range(reps):
        flush.fill_(1)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        torch.cuda.synchronize()
        times.append(s.elapsed_time(e))
    return statistics.median(times)


STAGES = ("pairs", "decode", "adversarial", "robust")


def stage_figures(dev, flush, peak, which=STAGES):
    import sparse_attention_indexer_radix_gb300 as satk
    st = {}
    if "pairs" in which:
        st.update(_stage_pairs(dev, flush, peak, satk))
    if "decode" in which:
        st.update(_stage_decode(dev, flush, peak, satk))
    if "adversarial" in which:
        st.update(_stage_adversarial(dev, flush, peak, satk))
    if "robust" in which:
        st.update(_stage_robust(dev, flush, peak, satk))
    return st


def _stage_pairs(dev, flush, peak, satk):
    st = {}
    # rank-major pairs merge: W=8, 6710 rows, top-2048 of 8 x 2048 candidates
    W, R, k = 8, 6710, 2048
    cand = inputs.pairs_merge(W=W, rows=R, k=k, local=16384, seed=1236, device=dev)
    ids = torch.empty((R, k), dtype=torch.int32, device=dev)
    fn = lambda: satk.dcp_merge_select(cand, k, packed=False, ids_out=ids)  # noqa: E731
    for _ in range(3):
        fn()
    ms = timed_calls(fn, 10, flush)
    nbytes = cand.numel() * 4 + ids.numel() * 4
    st["pairs_merge_W8_R6710_K2048"] = {
        "us": ms * 1e3, "rows_per_s": R / (ms * 1e-3), "gbs": nbytes / (ms * 1e-3) / 1e9,
        "frac": nbytes / (ms * 1e-3) / 1e9 / peak, "alg_bytes": nbytes}
    return st


def _stage_decode(dev, flush, peak, satk):
    st = {}
    # one-round decode merge: W=8, 128 rows, S=65536 bf16, N=384, K=2048
    W, T, S, n, k = 8, 128, 65536, 384, 2048
    lg, _, _ = inputs.decode_merge(W=W, rows=T, S=S, n=n, k=k, seed=1237, device=dev)
    flat = lg.view(W * T, S)
    local = torch.empty((W * T, n), dtype=torch.int32, device=dev)
    packed = torch.empty((W, T, n + n // 32), dtype=torch.int32, device=dev)
    sat = torch.zeros(T, dtype=torch.int32, device=dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    recv = torch.zeros(satk.rescue_recv_words(T, n, k), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    # rank 0's physical KV rows: 64-token blocks, a permuted block table
    B = 64
    width = (S + B - 1) // B
    g = torch.Generator(device=dev).manual_seed(1238)
    table = torch.randperm(T * width, generator=g, device=dev).to(torch.int32).view(T, width)
    req = torch.randperm(T, generator=g, device=dev).to(torch.int32)
    rows_out = torch.empty((T, k), dtype=torch.int32, device=dev)
    valid = torch.empty(T, dtype=torch.int32, device=dev)
    # the step: the local top-N written straight as B' rows, the round-1
    # merge with its saturation words, the rescue, this rank's KV rows
    parts = {
        "topN_pack": lambda: satk.dcp_topk_pack(flat, n, out=packed.view(W * T, -1)),
        "merge_select": lambda: satk.dcp_merge_select(packed, k, packed=True, ids_out=ids,
                                                      sat_word=sat, status=status),
        "rescue": lambda: satk.dcp_rescue_select(packed, lg, sat, ids, k, recv=recv,
                                                 status=status),
        "emit_rows": lambda: satk.dcp_emit_rows(ids, W, 0, req, table, B, B, rows_out=rows_out,
                                                valid_out=valid),
    }
    dec = {}
    for name, f in parts.items():
        for _ in range(3):
            f()
        dec[name + "_us"] = timed_calls(f, 10, flush) * 1e3
    dec["total_us"] = sum(dec.values())
    # the same step replayed as one CUDA graph (launches back to back, L2
    # flushed before each replay), as the pages time their kernels
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for f in parts.values():
            f()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            for f in parts.values():
                f()
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        graph.replay()
    dec["graph_us"] = timed_calls(graph.replay, 10, flush) * 1e3
    # the two calls the fused one replaces, for reference (not in the totals)
    ref = {"local_topN": lambda: satk.topk_rows(flat, n, out=local),
           "pack": lambda: satk.dcp_pack(flat, local, out=packed.view(W * T, -1))}
    for name, f in ref.items():
        for _ in range(3):
            f()
        dec["unfused_" + name + "_us"] = timed_calls(f, 10, flush) * 1e3
    nb = flat.numel() * 2 + packed.numel() * 4
    dec["topN_pack_gbs"] = nb / (dec["topN_pack_us"] * 1e-6) / 1e9
    dec["topN_pack_frac"] = dec["topN_pack_gbs"] / peak
    dec["saturated_rows"] = int(((sat >> 16) != 0).sum().item())
    st["decode_merge_W8_T128_S65536_N384_K2048"] = dec
    return st


def _stage_adversarial(dev, flush, peak, satk):
    st = {}
    # adversarial bf16 top-K: 256 x 131072, 64 levels, K=2048
    x, ends, _ = inputs.adversarial(seed=1239, device=dev)
    out = torch.empty((256, 2048 + 64), dtype=torch.int32, device=dev)
    fn = lambda: satk.topk_rows(x, 2048, row_ends=ends, out=out)  # noqa: E731
    for _ in range(3):
        fn()
    ms = timed_calls(fn, 10, flush)
    nb = int(ends.clamp(min=0).sum().item()) * 2 + 256 * 2048 * 4
    st["adversarial_bf16_256x131072_K2048"] = {
        "us": ms * 1e3, "rows_per_s": 256 / (ms * 1e-3), "gbs": nb / (ms * 1e-3) / 1e9,
        "frac": nb / (ms * 1e-3) / 1e9 / peak}
    return st


# The prefill page's other shapes (the query rows x logits columns of its
# captured chunks, here on synthetic N(0,1) logits) and its distribution
# ablation at 8192 x 8192: fp32, causal row ends, K = 512.
ROBUST_SHAPES = ((8192, 4096), (8192, 8192), (2048, 25600), (2048, 51200), (1310, 102400))
ROBUST_MODES = ("plus100", "times1e-8")


def _stage_robust(dev, flush, peak, satk):
    st = {}

    def one(name, x, ends):
        rows = x.shape[0]
        out = torch.empty((rows, K), dtype=torch.int32, device=dev)
        fn = lambda: satk.topk_rows(x, K, row_ends=ends, out=out)  # noqa: E731
        for _ in range(3):
            fn()
        ms = timed_calls(fn, 10, flush)
        nb = int(ends.clamp(min=0).sum().item()) * 4 + rows * K * 4
        st[name] = {"us": ms * 1e3, "rows_per_s": rows / (ms * 1e-3),
                    "gbs": nb / (ms * 1e-3) / 1e9, "frac": nb / (ms * 1e-3) / 1e9 / peak}

    for i, (rows, cols) in enumerate(ROBUST_SHAPES):
        x, ends = inputs.prefill(rows=rows, cols=cols, seed=1250 + i, device=dev)
        one(f"shape_{rows}x{cols}_f32_K512", x, ends)
        del x
    for mode in ROBUST_MODES:
        x, ends = inputs.prefill_shifted(8192, 8192, mode, device=dev)
        one(f"dist_{mode}_8192x8192_f32_K512", x, ends)
        del x
    # the score-sorted output option on the prefill 8192-column width
    x, ends = inputs.prefill(rows=ROWS, cols=8192, seed=1236, device=dev)
    out = torch.empty((ROWS, K), dtype=torch.int32, device=dev)
    fn = lambda: satk.topk_rows(x, K, row_ends=ends, out=out, sorted=True)  # noqa: E731
    for _ in range(3):
        fn()
    ms = timed_calls(fn, 10, flush)
    nb = int(ends.clamp(min=0).sum().item()) * 4 + ROWS * K * 4
    st["sorted_4096x8192_f32_K512"] = {"us": ms * 1e3, "rows_per_s": ROWS / (ms * 1e-3),
                                       "gbs": nb / (ms * 1e-3) / 1e9,
                                       "frac": nb / (ms * 1e-3) / 1e9 / peak}
    del x
    # decode-shaped few long rows (the DCP kernels page: the cluster variant
    # of its selector for <= 6 rows at >= 512K columns): bf16, K = 384
    x, ends = inputs.prefill(rows=4, cols=524288, seed=1260, device=dev, causal=False,
                             dtype=torch.bfloat16)
    out = torch.empty((4, 384), dtype=torch.int32, device=dev)
    fn = lambda: satk.topk_rows(x, 384, row_ends=ends, out=out)  # noqa: E731
    for _ in range(3):
        fn()
    ms = timed_calls(fn, 10, flush)
    nb = 4 * 524288 * 2 + 4 * 384 * 4
    st["few_rows_4x524288_bf16_K384"] = {"us": ms * 1e3, "gbs": nb / (ms * 1e-3) / 1e9,
                                         "frac": nb / (ms * 1e-3) / 1e9 / peak}
    return st


# ------------------------------------------------------------------- arms --

def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    host, sel = host_prefill_sample()
    cores = oracle.default_threads()
    for _ in range(args.warmup):
        time_oracle_prefill(host)
    times = []
    rows = 0
    for _ in range(args.steps):
        r, dt = time_oracle_prefill(host)
        rows = r
        times.append(dt)
    total = sum(times)
    value = rows * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": f"every {CPU_SAMPLE_STRIDE}th row of each width"},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": f"{len(sel)} rows of each of the 3 widths per step "
                                   f"(every {CPU_SAMPLE_STRIDE}th row)"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args):
    import sparse_attention_indexer_radix_gb300 as satk
    from sparse_attention_indexer_radix_gb300 import build as satk_build
    world, rank, local = dist_setup(args.gpus)
    if rank == 0:
        satk_build.build()
    barrier(world)
    dev = torch.device("cuda", torch.cuda.current_device())
    peak, peak_kind = measured_peaks()
    widths = WIDTHS if not args.only else tuple(int(c) for c in args.only.split(","))
    rows = args.rows
    data = make_prefill(dev, widths, rows)
    flush = inputs.flush_buffer(dev)
    stream = torch.cuda.current_stream(dev)

    def step(events=None):
        for j, (cols, x, ends, out) in enumerate(data):
            if events is not None:
                events[j][0].record(stream)
            satk.topk_rows(x, K, row_ends=ends, out=out)
            if events is not None:
                events[j][1].record(stream)

    for _ in range(max(args.warmup, 3) if args.warmup >= 0 else 3):
        step()
    torch.cuda.synchronize()

    # ---- device-timed region: inputs resident, K steps
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in widths] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for s in range(args.steps):
            step(ev[s])
        t1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    total_ms = max_over_ranks(t0.elapsed_time(t1), world)
    per_width_ms = [statistics.mean(ev[s][j][0].elapsed_time(ev[s][j][1])
                                    for s in range(args.steps)) for j in range(len(widths))]
    rows_step = rows * len(widths)
    value = replica_rows_per_s(rows_step, args.steps, world, total_ms)

    # ---- end to end: pinned host inputs -> device -> ids -> host, every step
    host_in = [(x.cpu().pin_memory(), e.cpu().pin_memory()) for (_, x, e, _) in data]
    host_out = [torch.empty_like(o, device="cpu").pin_memory() for (_, _, _, o) in data]
    h2d = sum(x.numel() * x.element_size() + e.numel() * 4 for x, e in host_in)
    d2h = sum(o.numel() * 4 for o in host_out)

    def e2e_step():
        for j, (cols, x, ends, out) in enumerate(data):
            hx, he = host_in[j]
            x.copy_(hx, non_blocking=True)
            ends.copy_(he, non_blocking=True)
            satk.topk_rows(x, K, row_ends=ends, out=out)
            host_out[j].copy_(out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e_steps = max(1, min(args.steps, 5))
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(e_steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b), world)
    e2e_value = replica_rows_per_s(rows_step, e_steps, world, e2e_ms)

    # ---- roofline of the dominant kernel (largest share of the step)
    j = int(np.argmax(per_width_ms))
    cols = widths[j]
    alg = algorithmic_bytes(cols, rows)
    achieved = alg / (per_width_ms[j] * 1e-3) / 1e9
    kernel_tag = f"topk_rows_kernel_f32_{cols}"
    traffic = recorded_traffic(kernel_tag)
    per_width = {}
    for jj, c in enumerate(widths):
        ab = algorithmic_bytes(c, rows)
        gbs = ab / (per_width_ms[jj] * 1e-3) / 1e9
        per_width[str(c)] = {"us": per_width_ms[jj] * 1e3,
                             "rows_per_s": rows / (per_width_ms[jj] * 1e-3),
                             "gbs": gbs, "frac": gbs / peak, "alg_bytes": ab}

    pages = pages_rows_per_s(widths, rows)
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None if pages is None else value / pages,
        "baseline": None if pages is None else {
            "value": pages, "unit": "rows/s",
            "source": "prefill page (vLLM PR #57206, Synthetic controls): native "
                      "top_k_per_row_prefill on one GB200, 80.9 + 321.4 + 688.3 us per step"},
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "rows_per_step": rows_step, "k": K,
                   "l2": "inputs (2.55 GB per step) larger than L2; flush buffer before stages",
                   "parallelism": f"replicas x{world} (rows independent, no collective)"},
        "gpu_launches": len(widths) * args.steps,
        "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e_steps},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": kernel_tag, "peak_kind": peak_kind,
                     "alg_bytes_per_launch": alg},
        "widths": per_width,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_stages:
        line["stages"] = stage_figures(dev, flush, peak)
    if args.only or rows != ROWS:
        line["config"]["workload"] = f"profiling subset: widths {list(widths)}, last {rows} rows"
    if rank == 0 and not args.no_cpu:
        import oracle
        oracle.build()
        host, sel = host_prefill_sample(data)
        rows, dt = time_oracle_prefill(host)
        line["cpu_baseline"] = {"value": rows / dt, "unit": "rows/s",
                                "cores": oracle.default_threads(), "kind": "oracle",
                                "sample": f"{len(sel)} rows of each of the 3 widths "
                                          f"(every {CPU_SAMPLE_STRIDE}th row), one pass"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="satk", choices=["satk", "reference"])
    ap.add_argument("--no-stages", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--only", default="", help="profiling aid: comma-separated widths")
    ap.add_argument("--rows", type=int, default=ROWS, help="profiling aid: rows per width")
    ap.add_argument("--stage-only", default="",
                    help="profiling aid: run only these stages (comma-separated: "
                         + ",".join(STAGES) + ") and print their figures")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.stage_only:
        from sparse_attention_indexer_radix_gb300 import build as satk_build
        satk_build.build()
        dev = torch.device("cuda", 0)
        peak, _ = measured_peaks()
        which = tuple(args.stage_only.split(","))
        print(json.dumps({"stages": stage_figures(dev, inputs.flush_buffer(dev), peak, which)}))
        return 0
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
