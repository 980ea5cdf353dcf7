#!/usr/bin/env python3
"""Benchmark of the paged KV-cache hot path on GB300.

Default workload: single-query decode, B=4, KV lengths {7168,7168,4171,513},
Hq=8, Hkv=2, Dh=128, page 16, interleaved pool of 2048 blocks with shuffled
pages.  One step = the whole hot path for one batch: the cache write of the
4 new tokens followed by paged attention, issued as one library call
(pa_reshape_and_paged_attention; the same step as the two separate calls is
timed beside it).  Metric: decode KV-read GB/s = bytes of K and V the
step must read (sum_b L_b * Hkv * Dh * 2 B * 2) / step time.

Timing: K steps are captured in CUDA graphs and replayed back to back on one
stream, bracketed by a barrier + synchronize and CUDA events.  Steps rotate
over R replicas of the workload (separate device copies) so a step's K/V was
last touched R-1 steps earlier; R*19.5 MB exceeds the 129 MB L2, so every
step reads its cache from HBM.

Also reported: the attention kernel's roofline (algorithmic bytes per launch
/ mean launch time from a graph of attention launches alone), long-prefill
TFLOP/s as a secondary figure, an end-to-end figure through the public API
with host buffers, SM clocks sampled during the timed region, and the CPU
oracle's throughput on a bounded sample.

`--impl reference` times the CPU oracle on the same workload and metric.
Multi-GPU (torchrun): replicas only -- each rank runs the same workload on
its own GPU, no data exchange; value = all ranks' bytes / max rank time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_kv_cache_178_gb300 import workloads as wl  # noqa: E402

METRIC = "paged-attn decode KV GB/s & prefill TFLOP/s, % of GB300 roofline"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "attn_kernel_decode_b4_kv7168.md")
KERNEL_SOURCES = [os.path.join(ROOT, "paged_kv_cache_178_gb300", "csrc", f)
                  for f in ("pa_decode.cu", "pa_split.cuh", "pa_attn_common.cuh", "pa_ptx.cuh")]


def kernel_source_hash() -> str:
    """First 16 hex digits of sha256 over the decode kernel's sources."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ ranks --

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend)


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """Largest value over ranks (the timing rule: slowest rank counts)."""
    if ws <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(units_per_rank: float, elapsed_s: float, ws: int, device=None) -> float:
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    t = max_over_ranks(elapsed_s, ws, device)
    return units_per_rank * ws / t


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """Samples SM clock and clock-event reasons during the timed region: an
    `nvidia-smi -lms` subprocess plus in-process NVML polling (read only)."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int):
        self.dev = device_index
        self.samples = []        # (sm_mhz, reasons bitmask)
        self.smi_lines = []
        self.sm_max = None
        self._stop = threading.Event()
        self._nvml = None
        self._handle = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() == 0:
                h = ctypes.c_void_p()
                uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
                if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0:
                    self._nvml, self._handle = nv, h
                    mx = ctypes.c_uint()
                    if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                        self.sm_max = float(mx.value)
        except Exception:
            self._nvml = None

    def _poll(self):
        nv, h = self._nvml, self._handle
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and fn(h, ctypes.byref(rs)) == 0:
                self.samples.append((float(clk.value), int(rs.value)))
            time.sleep(0.002)

    def __enter__(self):
        self._smi = None
        try:
            self._smi = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=clocks.sm,clocks.max.sm,"
                 "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self._smi = None
        self._thr = None
        if self._nvml is not None:
            self._thr = threading.Thread(target=self._poll, daemon=True)
            self._thr.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._thr is not None:
            self._thr.join()
        if self._smi is not None:
            self._smi.terminate()
            try:
                out, _ = self._smi.communicate(timeout=5)
                self.smi_lines = [ln for ln in out.splitlines() if ln.strip()]
            except Exception:
                pass
        return False

    def summary(self):
        clocks, mask = [], 0
        for ln in self.smi_lines:
            parts = [p.strip() for p in ln.split(",")]
            try:
                clocks.append(float(parts[0]))
                if self.sm_max is None:
                    self.sm_max = float(parts[1])
                mask |= int(parts[2], 16)
            except (ValueError, IndexError):
                pass
        src = "nvidia-smi"
        if self.samples:
            clocks = [c for c, _ in self.samples]
            for _, r in self.samples:
                mask |= r
            src = "nvml+nvidia-smi" if self.smi_lines else "nvml"
        reasons = [name for bit, name in self.REASONS.items() if mask & bit]
        return {"sm_mhz": statistics.median(clocks) if clocks else None, "sm_max_mhz": self.sm_max,
                "reasons": reasons, "samples": len(clocks), "source": src}


# ------------------------------------------------------- workload helpers --

def decode_bytes(w: wl.Workload) -> int:
    """K and V bytes a decode step must read (valid tokens only)."""
    return int(w.seq_lens.sum()) * w.num_kv_heads * w.head_dim * 2 * 2


def attn_io_bytes(w: wl.Workload) -> int:
    """Algorithmic bytes of one attention launch: K/V of valid tokens, q, out
    (BF16) and lse (fp32)."""
    tq = w.num_q_tokens
    return decode_bytes(w) + 2 * tq * w.num_q_heads * w.head_dim * 2 + tq * w.num_q_heads * 4


def causal_flops(w: wl.Workload) -> float:
    """4*Dh per (query row, head, attended key): QK^T and PV, causal keys only."""
    tot = 0
    for b in range(w.num_seqs):
        L = int(w.seq_lens[b])
        qn = int(w.query_start_loc[b + 1] - w.query_start_loc[b])
        # rows attend to L-qn+1 .. L keys
        tot += qn * (L - qn) + qn * (qn + 1) // 2
    return 4.0 * w.head_dim * w.num_q_heads * tot


def last_token_rows(w: wl.Workload):
    """Index (into w.key/w.value/slot_mapping) of each request's newest token."""
    rows, at = [], 0
    for L in w.seq_lens.tolist():
        rows.append(at + L - 1)
        at += L
    return rows


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def profile_traffic():
    """dram bytes per attention launch from the committed ncu summary, if it
    was taken on the current kernel source; else None."""
    try:
        text = open(PROFILE_SUMMARY).read()
        src = kernel_source_hash()
        m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
        m_bytes = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
        if m_hash and m_bytes and m_hash.group(1) == src:
            return int(m_bytes.group(1))
    except OSError:
        pass
    return None


# -------------------------------------------------------------- our arm ----

class GraphedSteps:
    """Capture `fn(i)` for i in range(n) into CUDA graphs of <= chunk steps and
    replay them so that exactly `total` steps run."""

    def __init__(self, fn, period: int, stream, chunk: int = 1000):
        self.fn, self.period, self.stream = fn, period, stream
        self.chunk = max(period, (chunk // period) * period)
        self.graphs = {}

    def _graph(self, n: int):
        if n not in self.graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                for i in range(n):
                    self.fn(i)
            self.graphs[n] = g
        return self.graphs[n]

    def prepare(self, total: int):
        """Capture every graph run(total) will replay (outside any timing)."""
        full, rem = divmod(total, self.chunk)
        if full:
            self._graph(self.chunk)
        if rem:
            self._graph(rem)

    def run(self, total: int):
        full, rem = divmod(total, self.chunk)
        with torch.cuda.stream(self.stream):
            for _ in range(full):
                self._graph(self.chunk).replay()
            if rem:
                self._graph(rem).replay()


def time_graphed(gs: GraphedSteps, steps: int, stream, ws: int) -> float:
    """Seconds for exactly `steps` steps (events on the work stream)."""
    gs.prepare(steps)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(ws)
    start.record(stream)
    gs.run(steps)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    return start.elapsed_time(end) / 1e3


def run_ours(args, ws, rank, local):
    from paged_kv_cache_178_gb300 import pagedattn
    from paged_kv_cache_178_gb300.device import DeviceWorkload

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(ws, "nccl")
    pagedattn.init()
    stream = torch.cuda.Stream(device=dev)
    peaks, peak_src = load_peaks()
    if args.workload in ("prefill", "wide"):
        pf = measure_prefill(args, dev, stream, ws, peaks, peak_src, launches=args.steps,
                             wide=args.workload == "wide")
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": pf["tflops"], "unit": "TFLOP/s",
                              "n_gpus": ws, "steps": args.steps, "warmup": max(args.warmup, 3),
                              "ms_per_step": pf["us_per_launch"] / 1e3, "higher_is_better": True,
                              "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                              "data": "synthetic", "config": {"workload": pf["workload"],
                                                               "schedule": pf["schedule"]},
                              "gpu_launches": args.steps,
                              "roofline": {"bound": "tensor", "achieved": pf["tflops"],
                                           "peak": pf["peak"], "unit": "TFLOP/s", "frac": pf["frac"],
                                           "traffic": None, "peak_source": pf["peak_source"]}}),
                  flush=True)
        return
    if args.workload == "decode_scaled":
        ds = measure_decode_scaled(args, dev, stream, ws, peaks, peak_src, launches=args.steps)
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": ds["gbs"], "unit": "GB/s",
                              "n_gpus": ws, "steps": args.steps, "warmup": max(args.warmup, 3),
                              "ms_per_step": ds["us_per_launch"] / 1e3, "higher_is_better": True,
                              "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                              "data": "synthetic", "config": {"workload": ds["workload"],
                                                               "schedule": ds["schedule"]},
                              "gpu_launches": args.steps,
                              "roofline": {"bound": "hbm", "achieved": ds["gbs"], "peak": ds["peak"],
                                           "unit": "GB/s", "frac": ds["frac"], "traffic": None,
                                           "peak_source": ds["peak_source"]}}),
                  flush=True)
        return
    if args.workload == "gather":
        ga = measure_gather(args, dev, stream, ws, peaks, peak_src, launches=args.steps)
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": ga["gbs"], "unit": "GB/s",
                              "n_gpus": ws, "steps": args.steps, "warmup": max(args.warmup, 3),
                              "ms_per_step": ga["us_per_launch"] / 1e3, "higher_is_better": True,
                              "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                              "data": "synthetic", "config": {"workload": ga["workload"]},
                              "gpu_launches": args.steps,
                              "roofline": {"bound": "hbm", "achieved": ga["gbs"], "peak": ga["peak"],
                                           "unit": "GB/s", "frac": ga["frac"], "traffic": None,
                                           "peak_source": ga["peak_source"]}}),
                  flush=True)
        return

    w = wl.decode()
    R = args.replicas
    reps = [DeviceWorkload(w, device=str(dev), fill_bits=None) for _ in range(R)]
    last = last_token_rows(w)
    step_in = []
    for dw in reps:
        dw.write_cache()                       # populate all L tokens once
        idx = torch.tensor(last, device=dev)
        step_in.append((dw.key.index_select(0, idx).contiguous(),
                        dw.value.index_select(0, idx).contiguous(),
                        dw.slot_mapping.index_select(0, idx).contiguous()))
    outs = [torch.empty_like(dw.q) for dw in reps]
    lses = [torch.empty(dw.q.shape[:2], dtype=torch.float32, device=dev) for dw in reps]
    torch.cuda.synchronize()
    st, idx = pagedattn.check_errors()
    assert st == pagedattn.PA_OK, (st, idx)

    def step(i):
        r = i % R
        k, v, s = step_in[r]
        reps[r].write_and_attend(key=k, value=v, slot_mapping=s, out=outs[r], lse=lses[r])

    def step_two_calls(i):
        r = i % R
        dw = reps[r]
        k, v, s = step_in[r]
        pagedattn.reshape_and_cache(k, v, dw.k_cache, dw.v_cache, s)
        dw.attention(out=outs[r], lse=lses[r])

    def attn_only(i):
        r = i % R
        reps[r].attention(out=outs[r], lse=lses[r])

    def attn_only_tile64(i):
        r = i % R
        reps[r].attention(out=outs[r], lse=lses[r], kv_tile=64)

    with torch.cuda.stream(stream):
        step(0)                                 # eager warm call (attributes, maps)
    torch.cuda.synchronize()
    info = pagedattn.last_launch_info()
    full = GraphedSteps(step, R, stream)
    full.run(max(args.warmup, 3))               # untimed warm-up steps
    torch.cuda.synchronize()
    # The timed region (exactly K steps) is repeated: at least `min_repeats`
    # times and until `min_timed_s` of timed work has run, so a short K still
    # gives a median over many regions and enough clock samples.  Each
    # repeat's time is the max over ranks; the reported value is the median.
    full.prepare(args.steps)
    reps_s = []
    clk = ClockSampler(local)
    with clk:
        while len(reps_s) < args.min_repeats or (sum(reps_s) < args.min_timed_s and len(reps_s) < 2000):
            reps_s.append(max_over_ranks(time_graphed(full, args.steps, stream, ws), ws, dev))
    clocks = clk.summary()
    st, idx = pagedattn.check_errors(stream)
    assert st == pagedattn.PA_OK, (st, idx)
    elapsed = statistics.median(reps_s)

    kv_bytes = decode_bytes(w)
    value = aggregate_value(kv_bytes * args.steps / 1e9, elapsed, ws, dev)
    ms_per_step = elapsed / args.steps * 1e3

    # The same step as two library calls (the attention waits at entry).
    two = GraphedSteps(step_two_calls, R, stream)
    two.run(max(args.warmup, 3))
    n_two = max(args.steps, 200)
    t_two = time_graphed(two, n_two, stream, ws) / n_two

    # Roofline of the dominant kernel: attention launches alone, same replicas.
    attn = GraphedSteps(attn_only, R, stream)
    attn.run(max(args.warmup, 3))
    n_attn = max(args.steps, 200)
    t_attn = time_graphed(attn, n_attn, stream, ws) / n_attn
    # The same launches in the second canon (64-key tiles).
    attn64 = GraphedSteps(attn_only_tile64, R, stream)
    attn64.run(max(args.warmup, 3))
    t_attn64 = time_graphed(attn64, n_attn, stream, ws) / n_attn
    attn_bytes = attn_io_bytes(w)
    achieved = attn_bytes / t_attn / 1e9

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": round(ms_per_step, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "decode B=4 Q=1 KV={7168,7168,4171,513} Hq=8 Hkv=2 Dh=128 page16 "
                               "interleaved pool 2048 blocks, shuffled pages",
                   "step": "pa_reshape_and_paged_attention (4 new tokens)",
                   "us_per_step_as_two_calls": round(t_two * 1e6, 3),
                   "kv_bytes_per_step": kv_bytes,
                   "l2": f"{R} rotating device replicas, {R * kv_bytes / 1e6:.0f} MB of K/V > 129 MB L2",
                   "launch": "CUDA graphs of up to 1000 steps replayed back to back",
                   "repeats": {"n": len(reps_s), "how": "the K-step region timed n times; value and "
                               "ms_per_step from the median region",
                               "ms_per_step_min": round(min(reps_s) / args.steps * 1e3, 6),
                               "ms_per_step_median": round(ms_per_step, 6),
                               "ms_per_step_max": round(max(reps_s) / args.steps * 1e3, 6)},
                   "schedule": info, "parallelism": f"replicas x{ws}"},
        "gpu_launches": 2 * args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": profile_traffic(),
                     "kernel": "dec_kernel<4> (split-KV decode, keys on the tensor-memory lanes)",
                     "bytes_per_launch": attn_bytes, "us_per_launch": round(t_attn * 1e6, 3),
                     "peak_source": f"{peak_src} hbm_gbs"},
        "clocks": clocks,
        "decode_tile64": {"workload": "the same attention launches with 64-key KV tiles (second canon)",
                          "gbs": round(attn_bytes / t_attn64 / 1e9, 1), "us_per_launch": round(t_attn64 * 1e6, 3),
                          "frac": round(attn_bytes / t_attn64 / 1e9 / peaks["hbm_gbs"], 4),
                          "peak_source": f"{peak_src} hbm_gbs"},
    }
    if not args.no_secondary:
        line["decode_scaled"] = measure_decode_scaled(args, dev, stream, ws, peaks, peak_src)
        line["gather"] = measure_gather(args, dev, stream, ws, peaks, peak_src)
        line["prefill"] = measure_prefill(args, dev, stream, ws, peaks, peak_src)
        line["prefill_tile64"] = measure_prefill(args, dev, stream, ws, peaks, peak_src, kv_tile=64)
        line["prefill_wide"] = measure_prefill(args, dev, stream, ws, peaks, peak_src, launches=20,
                                               wide=True)
        if rank == 0 and ws == 1 and not args.no_cpu_baseline:
            line["prefill"]["cpu_baseline"] = cpu_baseline_prefill(wl.long_prefill(4096), every_all=1,
                                                                   every_one=16)
            line["prefill_wide"]["cpu_baseline"] = cpu_baseline_prefill(wl.wide_head(args.wide_len),
                                                                        every_all=64, every_one=512)
    if not args.no_e2e:
        line["e2e"] = measure_e2e(args, w, reps, dev, kv_bytes, ws)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def measure_prefill(args, dev, stream, ws, peaks, peak_src, launches: int = 200, wide: bool = False,
                    kv_tile: int = 0):
    """Causal prefill, attention launches alone over rotating replicas;
    TFLOP/s over causal algorithmic flops.  Default: B=1 Q=KV=4096 Dh=128;
    wide: B=1 Q=KV=18432 Hq=16 Hkv=2 Dh=512.  kv_tile: the fixed
    arithmetic's KV tile (0: the head dim's default)."""
    from paged_kv_cache_178_gb300 import pagedattn
    from paged_kv_cache_178_gb300.device import DeviceWorkload
    w = wl.wide_head(args.wide_len) if wide else wl.long_prefill(4096)
    reps = [DeviceWorkload(w, device=str(dev), fill_bits=None) for _ in range(4)]
    for dw in reps:
        dw.write_cache()
    outs = [torch.empty_like(dw.q) for dw in reps]
    lses = [torch.empty(dw.q.shape[:2], dtype=torch.float32, device=dev) for dw in reps]

    def attn(i):
        reps[i % 4].attention(out=outs[i % 4], lse=lses[i % 4], kv_tile=kv_tile)

    with torch.cuda.stream(stream):
        attn(0)
    torch.cuda.synchronize()
    info = pagedattn.last_launch_info()
    g = GraphedSteps(attn, 4, stream, chunk=200)
    g.prepare(8)
    g.run(8)
    n = launches
    t = time_graphed(g, n, stream, ws) / n
    flops = causal_flops(w)
    tf = flops / t / 1e12
    name = (f"causal prefill B=1 Q=KV={args.wide_len} Hq=16 Hkv=2 Dh=512" if wide
            else "causal prefill B=1 Q=KV=4096 Hq=8 Hkv=2 Dh=128")
    return {"workload": name, "tflops": round(tf, 2),
            "us_per_launch": round(t * 1e6, 2), "flops_per_launch": flops,
            "peak": peaks["bf16_tflops"], "frac": round(tf / peaks["bf16_tflops"], 4),
            "peak_source": f"{peak_src} bf16_tflops (burst)", "schedule": info}


def measure_decode_scaled(args, dev, stream, ws, peaks, peak_src, copies: int = 16, launches: int = 50):
    """The decode length mix repeated `copies` times (B = 4*copies requests,
    the same Hq/Hkv/Dh and page size): attention launches alone, K/V bytes of
    valid tokens per launch over the launch time.  With 16 copies a launch
    reads 312 MB, more than twice the L2, so it reads from HBM."""
    from paged_kv_cache_178_gb300 import pagedattn
    from paged_kv_cache_178_gb300.device import DeviceWorkload
    lens = list(wl.DECODE_LENS) * copies
    total_pages = sum(wl.pages_needed(L) for L in lens)
    w = wl.decode(seq_lens=lens, num_blocks=total_pages + 64)
    dw = DeviceWorkload(w, device=str(dev), fill_bits=None)
    dw.write_cache()
    out = torch.empty_like(dw.q)
    lse = torch.empty(dw.q.shape[:2], dtype=torch.float32, device=dev)

    def attn(i):
        dw.attention(out=out, lse=lse)

    with torch.cuda.stream(stream):
        attn(0)
    torch.cuda.synchronize()
    info = pagedattn.last_launch_info()
    g = GraphedSteps(attn, 1, stream, chunk=50)
    g.prepare(launches)
    g.run(4)
    t = time_graphed(g, launches, stream, ws) / launches
    nbytes = attn_io_bytes(w)
    gbs = nbytes / t / 1e9
    return {"workload": f"decode B={len(lens)} (the B=4 length mix x{copies}) Q=1 Hq=8 Hkv=2 Dh=128",
            "gbs": round(gbs, 1), "us_per_launch": round(t * 1e6, 2), "bytes_per_launch": nbytes,
            "peak": peaks["hbm_gbs"], "frac": round(gbs / peaks["hbm_gbs"], 4),
            "peak_source": f"{peak_src} hbm_gbs", "schedule": info}


def measure_gather(args, dev, stream, ws, peaks, peak_src, copies: int = 16, launches: int = 50):
    """Compact active-block gather of one KV head (pa_gather_kv_head) over the
    decode length mix repeated `copies` times, alternating between the two KV
    heads and two packed buffers.  Algorithmic bytes per launch: the selected
    K and V pages of the head read once and written once, plus the table,
    lengths, compact table and offsets."""
    from paged_kv_cache_178_gb300 import pagedattn
    from paged_kv_cache_178_gb300.device import DeviceWorkload
    lens = list(wl.DECODE_LENS) * copies
    total_pages = sum(wl.pages_needed(L) for L in lens)
    w = wl.decode(seq_lens=lens, num_blocks=total_pages + 64)
    dw = DeviceWorkload(w, device=str(dev), fill_bits=None)
    dw.write_cache()
    B, mb = w.block_table.shape
    bufs = [(torch.empty((total_pages, 16, 1, 128), dtype=torch.bfloat16, device=dev),
             torch.empty((total_pages, 16, 1, 128), dtype=torch.bfloat16, device=dev),
             torch.empty((B, mb), dtype=torch.int32, device=dev),
             torch.empty((B + 1,), dtype=torch.int32, device=dev)) for _ in range(2)]
    calls = [pagedattn.prepare_gather_kv_head(dw.k_cache, dw.v_cache, h, dw.block_tables, dw.seq_lens,
                                              *bufs[h], stream=stream) for h in range(2)]

    def gather(i):
        calls[i % 2]()

    with torch.cuda.stream(stream):
        gather(0)
    torch.cuda.synchronize()
    assert pagedattn.check_errors(stream) == (pagedattn.PA_OK, -1)
    g = GraphedSteps(gather, 2, stream, chunk=50)
    g.prepare(launches)
    g.run(4)
    t = time_graphed(g, launches, stream, ws) / launches
    nbytes = 2 * 2 * total_pages * 16 * 128 * 2 + 2 * B * mb * 4 + B * 4 + (B + 1) * 4
    gbs = nbytes / t / 1e9
    return {"workload": f"gather of one KV head, B={B} (the decode length mix x{copies}), "
                        f"{total_pages} pages of 16x128 BF16 each for K and V",
            "gbs": round(gbs, 1), "us_per_launch": round(t * 1e6, 2), "bytes_per_launch": nbytes,
            "peak": peaks["hbm_gbs"], "frac": round(gbs / peaks["hbm_gbs"], 4),
            "peak_source": f"{peak_src} hbm_gbs"}


def _packed(tensors, device=None, pin=False):
    """One byte buffer holding the given tensors at 16-byte aligned offsets,
    and views of it shaped like them (copied in when on the host)."""
    offs, n = [], 0
    for t in tensors:
        offs.append(n)
        n += (t.numel() * t.element_size() + 15) // 16 * 16
    buf = torch.empty(n, dtype=torch.uint8, device=device)
    if pin:
        buf = buf.pin_memory()
    views = []
    for t, o in zip(tensors, offs):
        nb = t.numel() * t.element_size()
        views.append(buf[o:o + nb].view(t.dtype).view(t.shape))
    return buf, views


def measure_e2e(args, w, reps, dev, kv_bytes, ws):
    """Same metric through the public API with host buffers: each step moves
    its inputs (new K/V tokens, slots, q, tables, lengths) from pinned host
    memory to the device, issues the composed cache-write + attention call
    (prepared once: validated and marshalled outside the loop) and brings
    out + lse back to pinned host memory.  The value: the inputs copied by
    the library's staging kernel (pa_copy_to_device reads the pinned buffer
    over the CPU-GPU link), the results written by the attention kernels
    straight into the pinned host buffer.  Beside it, the same step with one
    copy-engine transfer each way (torch copies).  Both wall clock, the steps
    recorded once into CUDA graphs and replayed (how a serving loop issues a
    fixed-shape step); each step issued from Python is reported too."""
    from paged_kv_cache_178_gb300 import pagedattn
    last = last_token_rows(w)
    host_src = (w.key[last].contiguous(), w.value[last].contiguous(), w.slot_mapping[last].contiguous(),
                w.q.contiguous(), w.block_table.contiguous(), w.seq_lens.contiguous(),
                w.query_start_loc.contiguous())
    h_in, h_views = _packed(host_src, pin=True)
    for v, t in zip(h_views, host_src):
        v.copy_(t)
    res_shape = (torch.empty(w.q.shape, dtype=torch.bfloat16), torch.empty(w.q.shape[:2], dtype=torch.float32))
    h_res, (h_out, h_lse) = _packed(res_shape, pin=True)
    stream = torch.cuda.Stream(device=dev)
    staged, calls, calls2, d_ins, d_ress = [], [], [], [], []
    for dw in reps:
        d_in, (k, v, s, q, bt, sl, qsl) = _packed(host_src, device=dev)
        d_res, (out, lse) = _packed(res_shape, device=dev)
        staged.append((pagedattn.prepare_copy_to_device(d_in, h_in, stream=stream, src_ready=True),
                       pagedattn.prepare_reshape_and_paged_attention(
                           k, v, s, q, dw.k_cache, dw.v_cache, bt, sl, qsl, w.scale, w.max_query_len,
                           w.max_seq_len, h_out, h_lse, dw.workspace, stream=stream)))
        calls.append(pagedattn.prepare_reshape_and_paged_attention(
            k, v, s, q, dw.k_cache, dw.v_cache, bt, sl, qsl, w.scale, w.max_query_len, w.max_seq_len, out,
            lse, dw.workspace, stream=stream))
        calls2.append((pagedattn.prepare_reshape_and_cache(k, v, dw.k_cache, dw.v_cache, s, stream=stream),
                       pagedattn.prepare_paged_attention(q, dw.k_cache, dw.v_cache, bt, sl, qsl, w.scale,
                                                         w.max_query_len, w.max_seq_len, out, lse,
                                                         dw.workspace, stream=stream)))
        d_ins.append(d_in)
        d_ress.append(d_res)
    R = len(reps)
    bytes_in = sum(t.numel() * t.element_size() for t in host_src)
    bytes_out = sum(t.numel() * t.element_size() for t in res_shape)

    def step(i):
        r = i % R
        stage, call = staged[r]
        stage()
        call()

    def step_copy_engine(i):
        r = i % R
        d_ins[r].copy_(h_in, non_blocking=True)
        calls[r]()
        h_res.copy_(d_ress[r], non_blocking=True)

    def step_two_calls(i):
        r = i % R
        d_ins[r].copy_(h_in, non_blocking=True)
        write, attend = calls2[r]
        write()
        attend()
        h_res.copy_(d_ress[r], non_blocking=True)

    def wall(run, n):
        torch.cuda.synchronize()
        barrier(ws)
        t0 = time.perf_counter()
        run(n)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        barrier(ws)
        return t1 - t0

    def eager(n):
        with torch.cuda.stream(stream):
            for i in range(n):
                step(i)

    def graphed_time(fn, n):
        g = GraphedSteps(fn, R, stream, chunk=200)
        g.prepare(n)
        g.run(max(args.warmup, 3))
        return wall(g.run, n)

    n = min(args.steps, 2000)
    eager(max(args.warmup, 3))
    t_eager = wall(eager, n)
    t_graph = graphed_time(step, n)
    t_graph_ce = graphed_time(step_copy_engine, n)
    t_graph2 = graphed_time(step_two_calls, n)
    value = aggregate_value(kv_bytes * n / 1e9, t_graph, ws, dev)
    value_eager = aggregate_value(kv_bytes * n / 1e9, t_eager, ws, dev)
    value_ce = aggregate_value(kv_bytes * n / 1e9, t_graph_ce, ws, dev)
    return {"value": round(value, 2), "unit": "GB/s", "h2d_bytes_per_step": bytes_in,
            "d2h_bytes_per_step": bytes_out, "steps": n,
            "ms_per_step": round(t_graph / n * 1e3, 4),
            "eager_value": round(value_eager, 2), "eager_ms_per_step": round(t_eager / n * 1e3, 4),
            "copy_engine_value": round(value_ce, 2), "copy_engine_ms_per_step": round(t_graph_ce / n * 1e3, 4),
            "two_calls_ms_per_step": round(t_graph2 / n * 1e3, 4),
            "how": "public API calls prepared once; per step pa_copy_to_device (the staging kernel reads the "
                   "step's packed inputs from pinned host memory, which only the host writes: src_ready) and "
                   "the composed call, whose attention "
                   "writes out and lse into pinned host memory; steps replayed from CUDA graphs of 200, wall "
                   "clock (eager_*: the same steps issued one by one from Python; copy_engine_*: one torch "
                   "host-to-device and one device-to-host copy around the composed call instead; "
                   "two_calls_*: that, with the step as pa_reshape_and_cache + pa_paged_attention)"}


# ---------------------------------------------------- CPU oracle (baseline) --

def _oracle_decode_setup(w):
    import numpy as np
    from oracle import pa_oracle
    pool = pa_oracle.HostPool(w.num_blocks, w.num_kv_heads, w.head_dim, w.layout)
    kb = w.key.contiguous().view(torch.int16).numpy().view(np.uint16)
    vb = w.value.contiguous().view(torch.int16).numpy().view(np.uint16)
    pa_oracle.reshape_and_cache(kb, vb, w.slot_mapping.numpy(), pool)
    last = last_token_rows(w)
    qb = w.q.contiguous().view(torch.int16).numpy().view(np.uint16)
    return pa_oracle, pool, kb[last], vb[last], w.slot_mapping.numpy()[last], qb


def _oracle_step(ctx, w, threads):
    pa_oracle, pool, kb, vb, slots, qb = ctx
    pa_oracle.reshape_and_cache(kb, vb, slots, pool)
    pa_oracle.paged_attention(qb, pool, w.block_table.numpy(), w.seq_lens.numpy(),
                              w.query_start_loc.numpy(), w.scale, num_threads=threads)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w, seconds: float):
    """The oracle as it stands, full decode steps repeated for about
    `seconds` of CPU time on all host cores, then for a third of that on one
    thread."""
    cores = cpu_cores()
    ctx = _oracle_decode_setup(w)
    _oracle_step(ctx, w, cores)

    def run(threads, budget):
        n, t0 = 0, time.perf_counter()
        while True:
            _oracle_step(ctx, w, threads)
            n += 1
            el = time.perf_counter() - t0
            if el >= budget:
                return n, el

    n, el = run(cores, seconds)
    n1, el1 = run(1, seconds / 3)
    value = decode_bytes(w) * n / el / 1e9
    return {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} full decode steps (cache write of 4 tokens + fp64 attention for all "
                      f"4x8 rows) in {el:.1f} s",
            "one_thread": {"value": round(decode_bytes(w) * n1 / el1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                           "sample": f"{n1} full decode steps in {el1:.1f} s"}}


def _row_flops(w, rows):
    """Causal flops (4*Dh per query row, head and attended key) of the given
    rows of a single-request prefill."""
    L = int(w.seq_lens[0])
    qn = int(w.query_start_loc[1] - w.query_start_loc[0])
    return 4.0 * w.head_dim * w.num_q_heads * sum(L - qn + r + 1 for r in rows)


def cpu_baseline_prefill(w, every_all: int, every_one: int):
    """The oracle as it stands on a single-request causal prefill, timed on
    all host cores on every `every_all`-th query row and on one thread on
    every `every_one`-th row.  A sample of rows is extrapolated to the whole
    prefill by the exact ratio of causal flops (labelled so); the value is
    the sample's causal flops over its time, in TFLOP/s."""
    import numpy as np
    from oracle import pa_oracle
    cores = cpu_cores()
    pool = pa_oracle.HostPool(w.num_blocks, w.num_kv_heads, w.head_dim, w.layout)
    kb = w.key.contiguous().view(torch.int16).numpy().view(np.uint16)
    vb = w.value.contiguous().view(torch.int16).numpy().view(np.uint16)
    pa_oracle.reshape_and_cache(kb, vb, w.slot_mapping.numpy(), pool)
    qb = w.q.contiguous().view(torch.int16).numpy().view(np.uint16)
    n = w.num_q_tokens
    total = _row_flops(w, range(n))

    def timed(every, threads):
        rows = list(range(0, n, every))
        if rows[-1] != n - 1:
            rows.append(n - 1)
        t0 = time.perf_counter()
        pa_oracle.paged_attention(qb, pool, w.block_table.numpy(), w.seq_lens.numpy(),
                                  w.query_start_loc.numpy(), w.scale, rows=rows, num_threads=threads)
        el = time.perf_counter() - t0
        fl = _row_flops(w, rows)
        full = len(rows) == n
        return {"value": round(fl / el / 1e12, 8), "unit": "TFLOP/s", "cores": threads,
                "sample": ("all %d query rows" % n if full else
                           "every %d-th query row and the last (%d of %d rows, %.4f of the causal flops)"
                           % (every, len(rows), n, fl / total)) + f" in {el:.2f} s",
                "full_prefill_s": round(el * total / fl, 3),
                "full_prefill_s_is": "measured" if full else "extrapolated by the exact ratio of causal flops"}

    res = timed(every_all, cores)
    res["kind"] = "oracle"
    res["one_thread"] = timed(every_one, 1)
    return res


def run_reference(args, ws, rank):
    """CPU oracle on the same workload and metric (rank 0 only)."""
    if rank != 0:
        return
    w = wl.decode()
    cores = cpu_cores()
    ctx = _oracle_decode_setup(w)
    _oracle_step(ctx, w, cores)
    t0 = time.perf_counter()
    _oracle_step(ctx, w, cores)
    per_step = time.perf_counter() - t0
    budget = 150.0  # seconds for the whole run
    total = args.steps + max(args.warmup, 3)
    # each step processes a rotating sample of requests if the full step
    # would not fit the budget
    frac = min(1.0, budget / max(total * per_step, 1e-9))
    nreq = max(1, min(w.num_seqs, int(math.floor(frac * w.num_seqs))))
    sub = []
    for r0 in range(w.num_seqs):
        ids = [(r0 + j) % w.num_seqs for j in range(nreq)]
        sub.append(ids)
    import numpy as np
    pa_oracle, pool, kb, vb, slots, qb = ctx

    def ref_step(i):
        ids = sub[i % len(sub)]
        pa_oracle.reshape_and_cache(kb[ids], vb[ids], slots[ids], pool)
        qsl = np.arange(len(ids) + 1, dtype=np.int32)
        pa_oracle.paged_attention(qb[ids], pool, w.block_table.numpy()[ids], w.seq_lens.numpy()[ids],
                                  qsl, w.scale, num_threads=cores)
        return int(w.seq_lens[ids].sum()) * w.num_kv_heads * w.head_dim * 4

    for i in range(max(args.warmup, 3)):
        ref_step(i)
    t0 = time.perf_counter()
    nbytes = 0
    for i in range(args.steps):
        nbytes += ref_step(i)
    el = time.perf_counter() - t0
    value = nbytes / el / 1e9
    sample = ("full decode steps" if nreq == w.num_seqs else
              f"{nreq} of {w.num_seqs} requests per step, rotating; bytes counted for those requests")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": ws, "steps": args.steps, "warmup": max(args.warmup, 3),
            "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "decode B=4 Q=1 KV={7168,7168,4171,513} Hq=8 Hkv=2 Dh=128 page16 "
                                   "interleaved pool 2048 blocks, shuffled pages",
                       "step": "oracle cache write + fp64 attention", "parallelism": "host cores"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["decode", "prefill", "wide", "gather", "decode_scaled"],
                    default="decode",
                    help="decode (default, the headline), one causal prefill alone: prefill (Dh=128, "
                         "4096) or wide (Dh=512, 18432), the compact gather, or decode_scaled (the "
                         "decode length mix x16, attention launches alone)")
    ap.add_argument("--replicas", type=int, default=16)
    ap.add_argument("--wide-len", type=int, default=18432,
                    help="sequence length of the Dh=512 prefill (3072, 8192, 11264 or 18432)")
    ap.add_argument("--cpu-seconds", type=float, default=9.0)
    ap.add_argument("--min-repeats", type=int, default=7,
                    help="the headline's K-step region is timed at least this many times (median reported)")
    ap.add_argument("--min-timed-s", type=float, default=0.1,
                    help="... and repeated until this many seconds of timed steps have run")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    ws, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    run_ours(args, ws, rank, local)


if __name__ == "__main__":
    main()
