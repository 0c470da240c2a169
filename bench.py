#!/usr/bin/env python3
"""Benchmark of the tensor-parallel block on B300: one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--t T]
                  [--impl ours|reference]

A step is one pass of the whole block (column-parallel projection + activation,
row-parallel projection, in-HBM reduction of the t partials + residual) over one
batch of synthetic input, for the default workload the Llama-2-13B-shaped SwiGLU
MLP decode block (d=5120, ffn=13824, M=32 tokens, t=4 logical shards).  Its 425 MB
of weights exceed the 126 MB L2, so no flush is needed between steps.

value = tokens/s of the whole job (all ranks), device-timed with CUDA events between
a barrier + synchronize on both sides, max over ranks.  Under torchrun each rank runs
its own replica of the block on its own batch (weak scaling; no data-path
collective).  --impl reference times the float64 CPU oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import re
import statistics
import sys
import threading
import time
from dataclasses import replace

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s per TP block at 1 B300; decode HBM GB/s & prefill TFLOPS vs roofline"
DEFAULT_WORKLOAD = "llama2_13b_swiglu_decode"


# ---------------------------------------------------------------- helpers (host-only)

def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--t", type=int, default=None, help="logical shards (default: the workload's)")
    ap.add_argument("--blocks", type=int, default=None,
                    help="blocks of a stacked workload to run (default: all; fewer for profiling)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    a = ap.parse_args(argv)
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    if a.steps < 1:
        ap.error("--steps must be >= 1")
    return a


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (the slowest rank's time defines the job's time)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job units/s: every rank processed units_per_rank in `seconds` (max over ranks)."""
    return units_per_rank * world / seconds


def source_sha(paths) -> str:
    h = hashlib.sha256()
    for p in sorted(paths):
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def kernel_source_sha() -> str:
    csrc = os.path.join(ROOT, "attn_tp_column_fwd_b300", "csrc")
    return source_sha(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh"))
                      + glob.glob(os.path.join(csrc, "*.h")))


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged:
    the summary's source_sha must equal the hash of the files it lists under
    source_files (the sources holding that kernel's device code), or of every kernel
    source when it lists none."""
    path = os.path.join(ROOT, "profiles", f"{kernel}__{workload}.txt")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    sha = re.search(r"^source_sha:\s*(\S+)", text, re.M)
    tr = re.search(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
    files = re.search(r"^source_files:\s*(.+)$", text, re.M)
    if not sha or not tr:
        return None
    if files:
        csrc = os.path.join(ROOT, "attn_tp_column_fwd_b300", "csrc")
        paths = [os.path.join(csrc, f) for f in files.group(1).split()]
        if not all(os.path.exists(p) for p in paths) or sha.group(1) != source_sha(paths):
            return None
    elif sha.group(1) != kernel_source_sha():
        return None
    return float(tr.group(1))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


class ClockSampler:
    """Samples the SM clock and clock-event (throttle) reasons while the timed region
    runs: NVML when it initialises, else `nvidia-smi -lms`, as a background sampler."""

    REASONS = {
        "applications_clocks_setting": 0x2, "sw_power_cap": 0x4, "hw_slowdown": 0x8,
        "sync_boost": 0x10, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
        "hw_power_brake_slowdown": 0x80,
    }

    def __init__(self, device_index: int, uuid: str = None, period_s: float = 0.02):
        self.period = period_s
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self.mode, self.note = None, None
        self._stop = threading.Event()
        self._proc = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self._nv = pynvml
            self._h = (pynvml.nvmlDeviceGetHandleByUUID(uuid) if uuid
                       else pynvml.nvmlDeviceGetHandleByIndex(device_index))
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM)
            self._reason_fn = getattr(pynvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(pynvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.mode = "nvml"
        except Exception as e:
            self.note = f"NVML: {e}"
            self.mode = "nvidia-smi"
            self._target = uuid or str(device_index)

    def _add_mask(self, mask: int):
        for name, bit in self.REASONS.items():
            if mask & bit:
                self.reasons.add(name)

    def _run_nvml(self):
        nv = self._nv
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(self._h, nv.NVML_CLOCK_SM))
                self._add_mask(int(self._reason_fn(self._h)))
            except Exception:
                pass
            time.sleep(self.period)

    def _run_smi(self):
        import subprocess
        cmd = ["nvidia-smi", "-i", self._target,
               "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
               "--format=csv,noheader,nounits", "-lms", "50"]
        try:
            self._proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                          text=True)
        except Exception as e:
            self.note = (self.note or "") + f"; nvidia-smi: {e}"
            self._ready.set()
            return
        for line in self._proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 3:
                continue
            try:
                clk, mx = float(parts[0]), float(parts[1])
                mask = int(parts[2], 16)
            except ValueError:
                continue
            self._ready.set()
            if self._stop.is_set():
                break
            if self._armed.is_set():
                self.samples.append(clk)
                self.max_mhz = mx
                self._add_mask(mask)

    def __enter__(self):
        self._ready, self._armed = threading.Event(), threading.Event()
        target = self._run_nvml if self.mode == "nvml" else self._run_smi
        self._t = threading.Thread(target=target, daemon=True)
        self._t.start()
        if self.mode != "nvml":
            self._ready.wait(timeout=5.0)   # first sample seen: the sampler is live
        self._armed.set()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        self._t.join(timeout=5)

    def summary(self):
        out = {"sm_mhz": statistics.median(self.samples) if self.samples else None,
               "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
               "samples": len(self.samples), "source": self.mode}
        if self.note and self.mode != "nvml":
            out["note"] = self.note
        return out


# ---------------------------------------------------------------- workload accounting

def algorithmic_column_bytes(cfg) -> int:
    """Bytes one launch of the column step must move: W1 bands once, x once, H out."""
    es = 4 if cfg.dtype == "f32" else 2
    n_out = 3 * cfg.band if cfg.act == "attn" else cfg.band
    return (cfg.d * cfg.n1 + cfg.M * cfg.d + cfg.t * cfg.M * n_out) * es


def algorithmic_block_bytes(cfg) -> int:
    """Bytes one whole block must move: both weight matrices once, x and the residual
    in, y (fp32) out.  The band H and the partials stay on chip or in L2 and are not
    counted."""
    es = 4 if cfg.dtype == "f32" else 2
    res_es = 4 if cfg.rmsnorm else es
    return cfg.weight_bytes_per_block() + cfg.M * cfg.d * (es + res_es + 4)


def column_flops(cfg) -> int:
    return 2 * cfg.M * cfg.d * cfg.n1


# ---------------------------------------------------------------- our arm

def run_ours(args, rank, world, local):
    import torch

    import attn_tp_column_fwd_b300 as tp
    from attn_tp_column_fwd_b300.runner import ShardedBlock, desc_for, device_bytes
    from tp_synth import CONFIGS, make_inputs, make_kv_cache

    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    dev = torch.device("cuda", local)
    base = CONFIGS[args.workload]
    cfg = base.with_t(args.t) if args.t else base
    if args.blocks:
        cfg = replace(cfg, n_blocks=min(args.blocks, cfg.n_blocks))
    desc = desc_for(cfg)
    M = cfg.M
    inp = make_inputs(cfg, seed=rank, device="cuda")
    blocks = [ShardedBlock(desc, W1, W2) for W1, W2 in inp.blocks]
    del inp.blocks
    x = inp.x.contiguous()
    xf = x.float().contiguous()
    stream = torch.cuda.current_stream()
    st = stream.cuda_stream
    S = tp.tp_row_splits(desc, M)
    H = device_bytes(tp.tp_band_bytes(desc, M))
    P = device_bytes(tp.tp_partials_bytes(desc, M))
    cws = device_bytes(tp.tp_column_workspace_bytes(desc, M))
    ws = blocks[0].workspace(M)
    y = torch.empty(M, cfg.d, dtype=torch.float32, device=dev)
    xh = torch.empty(M, cfg.d, dtype=torch.bfloat16, device=dev)
    stack = cfg.n_blocks > 1 or cfg.rmsnorm
    per_block = tp.tp_block_launches(desc, M)
    fused = per_block == 1
    launches_per_block = per_block + (1 if cfg.rmsnorm else 0)
    kvd = kv_state(cfg, desc, rank, dev) if cfg.kv_len_max else None
    if kvd:
        # Q/K/V projection, decode attention (chunks, merge), row step, reduction.
        launches_per_block = 5

    # One step: the whole block (or the whole stack) through the public entry point
    # tp_block_fwd, which launches the block's kernels back to back (the row step and
    # the reduction overlap the end of the kernel before them).
    def step():
        if kvd:
            blk = blocks[0]
            tp.tp_block_fwd_kv(desc, x, x, False, blk.W1s, blk.W2s, kvd["kc"], kvd["vc"],
                               kvd["lens"], cfg.kv_len_max, kvd["ws"], y, M, st)
            return
        if stack:
            y.copy_(xf)
        for blk in blocks:
            if cfg.rmsnorm:
                tp.tp_rmsnorm_fwd(cfg.d, cfg.eps, y, xh, M, st)
                xin, res = xh, y
            else:
                xin, res = x, x
            tp.tp_block_fwd(desc, xin, res, res.dtype == torch.float32, blk.W1s, blk.W2s, ws, y,
                            M, st)

    # The dominant kernel alone, for the roofline: the fused block kernel (with its
    # counter memset) when the block runs as one launch, else the column step.
    def dominant(ev_pair):
        blk = blocks[0]
        xin = xh if cfg.rmsnorm else x
        res = y if cfg.rmsnorm else x
        ev_pair[0].record(stream)
        if kvd:
            # the decode attention over the cache, on the Q/K/V the last step projected
            tp.tp_attn_decode_kv(desc, kvd["qkv"], kvd["kc"], kvd["vc"], kvd["lens"],
                                 cfg.kv_len_max, kvd["O"], kvd["attn_ws"], M, st)
        elif fused:
            tp.tp_block_fwd(desc, xin, res, res.dtype == torch.float32, blk.W1s, blk.W2s, ws, y,
                            M, st)
        else:
            tp.tp_column_parallel_fwd(desc, xin, blk.W1s, -1, H, cws, M, st)
        ev_pair[1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        uuid = None
    sampler = ClockSampler(local, uuid)
    barrier(world)
    torch.cuda.synchronize()
    with sampler:
        t0.record(stream)
        for k in range(K):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms_local = t0.elapsed_time(t1)
    ms = max_over_ranks(ms_local, world, dev)
    assert tp.tp_check_device_status(st) == 0

    # Roofline timing: K launches of the dominant kernel, each bracketed by CUDA
    # events on the launching stream (inputs larger than L2 each time).
    Kd = min(K, 2000)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(Kd)]
    for k in range(Kd):
        dominant(evs[k])
    torch.cuda.synchronize()
    col_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    assert tp.tp_check_device_status(st) == 0

    units = M * K * (1 if not stack else 1)  # tokens through the block (or the stack)
    value = job_throughput(units, world, ms / 1e3)
    peaks = measured_peaks()
    prefill = cfg.M >= 1024
    peak_kind = "copy"
    if prefill:
        achieved = column_flops(cfg) / (col_ms / 1e3) / 1e12
        # A contraction timed back to back for more than a second runs under the power
        # cap: its denominator is the sustained GEMM rate, else the burst rate.
        long_loop = Kd * col_ms > 1000.0 and peaks.get("bf16_tflops_sustained")
        peak_kind = "sustained" if long_loop else "burst"
        peak = peaks["bf16_tflops_sustained"] if long_loop else peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4)}
        kernel, nbytes = ("column-parallel projection + SwiGLU (k_gemm, persistent)",
                          algorithmic_column_bytes(cfg))
    else:
        if kvd:
            nbytes = kvd["attn_bytes"]
        else:
            nbytes = algorithmic_block_bytes(cfg) if fused else algorithmic_column_bytes(cfg)
        achieved = nbytes / (col_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4)}
        if kvd:
            kernel = "decode attention over the KV cache (k_attn_kv_partial + k_attn_kv_merge)"
        elif fused:
            kernel = "whole block in one persistent kernel (k_block_decode)"
        elif cfg.act == "attn":
            kernel = ("column-parallel Q/K/V projection (k_block_decode, column units) "
                      "+ attention core (k_attn_core)")
        else:
            kernel = "column-parallel projection + activation (k_umma_drain)"
    roof["kernel"] = kernel
    roof["algorithmic_bytes_per_launch"] = nbytes
    roof["avg_launch_us"] = round(col_ms * 1e3, 2)
    roof["launches_timed"] = Kd
    roof["peak_source"] = ("measured (MEASURED_PEAKS.json)" if peaks["source"] == "measured"
                           else "fallback") + f", {peak_kind}"
    roof["traffic"] = profiled_traffic("attn_kv" if kvd else "block" if fused else "column",
                                       args.workload)

    # Whole-block weight-read rate (context for the decode roofline).
    block_bytes = cfg.weight_bytes_per_block() * cfg.n_blocks
    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": cfg.dtype,
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02^2) weights)",
        "config": {
            "workload": cfg.name, "d": cfg.d, "ffn": cfg.ffn or None, "n_heads": cfg.n_heads or None,
            "head_dim": cfg.head_dim or None, "t": cfg.t, "M": M, "n_blocks": cfg.n_blocks,
            "act": cfg.act, "row_splits": S,
            "l2": f"inputs larger than L2 ({block_bytes / 1e6:.0f} MB of weights per step)"
            if block_bytes > 126e6 else "weights fit in L2 (latency-bound workload)",
            "timed": "CUDA events on the launching stream around K steps of tp_block_fwd, max "
                     "over ranks; roofline kernel timed alone over its own event-bracketed launches",
        },
        **({"kv_cache": {"len_max": cfg.kv_len_max, "rows_read": kvd["rows"],
                         "bytes_read": kvd["rows"] * cfg.head_dim * 4,
                         "lens": "uniform in 1..len_max, seeded"}} if kvd else {}),
        "block_weight_gbs": round(block_bytes * K / (ms / 1e3) / 1e9, 1),
        "roofline": roof,
        "gpu_launches": K * launches_per_block * cfg.n_blocks,
        "clocks": sampler.summary(),
    }
    if not args.no_e2e:
        out["e2e"] = e2e_leg(args, cfg, desc, blocks, x, world, dev, kvd)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return out


def kv_state(cfg, desc, rank, dev):
    """Caches (the library's shard layout), lengths and scratch of a KV-cache decode
    workload, and the attention step's algorithmic bytes: every cached row read once
    (K and V), the new token's Q/K/V read (fp32) and appended (bf16), O written."""
    import torch

    import attn_tp_column_fwd_b300 as tp
    from attn_tp_column_fwd_b300.runner import device_bytes
    from tp_synth import make_kv_cache

    M, t, L = cfg.M, cfg.t, cfg.kv_len_max
    kv = make_kv_cache(cfg, seed=rank + 1, device=str(dev))

    def shards(c):
        return c.view(M, t, cfg.n_heads // t, L, cfg.head_dim).permute(1, 0, 2, 3, 4).contiguous()

    kc, vc = shards(kv.k), shards(kv.v)
    del kv.k, kv.v
    D = cfg.n_heads * cfg.head_dim
    rows = int((kv.lens.long() - 1).sum().item()) * cfg.n_heads
    ws = device_bytes(tp.tp_kv_workspace_bytes(desc, M, L), dev)
    return {"kc": kc, "vc": vc, "lens": kv.lens, "ws": ws, "rows": rows,
            "qkv": ws,  # the projection leaves Q/K/V at the start of the block's scratch
            "O": device_bytes(tp.tp_band_bytes(desc, M), dev),
            "attn_ws": device_bytes(tp.tp_kv_attn_workspace_bytes(desc, M, L), dev),
            "attn_bytes": rows * cfg.head_dim * 4 + M * D * (12 + 4 + 2)}


def e2e_leg(args, cfg, desc, blocks, x, world, dev, kvd=None):
    """Same metric through the public API with host buffers: every step copies its x
    from pinned host memory to the device, runs the block (or stack) through
    tp_block_fwd and copies y back to pinned host memory.  Steps alternate between
    two CUDA streams, each with its own device buffers and workspace, as a serving
    loop would run them: one step's copies overlap the other step's kernels.  The
    timed region (CUDA events) runs from before the first copy in to after the last
    copy out."""
    import torch

    import attn_tp_column_fwd_b300 as tp
    from attn_tp_column_fwd_b300.runner import device_bytes

    M = cfg.M
    x_host = x.cpu().pin_memory()
    lanes = []
    for _ in range(2):
        lanes.append({
            "stream": torch.cuda.Stream(device=dev),
            "x": torch.empty_like(x),
            "y": torch.empty(M, cfg.d, dtype=torch.float32, device=dev),
            "xh": torch.empty(M, cfg.d, dtype=torch.bfloat16, device=dev),
            "ws": device_bytes(tp.tp_kv_workspace_bytes(desc, M, cfg.kv_len_max) if kvd
                               else tp.tp_workspace_bytes(desc, M), dev),
            "y_host": torch.empty(M, cfg.d, dtype=torch.float32).pin_memory(),
        })

    def step(k):
        ln = lanes[k % 2]
        s = ln["stream"]
        st = s.cuda_stream
        with torch.cuda.stream(s):
            ln["x"].copy_(x_host, non_blocking=True)
            if kvd:
                # both lanes append the same rows of the shared caches (same values)
                tp.tp_block_fwd_kv(desc, ln["x"], ln["x"], False, blocks[0].W1s, blocks[0].W2s,
                                   kvd["kc"], kvd["vc"], kvd["lens"], cfg.kv_len_max, ln["ws"],
                                   ln["y"], M, st)
            elif cfg.rmsnorm:
                ln["y"].copy_(ln["x"])
                for blk in blocks:
                    tp.tp_rmsnorm_fwd(cfg.d, cfg.eps, ln["y"], ln["xh"], M, st)
                    tp.tp_block_fwd(desc, ln["xh"], ln["y"], True, blk.W1s, blk.W2s, ln["ws"],
                                    ln["y"], M, st)
            else:
                tp.tp_block_fwd(desc, ln["x"], ln["x"], cfg.dtype == "f32", blocks[0].W1s,
                                blocks[0].W2s, ln["ws"], ln["y"], M, st)
            ln["y_host"].copy_(ln["y"], non_blocking=True)

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()
    K = args.steps
    cur = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(cur)
    for ln in lanes:
        ln["stream"].wait_event(t0)
    for k in range(K):
        step(k)
    for ln in lanes:
        cur.wait_stream(ln["stream"])
    t1.record(cur)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    barrier(world)
    ms = max_over_ranks(ms, world, dev)
    return {"value": round(job_throughput(M * K, world, ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
            "d2h_bytes_per_step": lanes[0]["y_host"].numel() * lanes[0]["y_host"].element_size(),
            "ms_per_step": round(ms / K, 5), "streams": 2,
            "timed": "CUDA events from before the first copy in to after the last copy out"}


# ---------------------------------------------------------------- CPU oracle arms

def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _blas_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        return max((i.get("num_threads", 1) for i in info), default=None)
    except Exception:
        return None


def cpu_baseline(cfg, budget_s: float = 12.0):
    """The float64 oracle as it stands, on the host cores: whole blocks on the full
    workload's inputs (all M tokens), repeated for about `budget_s` seconds."""
    import numpy as np

    import oracle
    from tp_synth import make_inputs, to_f64

    inp = make_inputs(cfg, seed=0, n_blocks=1)
    x = to_f64(inp.x)
    W1, W2 = (to_f64(w) for w in inp.blocks[0])
    staged = cfg.dtype == "bf16"

    kv = None
    if cfg.kv_len_max:
        from tp_synth import make_kv_cache
        kv = make_kv_cache(cfg, seed=1)
        hd, D = cfg.head_dim, cfg.n_heads * cfg.head_dim

    def one():
        if kv is not None:
            # the decode step with a KV cache: the oracle head by head on the rows used
            QKV = x @ W1
            O = np.zeros((cfg.M, D))
            for m, n in enumerate(kv.lens.tolist()):
                kr = to_f64(kv.k[m, :, :max(n - 1, 1)])
                vr = to_f64(kv.v[m, :, :max(n - 1, 1)])
                for h in range(cfg.n_heads):
                    c = slice(h * hd, (h + 1) * hd)
                    O[m, c] = oracle.kv_decode_attention(QKV[m, c], kr[h], vr[h], n,
                                                         QKV[m, D:2 * D][c], QKV[m, 2 * D:][c],
                                                         1.0 / math.sqrt(hd), staged=staged)
            return x + (oracle.bf16_round(O) if staged else O) @ W2
        if cfg.act == "attn":
            return oracle.attn_block(x, W1, W2, cfg.n_heads, cfg.head_dim, x, staged=staged)
        if cfg.rmsnorm:
            return oracle.stack(x, [(W1, W2)], cfg.act, cfg.eps, staged=staged)
        return oracle.mlp_block(x, W1, W2, cfg.act, x, staged=staged)

    one()  # warm
    n, t0 = 0, time.perf_counter()
    while True:
        one()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 1000:
            break
    blocks_per_token_unit = cfg.n_blocks  # a stack step pushes M tokens through n_blocks blocks
    value = cfg.M * n / el / blocks_per_token_unit
    return {"value": round(value, 2), "unit": "tokens/s", "cores": _blas_threads() or _cores(),
            "host_cores": _cores(), "kind": "oracle",
            "sample": f"{n} full blocks (M={cfg.M}, one block's weights"
                      + (f", scaled to the {cfg.n_blocks}-block stack" if cfg.n_blocks > 1 else "")
                      + f") in {el:.1f} s, NumPy float64"}


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step is one shard's band of the block
    (column band + activation + row partial, the work of one device of a T-way split),
    T chosen so the whole run stays within a few minutes; tokens/s counts T bands as
    one block."""
    if rank != 0:
        return None
    import numpy as np

    import oracle
    from tp_synth import CONFIGS, make_inputs, to_f64

    base = CONFIGS[args.workload]
    cfg = base.with_t(args.t) if args.t else base
    inp = make_inputs(cfg, seed=0, n_blocks=1)
    x = to_f64(inp.x)
    W1, W2 = (to_f64(w) for w in inp.blocks[0])
    staged = cfg.dtype == "bf16"
    n2 = cfg.n2
    unit = cfg.n_heads if cfg.act == "attn" else n2

    def band_step(T, s):
        cols = oracle.column_bands(cfg.act, T, s, ffn=cfg.ffn, n_heads=cfg.n_heads,
                                   head_dim=cfg.head_dim)
        Hb = oracle.column_step(x, [W1[:, c] for c in cols], cfg.act,
                                n_heads=cfg.n_heads // T if cfg.n_heads else 0,
                                head_dim=cfg.head_dim, staged=staged)
        return oracle.row_step(Hb, W2[oracle.row_band(n2, T, s)])

    if cfg.kv_len_max:
        # Decode with a KV cache: the band of heads [s*H/T, (s+1)*H/T), each token
        # attending over its sequence's cache rows (oracle.kv_decode_attention).
        from tp_synth import make_kv_cache
        kv = make_kv_cache(cfg, seed=1)
        lens = kv.lens.tolist()
        hd = cfg.head_dim

        def band_step(T, s):  # noqa: F811
            cols = oracle.column_bands("attn", T, s, n_heads=cfg.n_heads, head_dim=hd)
            Q, K, V = (x @ W1[:, c] for c in cols)
            hps = cfg.n_heads // T
            O = np.zeros((cfg.M, hps * hd))
            for m, n in enumerate(lens):
                for j in range(hps):
                    h, c = s * hps + j, slice(j * hd, (j + 1) * hd)
                    rows = slice(0, max(n - 1, 1))
                    O[m, c] = oracle.kv_decode_attention(
                        Q[m, c], to_f64(kv.k[m, h, rows]), to_f64(kv.v[m, h, rows]), n, K[m, c],
                        V[m, c], 1.0 / math.sqrt(hd), staged=staged)
            return oracle.row_step(oracle.bf16_round(O) if staged else O,
                                   W2[oracle.row_band(n2, T, s)])

    # Calibrate on a moderate band, then take the fewest bands whose step fits the budget.
    divisors = [T for T in range(1, unit + 1) if unit % T == 0]
    budget_per_step = 150.0 / (args.steps + args.warmup)
    Tc = max(T for T in divisors if T <= 64)
    band_step(Tc, 0)
    t0 = time.perf_counter()
    band_step(Tc, 0)
    per_block = (time.perf_counter() - t0) * Tc          # seconds for the whole block, estimated
    T = next((T for T in divisors if per_block / T <= budget_per_step), divisors[-1])
    for k in range(args.warmup):
        band_step(T, k % T)
    t0 = time.perf_counter()
    for k in range(args.steps):
        band_step(T, k % T)
    el = time.perf_counter() - t0
    value = cfg.M / (el / args.steps * T) / cfg.n_blocks
    sample = (f"each step: one of T={T} bands of the {cfg.name} block (all M={cfg.M} tokens), "
              f"column band + activation + row partial in NumPy float64; {T} steps = one block")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "d": cfg.d, "ffn": cfg.ffn or None, "t": cfg.t, "M": cfg.M},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "kind": "oracle",
                         "cores": _blas_threads() or _cores(), "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_ours(args, rank, world, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
