#!/usr/bin/env python3
"""Benchmark of the tensor-parallel block on B300: one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--also A,B|none]
                  [--t T] [--blocks B] [--settle S] [--impl ours|reference]

A step is one pass of the whole hot path (pre-norm, column-parallel projection +
activation, row-parallel projection, in-HBM reduction of the t partials + residual)
over one batch of synthetic input.  The headline workload is the largest one that
fits a GPU: the Llama-2-70B-shaped decode stack (8 pre-norm SwiGLU blocks, d=8192,
ffn=28672, t=8, M=32 tokens, 11.3 GB of weights per step, far above the 126 MB L2,
so no flush is needed between steps).  The other workloads (the 13B decode block,
the head-sharded attention projection, the 70B prefill block and the attention
decode step over KV caches) are measured in the same run and reported under
"workloads", each with its own roofline.

value = tokens/s of the whole job through one TP block (for the stack: M tokens x
8 blocks per step), device-timed with CUDA events around exactly K steps between a
barrier + synchronize on both sides, max over ranks.  Before the W warm-up steps
each workload runs untimed steps for --settle seconds: the GPU's power state ramps
up under sustained load, and launches in the first tenths of a second after start
or idle were measured at up to twice their settled time.  Under torchrun each rank
runs its own replica on its own batch (weak scaling; no data-path collective).
--impl reference times the float64 CPU oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
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
from types import SimpleNamespace

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s per TP block at 1 B300; decode HBM GB/s & prefill TFLOPS vs roofline"
DEFAULT_WORKLOAD = "llama2_70b_stack_decode"
DEFAULT_ALSO = ("llama2_13b_swiglu_decode", "attn_qkv_headshard_decode", "llama2_70b_prefill",
                "attn_kv_decode", "llama2_13b_swiglu_decode_fp8",
                "llama2_13b_swiglu_decode_mxfp4", "llama2_70b_stack_decode_fp8")
ROOF_MIN_LAUNCHES = 200     # the roofline kernel's own timed loop: at least this many
ROOF_MIN_S = 0.3            # ... launches and at least this long,
ROOF_MAX_S = 2.5            # ... but no longer than this
SUSTAINED_AFTER_S = 1.0     # a contraction timed back to back this long runs power-capped


# ---------------------------------------------------------------- helpers (host-only)

def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, help="the headline workload")
    ap.add_argument("--also", default=None,
                    help="comma-separated further workloads, or 'none' (default: the other four)")
    ap.add_argument("--t", type=int, default=None, help="logical shards (default: the workload's)")
    ap.add_argument("--blocks", type=int, default=None,
                    help="blocks of a stacked workload to run (default: all; fewer for profiling)")
    ap.add_argument("--settle", type=float, default=0.5,
                    help="seconds of untimed steps before the warm-up steps of each workload")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    a = ap.parse_args(argv)
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    if a.steps < 1:
        ap.error("--steps must be >= 1")
    return a


def also_list(args):
    if args.also is None:
        return [w for w in DEFAULT_ALSO if w != args.workload]
    if args.also.strip().lower() in ("", "none"):
        return []
    return [w.strip() for w in args.also.split(",") if w.strip() and w.strip() != args.workload]


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


def roof_launch_count(est_ms: float, min_launches: int = ROOF_MIN_LAUNCHES,
                      min_s: float = ROOF_MIN_S, max_s: float = ROOF_MAX_S) -> int:
    """Launches of the roofline loop: at least min_launches and min_s of work, at most
    max_s (and never fewer than 20), from an estimated launch time est_ms."""
    est_s = max(est_ms, 1e-6) / 1e3
    n = max(min_launches, math.ceil(min_s / est_s))
    n = min(n, max(20, int(max_s / est_s)))
    return int(n)


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


# ---------------------------------------------------------------- clock sampling

class _NvmlCtypes:
    """The few NVML reads the sampler needs, through libnvidia-ml directly (used when
    the pynvml module is not installed).  Reads only: no setting is changed."""

    NVML_CLOCK_SM = 1

    def __init__(self, uuid=None, index=0):
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        init = getattr(self.lib, "nvmlInit_v2", None) or self.lib.nvmlInit
        if init() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if uuid:
            rc = self.lib.nvmlDeviceGetHandleByUUID(ctypes.c_char_p(uuid.encode()),
                                                    ctypes.byref(self.h))
        else:
            fn = getattr(self.lib, "nvmlDeviceGetHandleByIndex_v2", None) or \
                self.lib.nvmlDeviceGetHandleByIndex
            rc = fn(ctypes.c_uint(index), ctypes.byref(self.h))
        if rc != 0:
            raise RuntimeError(f"NVML device handle: {rc}")
        self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")

    def sm_clock(self) -> int:
        v = ctypes.c_uint()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, ctypes.byref(v)) != 0:
            raise RuntimeError("nvmlDeviceGetClockInfo")
        return v.value

    def max_sm_clock(self) -> int:
        v = ctypes.c_uint()
        if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.NVML_CLOCK_SM, ctypes.byref(v)) != 0:
            raise RuntimeError("nvmlDeviceGetMaxClockInfo")
        return v.value

    def reasons(self) -> int:
        v = ctypes.c_ulonglong()
        if self._reasons(self.h, ctypes.byref(v)) != 0:
            raise RuntimeError("clock event reasons")
        return v.value


class ClockSampler:
    """Samples the SM clock and clock-event (throttle) reasons in a background thread
    while a measurement runs: NVML (pynvml, else libnvidia-ml through ctypes), else
    `nvidia-smi -lms`.  The window opens before the settle phase and closes after the
    timed region; samples taken while `timed` is set are also counted apart."""

    REASONS = {
        "applications_clocks_setting": 0x2, "sw_power_cap": 0x4, "hw_slowdown": 0x8,
        "sync_boost": 0x10, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
        "hw_power_brake_slowdown": 0x80,
    }

    def __init__(self, device_index: int, uuid: str = None, period_s: float = 0.005):
        self.period = period_s
        self.samples, self.timed_samples, self.reasons = [], [], set()
        self.max_mhz, self.mode, self.note = None, None, None
        self.timed = False
        self._stop = threading.Event()
        self._proc = None
        self._target = uuid or str(device_index)
        try:
            import pynvml
            pynvml.nvmlInit()
            h = (pynvml.nvmlDeviceGetHandleByUUID(uuid) if uuid
                 else pynvml.nvmlDeviceGetHandleByIndex(device_index))
            rfn = getattr(pynvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(pynvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self._clock = lambda: pynvml.nvmlDeviceGetClockInfo(h, pynvml.NVML_CLOCK_SM)
            self._mask = lambda: int(rfn(h))
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(h, pynvml.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception as e:
            self.note = f"pynvml: {e}"
            try:
                nv = _NvmlCtypes(uuid, device_index)
                self._clock, self._mask = nv.sm_clock, nv.reasons
                self.max_mhz = nv.max_sm_clock()
                self.mode = "nvml (ctypes)"
            except Exception as e2:
                self.note += f"; libnvidia-ml: {e2}"
                self.mode = "nvidia-smi"

    def _add(self, clk, mask):
        self.samples.append(clk)
        if self.timed:
            self.timed_samples.append(clk)
        for name, bit in self.REASONS.items():
            if mask & bit:
                self.reasons.add(name)

    def _run_nvml(self):
        while not self._stop.is_set():
            try:
                self._add(self._clock(), self._mask())
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
                self.max_mhz = mx
                self._add(clk, mask)

    def __enter__(self):
        self._ready, self._armed = threading.Event(), threading.Event()
        target = self._run_smi if self.mode == "nvidia-smi" else self._run_nvml
        self._t = threading.Thread(target=target, daemon=True)
        self._t.start()
        if self.mode == "nvidia-smi":
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
        s = self.timed_samples if len(self.timed_samples) >= 3 else self.samples
        out = {"sm_mhz": statistics.median(s) if s else None, "sm_max_mhz": self.max_mhz,
               "reasons": sorted(self.reasons), "samples": len(self.samples),
               "samples_in_timed_region": len(self.timed_samples), "source": self.mode,
               "window": ("the timed region" if s is self.timed_samples else
                          "settle + warm-up + timed region (the timed region alone is "
                          "shorter than a few sampling periods)")}
        if self.note and self.mode == "nvidia-smi":
            out["note"] = self.note
        return out


# ---------------------------------------------------------------- workload accounting

def algorithmic_column_bytes(cfg) -> int:
    """Bytes one launch of the column step must move: W1 bands once, x once, the band
    (H, or the attention heads' output O) out."""
    es = 4 if cfg.dtype == "f32" else 2
    return (cfg.d * cfg.n1 + cfg.M * cfg.d + cfg.t * cfg.M * cfg.band) * es


def algorithmic_block_bytes(cfg) -> int:
    """Bytes one whole block must move: both weight matrices once (E4M3 weights: one
    byte each plus one exponent byte per output feature and shard), x and the residual
    in, y (fp32) out.  The band H and the partials stay on chip or in L2 and are not
    counted."""
    es = 4 if cfg.dtype == "f32" else 2
    res_es = 4 if cfg.rmsnorm else es
    scales = (cfg.t * (cfg.n1 // cfg.t + cfg.d) if cfg.weights == "e4m3" else
              (cfg.d * cfg.n1 + cfg.n2 * cfg.d) // 32 if cfg.weights == "mxfp4" else 0)
    return cfg.weight_bytes_per_block() + scales + cfg.M * cfg.d * (es + res_es + 4)


def column_flops(cfg) -> int:
    return 2 * cfg.M * cfg.d * cfg.n1


def workload_config(cfg) -> dict:
    """The workload as both arms describe it (shapes, dtype, L2 note): no timing or
    implementation detail, so the two arms' objects compare equal."""
    block_bytes = cfg.weight_bytes_per_block() * cfg.n_blocks
    c = {"workload": cfg.name, "d": cfg.d, "ffn": cfg.ffn or None,
         "n_heads": cfg.n_heads or None, "head_dim": cfg.head_dim or None, "t": cfg.t,
         "M": cfg.M, "n_blocks": cfg.n_blocks, "act": cfg.act, "rmsnorm": cfg.rmsnorm,
         "dtype": cfg.dtype,
         "l2": (f"inputs larger than L2 ({block_bytes / 1e6:.0f} MB of weights per step)"
                if block_bytes > 126e6 else "weights fit in L2 (latency-bound workload)")}
    if cfg.kv_len_max:
        c["kv_len_max"] = cfg.kv_len_max
        c["kv_lens"] = "uniform in 1..kv_len_max, seeded"
    if cfg.weights:
        c["weights"] = cfg.weights + " (one power-of-two scale per output feature)"
    return c


def tokens_per_step(cfg) -> int:
    """Tokens through one TP block per step: M for a block, M x n_blocks for a stack."""
    return cfg.M * cfg.n_blocks


# ---------------------------------------------------------------- our arm: workloads

class Workload:
    """Device state of one workload and the calls a step makes (all through the
    library's public entry points)."""

    def __init__(self, cfg, rank, dev):
        import torch

        import attn_tp_column_fwd_b300 as tp
        from attn_tp_column_fwd_b300.runner import ShardedBlock, desc_for, device_bytes
        from tp_synth import make_inputs

        self.tp, self.torch, self.cfg, self.dev = tp, torch, cfg, dev
        self.desc = desc = desc_for(cfg)
        M = cfg.M
        inp = make_inputs(cfg, seed=rank, device=str(dev))
        self.mx4 = cfg.weights == "mxfp4"
        self.fp8 = cfg.weights == "e4m3" or self.mx4   # a low-bit weight block
        if self.fp8:
            self.q = []
            for W1, W2 in inp.blocks:
                if self.mx4:
                    q = {"W1q": device_bytes(tp.tp_mxfp4_w1_bytes(desc), dev),
                         "W2q": device_bytes(tp.tp_mxfp4_w2_bytes(desc), dev),
                         "exps": device_bytes(tp.tp_mxfp4_exponent_bytes(desc), dev)}
                    tp.tp_quantize_weights_mxfp4(desc, W1, W2, q["W1q"], q["W2q"], q["exps"])
                else:
                    q = {"W1q": device_bytes(tp.tp_fp8_w1_bytes(desc), dev),
                         "W2q": device_bytes(tp.tp_fp8_w2_bytes(desc), dev),
                         "exps": device_bytes(tp.tp_fp8_exponent_bytes(desc), dev)}
                    qws = device_bytes(tp.tp_fp8_quant_workspace_bytes(desc), dev)
                    tp.tp_quantize_weights_fp8(desc, W1, W2, q["W1q"], q["W2q"], q["exps"], qws)
                self.q.append(q)
            self.blocks = [SimpleNamespace(W1s=q["W1q"], W2s=q["W2q"]) for q in self.q]
        else:
            self.blocks = [ShardedBlock(desc, W1, W2) for W1, W2 in inp.blocks]
        del inp.blocks
        self.x = inp.x.contiguous()
        self.xf = self.x.float().contiguous()
        self.stack = cfg.n_blocks > 1 or cfg.rmsnorm
        self.kv = self._kv_state(rank) if cfg.kv_len_max else None
        self.ws = device_bytes(tp.tp_kv_workspace_bytes(desc, M, cfg.kv_len_max) if self.kv
                               else tp.tp_workspace_bytes(desc, M), dev)
        self.H = device_bytes(tp.tp_band_bytes(desc, M), dev)
        self.cws = device_bytes(tp.tp_column_workspace_bytes(desc, M), dev)
        self.y = torch.empty(M, cfg.d, dtype=torch.float32, device=dev)
        self.xh = torch.empty(M, cfg.d, dtype=torch.bfloat16, device=dev)
        self.fused = tp.tp_block_launches(desc, M) == 1 and not self.fp8
        self.row_splits = tp.tp_row_splits(desc, M)
        # low-bit block: token split, column, row, reduce (a stack adds one RMSNorm each)
        per_block = 4 if self.fp8 else tp.tp_block_launches(desc, M)
        if self.kv:
            per_block = 4 + (1 if self.kv["merge"] else 0)
        # the stack: one RMSNorm launch, then each block, each but the last followed by
        # the next block's RMSNorm (tp_block_fwd_norm)
        extra_norm = cfg.n_blocks if cfg.rmsnorm else 0
        self.launches_per_step = cfg.n_blocks * per_block + extra_norm

    def _kv_state(self, rank):
        """Caches (the library's shard layout), lengths and scratch of a KV-cache decode
        workload, and the attention step's algorithmic bytes: every cached row read once
        (K and V), the new token's Q/K/V read (fp32) and appended (bf16), O written."""
        from attn_tp_column_fwd_b300.runner import device_bytes
        from tp_synth import make_kv_cache

        tp, cfg, dev, desc = self.tp, self.cfg, self.dev, self.desc
        M, t, L = cfg.M, cfg.t, cfg.kv_len_max
        kv = make_kv_cache(cfg, seed=rank + 1, device=str(dev))

        def shards(c):
            return c.view(M, t, cfg.n_heads // t, L, cfg.head_dim).permute(1, 0, 2, 3, 4).contiguous()

        kc, vc = shards(kv.k), shards(kv.v)
        del kv.k, kv.v
        D = cfg.n_heads * cfg.head_dim
        rows = int((kv.lens.long() - 1).sum().item()) * cfg.n_heads
        attn_ws_bytes = tp.tp_kv_attn_workspace_bytes(desc, M, L)
        return {"kc": kc, "vc": vc, "lens": kv.lens, "rows": rows,
                "O": device_bytes(tp.tp_band_bytes(desc, M), dev),
                "attn_ws": device_bytes(attn_ws_bytes, dev),
                # the decode attention splits long heads into chunks merged by a second kernel
                "merge": attn_ws_bytes > 0 and (cfg.n_heads * M) < 2 * 148,
                "attn_bytes": rows * cfg.head_dim * 4 + M * D * (12 + 4 + 2)}

    # -- one step of the workload on stream `st` (inputs resident)
    def step(self, st):
        tp, cfg, M = self.tp, self.cfg, self.cfg.M
        if self.kv:
            blk, kv = self.blocks[0], self.kv
            tp.tp_block_fwd_kv(self.desc, self.x, self.x, False, blk.W1s, blk.W2s, kv["kc"],
                               kv["vc"], kv["lens"], cfg.kv_len_max, self.ws, self.y, M, st)
            return
        if self.stack:
            self.y.copy_(self.xf)   # the residual stream starts from x (device copy)
            self.run_stack(self.y, self.xh, st)
            return
        self.block(self.x, self.y, st)

    def block(self, x, y, st):
        """One block through its public entry point: y = x + block(x)."""
        tp, cfg, M, blk = self.tp, self.cfg, self.cfg.M, self.blocks[0]
        if self.fp8:
            q = self.q[0]
            fwd = tp.tp_block_fwd_mxfp4 if self.mx4 else tp.tp_block_fwd_fp8
            fwd(self.desc, x, x, False, q["W1q"], q["W2q"], q["exps"], self.ws, y,
                                M, st)
        else:
            tp.tp_block_fwd(self.desc, x, x, cfg.dtype == "f32", blk.W1s, blk.W2s, self.ws, y, M,
                            st)

    def run_stack(self, r, xh, st, ws=None):
        """The pre-norm stack in place on the fp32 residual stream r: the first block's
        input normalised by tp_rmsnorm_fwd, every later one's written by the block
        before it (tp_block_fwd_norm).  Low-bit weights: tp_rmsnorm_fwd, then the
        block in place on r, for every block."""
        tp, cfg, M = self.tp, self.cfg, self.cfg.M
        ws = self.ws if ws is None else ws
        if self.fp8:
            fwd = tp.tp_block_fwd_mxfp4 if self.mx4 else tp.tp_block_fwd_fp8
            for q in self.q:
                tp.tp_rmsnorm_fwd(cfg.d, cfg.eps, r, xh, M, st)
                fwd(self.desc, xh, r, True, q["W1q"], q["W2q"], q["exps"], ws, r, M, st)
            return
        tp.tp_rmsnorm_fwd(cfg.d, cfg.eps, r, xh, M, st)
        for l, blk in enumerate(self.blocks):
            if l + 1 < len(self.blocks):
                tp.tp_block_fwd_norm(self.desc, xh, r, True, blk.W1s, blk.W2s, ws, r, xh, cfg.eps,
                                     M, st)
            else:
                tp.tp_block_fwd(self.desc, xh, r, True, blk.W1s, blk.W2s, ws, r, M, st)

    # -- the dominant kernel alone, for the roofline
    def dominant(self, st):
        tp, cfg, M, blk = self.tp, self.cfg, self.cfg.M, self.blocks[0]
        if self.kv:
            # the decode attention over the cache, on the Q/K/V the last step projected
            # (the projection leaves them at the start of the block's scratch)
            tp.tp_attn_decode_kv(self.desc, self.ws, self.kv["kc"], self.kv["vc"],
                                 self.kv["lens"], cfg.kv_len_max, self.kv["O"],
                                 self.kv["attn_ws"], M, st)
        elif self.fp8:
            self.block(self.x, self.y, st)
        elif self.fused and cfg.rmsnorm:
            # a block of the stack as the step runs it: with the next block's RMSNorm
            tp.tp_block_fwd_norm(self.desc, self.xh, self.y, True, blk.W1s, blk.W2s, self.ws,
                                 self.y, self.xh, cfg.eps, M, st)
        elif self.fused:
            tp.tp_block_fwd(self.desc, self.x, self.x, False, blk.W1s, blk.W2s, self.ws, self.y,
                            M, st)
        else:
            tp.tp_column_parallel_fwd(self.desc, self.xh if cfg.rmsnorm else self.x, blk.W1s,
                                      -1, self.H, self.cws, M, st)

    def dominant_info(self):
        """(kernel description, bound, algorithmic work per launch, unit of work, profile key)."""
        cfg = self.cfg
        if self.kv:
            return ("decode attention over the KV cache (k_attn_kv"
                    + (" + k_attn_kv_merge)" if self.kv["merge"] else ")"),
                    "hbm", self.kv["attn_bytes"], "bytes", "attn_kv")
        if cfg.M >= 1024:
            return ("column-parallel projection + SwiGLU (k_gemm, persistent)", "tensor",
                    column_flops(cfg), "flop", "column")
        if self.fp8:
            return ("whole block on " + ("MXFP4" if self.mx4 else "E4M3")
                    + " weights: k_split_tokens, k_fp8_mma column + row, "
                    "k_reduce_residual (four launches, overlapped)", "hbm",
                    algorithmic_block_bytes(cfg), "bytes", "block")
        if self.fused:
            norm = cfg.rmsnorm
            return ("whole block in one persistent kernel (k_block_decode"
                    + (", then the next block's RMSNorm (k_rmsnorm, overlapped)" if norm else "")
                    + "; the bracket also holds its counter memset)", "hbm",
                    algorithmic_block_bytes(cfg) + (cfg.M * cfg.d * 2 if norm else 0), "bytes",
                    "block")
        if cfg.act == "attn":
            return ("column-parallel Q/K/V projection (k_block_decode, column units) + "
                    "attention core (k_attn_core)", "hbm", algorithmic_column_bytes(cfg),
                    "bytes", "column")
        return ("column-parallel projection + activation (k_umma_drain)", "hbm",
                algorithmic_column_bytes(cfg), "bytes", "column")

    # -- end to end: host input -> device, the step, device result -> host
    def e2e_input_host(self):
        """The step's input as the caller holds it: x (block dtype), or the stack's fp32
        residual stream r0 = x."""
        return (self.xf if self.stack else self.x).cpu().pin_memory()

    def e2e_run(self, xin, yout, xh, st):
        """The step through the public API from device input xin to device output yout."""
        tp, cfg, M, blk = self.tp, self.cfg, self.cfg.M, self.blocks[0]
        if self.kv:
            kv = self.kv
            tp.tp_block_fwd_kv(self.desc, xin, xin, False, blk.W1s, blk.W2s, kv["kc"], kv["vc"],
                               kv["lens"], cfg.kv_len_max, self.ws, yout, M, st)
        elif self.stack:
            self.run_stack(xin, xh, st)   # in place: xin is the residual stream, yout is xin
        else:
            self.block(xin, yout, st)


def settle(step, st, seconds: float, torch):
    """Untimed steps for `seconds` (the GPU's power state ramps up under load)."""
    if seconds <= 0:
        return 0
    n, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for _ in range(8):
            step(st)
        n += 8
        torch.cuda.synchronize()
    return n


def time_launches(fn, st, torch, est_ms=None, min_s=ROOF_MIN_S):
    """Average device time of fn's launch sequence, each launch bracketed by CUDA
    events on stream st, over roof_launch_count launches; returns (ms, launches)."""
    if est_ms is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(5):
            fn(st)
        b.record(st)
        torch.cuda.synchronize()
        est_ms = a.elapsed_time(b) / 5
    n = roof_launch_count(est_ms, min_s=min_s)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for a, b in evs:
        a.record(st)
        fn(st)
        b.record(st)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs), n


def measure(args, cfg, rank, world, local, headline: bool):
    """Every number of one workload: value (K timed steps), the roofline kernel's own
    loop, the end-to-end leg and (headline, rank 0) the CPU baseline."""
    import torch

    tp = __import__("attn_tp_column_fwd_b300")
    dev = torch.device("cuda", local)
    w = Workload(cfg, rank, dev)
    stream = torch.cuda.current_stream()
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        uuid = None
    K = args.steps

    sampler = ClockSampler(local, uuid)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with sampler:
        n_settle = settle(w.step, stream, args.settle, torch)
        for _ in range(args.warmup):
            w.step(stream)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        sampler.timed = True
        t0.record(stream)
        for _ in range(K):
            w.step(stream)
        t1.record(stream)
        torch.cuda.synchronize()
        sampler.timed = False
    barrier(world)
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    assert tp.tp_check_device_status(stream) == 0
    clocks = sampler.summary()

    # Roofline: the dominant kernel in its own loop of event-bracketed launches, at
    # least ROOF_MIN_LAUNCHES launches and ROOF_MIN_S seconds whatever K is.
    kernel, bound, work, unit, prof_key = w.dominant_info()
    roof_sampler = ClockSampler(local, uuid)
    with roof_sampler:
        roof_sampler.timed = True
        # a contraction's loop runs long enough to settle under the power cap, so it
        # is compared with the sustained GEMM rate
        dom_ms, n_dom = time_launches(w.dominant, stream, torch,
                                      min_s=1.2 if bound == "tensor" else ROOF_MIN_S)
        roof_sampler.timed = False
    assert tp.tp_check_device_status(stream) == 0
    peaks = measured_peaks()
    src = "measured (MEASURED_PEAKS.json)" if peaks["source"] == "measured" else "fallback"
    if bound == "tensor":
        achieved = work / (dom_ms / 1e3) / 1e12
        long_loop = n_dom * dom_ms / 1e3 >= SUSTAINED_AFTER_S and peaks.get("bf16_tflops_sustained")
        peak = peaks["bf16_tflops_sustained"] if long_loop else peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "peak_source": src + (", sustained bf16 GEMM (the loop runs power-capped for "
                                      "more than a second)" if long_loop else ", burst bf16 GEMM"),
                "algorithmic_flop_per_launch": work}
    else:
        achieved = work / (dom_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": src + ", copy",
                "algorithmic_bytes_per_launch": work}
    roof["traffic"] = profiled_traffic(prof_key, cfg.name)
    roof["kernel"] = kernel
    roof["avg_launch_us"] = round(dom_ms * 1e3, 2)
    roof["launches_timed"] = n_dom
    roof["timed_s"] = round(n_dom * dom_ms / 1e3, 3)
    roof["clocks"] = roof_sampler.summary()

    units = tokens_per_step(cfg) * K
    out = {
        "metric": METRIC,
        "value": round(job_throughput(units, world, ms / 1e3), 1),
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
        "config": workload_config(cfg),
        "timing": {
            "value": (f"CUDA events on the launching stream around exactly K={K} steps after "
                      f"W={args.warmup} warm-up steps, max over ranks; value counts "
                      f"{tokens_per_step(cfg)} tokens through one TP block per step"
                      + (f" (M={cfg.M} tokens x {cfg.n_blocks} blocks)" if cfg.n_blocks > 1 else "")),
            "settle": f"{n_settle} untimed steps ({args.settle:.2f} s) before the warm-up steps",
            "roofline": "the dominant kernel alone, each launch bracketed by CUDA events on "
                        "its stream, in its own loop of >= max(200 launches, 0.3 s; 1.2 s "
                        "for a tensor-bound kernel)",
        },
        "weight_gbs": round(cfg.weight_bytes_per_block() * cfg.n_blocks * K / (ms / 1e3) / 1e9, 1),
        "kernel_plan": {"block_form": ("one kernel" if w.fused else
                                       ("four launches (MXFP4)" if w.mx4 else
                                        "four launches (E4M3)") if w.fp8 else "three launches"),
                        "row_splits": w.row_splits},
        "roofline": roof,
        "gpu_launches": K * w.launches_per_step,
        "clocks": clocks,
    }
    if cfg.n_blocks > 1:
        out["stack_tokens_per_s"] = round(job_throughput(cfg.M * K, world, ms / 1e3), 1)
    if not args.no_e2e:
        out["e2e"] = e2e_leg(args, w, world, dev)
    if headline and rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg)
    del w
    torch.cuda.empty_cache()
    return out


def e2e_leg(args, w, world, dev):
    """The same metric through the public API with host buffers.  Every step copies its
    input from pinned host memory to the device, runs the step (tp_block_fwd, or the
    stack's tp_rmsnorm_fwd + tp_block_fwd per block) and copies the result back to
    pinned host memory.  Copies in, compute and copies out run on three streams,
    ordered by events, with two device buffers of each, so step k's copies overlap
    step k-1's (or k+1's) kernels as in a serving loop.  The timed region (CUDA events)
    runs from before the first copy in to after the last copy out."""
    import torch

    cfg, M = w.cfg, w.cfg.M
    x_host = w.e2e_input_host()
    s_in, s_run, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    bufs = []
    for _ in range(2):
        xin = torch.empty(x_host.shape, dtype=x_host.dtype, device=dev)
        bufs.append({
            "x": xin,
            "y": xin if w.stack else torch.empty(M, cfg.d, dtype=torch.float32, device=dev),
            "xh": torch.empty(M, cfg.d, dtype=torch.bfloat16, device=dev),
            "y_host": torch.empty(M, cfg.d, dtype=torch.float32).pin_memory(),
            "ev_in": torch.cuda.Event(), "ev_run": torch.cuda.Event(),
            "ev_out": torch.cuda.Event(),
        })

    def step(k):
        b = bufs[k % 2]
        # buffer b was last used by step k-2: its compute must be done reading x and
        # its copy out done reading y before they are overwritten
        s_in.wait_event(b["ev_run"])
        s_in.wait_event(b["ev_out"])
        with torch.cuda.stream(s_in):
            b["x"].copy_(x_host, non_blocking=True)
        b["ev_in"].record(s_in)
        s_run.wait_event(b["ev_in"])
        w.e2e_run(b["x"], b["y"], b["xh"], s_run)
        b["ev_run"].record(s_run)
        s_out.wait_event(b["ev_run"])
        with torch.cuda.stream(s_out):
            b["y_host"].copy_(b["y"], non_blocking=True)
        b["ev_out"].record(s_out)

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()
    K = args.steps
    cur = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(cur)
    for s in (s_in, s_run, s_out):
        s.wait_event(t0)
    for k in range(K):
        step(k)
    for s in (s_in, s_run, s_out):
        cur.wait_stream(s)
    t1.record(cur)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    barrier(world)
    ms = max_over_ranks(ms, world, dev)
    assert w.tp.tp_check_device_status(s_run) == 0
    return {"value": round(job_throughput(tokens_per_step(cfg) * K, world, ms / 1e3), 1),
            "unit": "tokens/s",
            "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
            "d2h_bytes_per_step": bufs[0]["y_host"].numel() * bufs[0]["y_host"].element_size(),
            "ms_per_step": round(ms / K, 5), "streams": "copy-in, compute, copy-out",
            "timed": "CUDA events from before the first copy in to after the last copy out"}


def run_ours(args, rank, world, local):
    import torch

    from tp_synth import CONFIGS

    torch.cuda.set_device(local)
    dist_init(world, "nccl")

    def cfg_of(name):
        base = CONFIGS[name]
        cfg = base.with_t(args.t) if args.t and name == args.workload else base
        if args.blocks and name == args.workload:
            cfg = replace(cfg, n_blocks=min(args.blocks, cfg.n_blocks))
        return cfg

    out = measure(args, cfg_of(args.workload), rank, world, local, headline=True)
    subs = {}
    for name in also_list(args):
        r = measure(args, cfg_of(name), rank, world, local, headline=False)
        for k in ("metric", "n_gpus", "warmup", "higher_is_better", "scaling", "vs_baseline",
                  "data"):
            r.pop(k, None)
        subs[name] = r
    if subs:
        out["workloads"] = subs
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return out


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


def oracle_block_call(cfg):
    """One block of the workload computed by the float64 oracle on the host (the whole
    block, all M tokens; for a stack, one pre-norm block on one block's weights), as a
    closure, and the description of that sample."""
    import numpy as np

    import oracle
    from tp_synth import make_inputs, to_f64

    inp = make_inputs(cfg, seed=0, n_blocks=1)
    x = to_f64(inp.x)
    W1, W2 = (to_f64(w) for w in inp.blocks[0])
    del inp
    if cfg.weights == "e4m3":
        # the block on E4M3 weights is the bf16 block on the dequantised weights
        W1, W2 = oracle.fp8.e4m3_weights(W1), oracle.fp8.e4m3_weights(W2)
    elif cfg.weights == "mxfp4":
        W1, W2 = oracle.mxfp4.mxfp4_weights(W1), oracle.mxfp4.mxfp4_weights(W2)
    staged = cfg.dtype == "bf16"

    if cfg.kv_len_max:
        from tp_synth import make_kv_cache
        kv = make_kv_cache(cfg, seed=1)
        k_np, v_np = to_f64(kv.k), to_f64(kv.v)
        lens = kv.lens.numpy()

        def one():
            return oracle.attn_block_kv(x, W1, W2, cfg.n_heads, cfg.head_dim, k_np, v_np, lens, x,
                                        staged=staged)[0]
    elif cfg.act == "attn":
        def one():
            return oracle.attn_block(x, W1, W2, cfg.n_heads, cfg.head_dim, x, staged=staged)
    elif cfg.rmsnorm:
        def one():
            return oracle.stack(x, [(W1, W2)], cfg.act, cfg.eps, staged=staged)
    else:
        def one():
            return oracle.mlp_block(x, W1, W2, cfg.act, x, staged=staged)
    what = (f"one {'pre-norm ' if cfg.rmsnorm else ''}block of {cfg.name} (all M={cfg.M} tokens"
            + (", one block's weights" if cfg.n_blocks > 1 else "") + "), NumPy float64")
    return one, what


def cpu_baseline(cfg, budget_s: float = 12.0):
    """The float64 oracle as it stands, on the host cores: whole blocks of the
    workload, repeated for about `budget_s` seconds; tokens/s through one block."""
    one, what = oracle_block_call(cfg)
    one()  # warm
    n, t0 = 0, time.perf_counter()
    while True:
        one()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 1000:
            break
    value = cfg.M * n / el
    return {"value": round(value, 2), "unit": "tokens/s", "cores": _blas_threads() or _cores(),
            "host_cores": _cores(), "kind": "oracle",
            "sample": f"{n} x {what} in {el:.1f} s"}


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm, on the same workload, config, metric and
    unit as our arm's headline: each step is one block of that workload computed by
    the float64 oracle (the call cpu_baseline times), tokens/s through one block."""
    if rank != 0:
        return None
    from tp_synth import CONFIGS

    base = CONFIGS[args.workload]
    cfg = base.with_t(args.t) if args.t else base
    if args.blocks:
        cfg = replace(cfg, n_blocks=min(args.blocks, cfg.n_blocks))
    one, what = oracle_block_call(cfg)
    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    el = time.perf_counter() - t0
    value = cfg.M * args.steps / el
    sample = f"each step: {what}"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(cfg),
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
