#!/usr/bin/env python3
"""Benchmark of the fused residual-add + RMSNorm + quantisation path on GB300.

One step = one launch of the fused kernel over the whole batch (all steps of
the path: residual add, residual write-back, RMSNorm, scale, quantise, pack).
Default workload: the DeepSeek-V3-shaped layer, 8192 tokens x 7168 hidden
bf16 with 1 % outlier channels, residual add on, FP8 E4M3 per-group scales
(group 128, row-major) -- the largest configuration of the path that fits one
GPU.

Prints ONE JSON line (rank 0).  ``value`` is algorithmic HBM GB/s (bytes the
op must move / device time), whole job over all ranks.  Inputs are resident in
HBM before the timed region; consecutive steps rotate over buffer sets whose
total size is more than 4x the L2 cache, so no step reads the previous step's
data from L2.  ``e2e`` is the same metric with every step's inputs copied from
pinned host memory and its outputs read back inside the timed region (copies
in, launches and copies out pipelined on three streams).  ``parity`` compares
the outputs of a timed step with the oracle over every row (computed in the
CPU-baseline leg, after the timed region).  ``clocks`` are nvidia-smi samples
over a window of continuous replays of the same launches that brackets the
timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused add-RMSNorm+quant HBM GB/s and tokens/s on 1 GB300 vs ~8 TB/s peak"
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0
VARIANT = "auto"       # kernel variant for every launch (set by --variant)


# --------------------------------------------------------------------------- bytes
def algorithmic_bytes(mode: str, n: int, H: int, es: int, residual: bool) -> int:
    """Bytes the op must move for one launch over n rows of width H."""
    per_tok = H * es                              # x
    if residual:
        per_tok += 2 * H * es                     # residual in, residual_out
    per_tok += H // 2 if mode == "nvfp4" else H   # codes
    if mode == "fp8_per_token":
        per_tok += 4
    elif mode.startswith("fp8_group"):
        per_tok += 4 * H // (128 if "128" in mode else 64)
    elif mode == "nvfp4":
        per_tok += H // 16
    fixed = H * es + (4 if mode in ("fp8_static", "nvfp4") else 0)   # weight, scale_in
    return n * per_tok + fixed


def max_over_ranks(ms: float, dist, device: str) -> float:
    """The slowest rank's time per step (every rank gets it); `dist` is
    torch.distributed (any backend) or None for a single process."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rates(bytes_per_rank_step: int, tokens_per_rank_step: int, world: int, ms: float):
    """Whole-job GB/s and tokens/s: every rank processes its own batch (the
    rows are independent, so ranks shard by tokens with no collective on the
    data path) and the job takes as long as its slowest rank."""
    sec = ms / 1e3
    return bytes_per_rank_step * world / sec / 1e9, tokens_per_rank_step * world / sec


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (host timestamped) of SM clock and throttle reasons."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int = 0, period_ms: int = 20):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        note = "samples inside the timed region"
        if not inside and self.samples:
            mid = (t0 + t1) / 2
            inside = [min(self.samples, key=lambda s: abs(s[0] - mid))[1]]
            note = "timed region shorter than the sampling period: nearest sample"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        reasons = set()
        for p in inside:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                "sw_power_cap"), p[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(inside[0][1]), "reasons": sorted(reasons),
                "samples": len(inside), "note": note}


# --------------------------------------------------------------------------- helpers
def measured_peak() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_digest() -> str:
    from residual_add_rmsnorm_rmsq_gb300 import _build
    return _build.source_digest()


def profiled_traffic(kernel_name: str, digest: str):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
    except (OSError, ValueError):
        return None
    e = d.get(kernel_name)
    if not e or e.get("source_digest") != digest:
        return None
    return e.get("dram_bytes_per_launch")


def launch_shape(wl, mode: str, residual: bool, torch) -> dict:
    """The launch the library makes for this workload on this device
    (rmsq_query_launch): kernel variant, chunks per thread, ring stages, CTAs,
    threads per CTA."""
    import residual_add_rmsnorm_rmsq_gb300 as rq
    qmode = "nvfp4" if mode == "nvfp4_dynamic" else mode
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
    return rq.query_launch(qmode, wl.n_tokens, wl.hidden, residual, tdt, VARIANT)


def kernel_name(wl, mode: str, residual: bool, torch) -> str:
    """Name (as ncu prints it, without the namespace) of the row kernel the
    library launches for this workload (for the data-derived NVFP4 scale, its
    first kernel), from the library's own launch choice."""
    import residual_add_rmsnorm_rmsq_gb300 as rq
    shape = launch_shape(wl, mode, residual, torch)
    e = "Bf16T" if wl.dtype == "bf16" else "Fp16T"
    m = 7 if mode == "nvfp4_dynamic" else rq.MODES[mode]
    kind = "pipe_entry" if shape["pipelined"] else "rows_kernel"
    return f"{kind}<{e}, {m}, {int(residual)}, {shape['chunks_per_thread']}>"


def workload_spec(name: str):
    import rmsq_inputs as ri
    specs = {
        "llama_fp8_per_token": (lambda: ri.llama(4096, True), "fp8_per_token"),
        "llama_fp8_per_token_nores": (lambda: ri.llama(4096, False), "fp8_per_token"),
        "llama_fp8_static": (lambda: ri.llama(4096, True), "fp8_static"),
        "dsv3_fp8_group128_row": (lambda: ri.dsv3(8192), "fp8_group128_row"),
        "dsv3_fp8_group128_col": (lambda: ri.dsv3(8192), "fp8_group128_col"),
        "dsv3_fp8_group64_row": (lambda: ri.dsv3(8192), "fp8_group64_row"),
        "dsv3_fp8_group64_col": (lambda: ri.dsv3(8192), "fp8_group64_col"),
        "qwen_nvfp4_4096": (lambda: ri.qwen_nvfp4(4096), "nvfp4"),
        "qwen_nvfp4_16384": (lambda: ri.qwen_nvfp4(16384), "nvfp4"),
        "qwen_nvfp4_dynamic_4096": (lambda: ri.qwen_nvfp4(4096), "nvfp4_dynamic"),
        "qwen_nvfp4_dynamic_16384": (lambda: ri.qwen_nvfp4(16384), "nvfp4_dynamic"),
    }
    return specs[name]


def gpu_scale_in(torch, rq, wl, mode, x, r, w):
    """scale_in for the timed launches: the workload's static scale, or for
    NVFP4 gs = 2688 / amax(y) over the batch, computed on the device by the
    library's data-derived-scale entry point (outside the timed region)."""
    if mode == "fp8_static":
        return torch.tensor([wl.static_scale or 0.1], dtype=torch.float32, device="cuda")
    if mode != "nvfp4":
        return None
    _, _, gs, _ = rq.fused_add_rmsnorm_nvfp4_dynamic(x, r, w, wl.eps)
    torch.cuda.synchronize()
    return gs


class Buffers:
    """Rotating device buffer sets for one workload and mode."""

    def __init__(self, torch, rq, wl, mode, min_total_bytes, max_sets=None):
        tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
        n, H = wl.n_tokens, wl.hidden
        self.rq, self.wl, self.mode = rq, wl, mode
        self.dynamic = mode == "nvfp4_dynamic"
        qmode = "nvfp4" if self.dynamic else mode
        self.es = 2
        self.res = wl.residual is not None
        # the data-derived global scale is one more 4-byte output; the second
        # pass's re-read of h is not counted (it is not required by the op)
        self.bytes = algorithmic_bytes(qmode, n, H, 2, self.res) + (4 if self.dynamic else 0)
        self.sets = max(2, math.ceil(min_total_bytes / self.bytes))
        if max_sets is not None:
            self.sets = min(self.sets, max_sets)
        x0 = torch.from_numpy(wl.x.view(np.int16)).view(tdt).cuda()
        r0 = None if not self.res else torch.from_numpy(wl.residual.view(np.int16)).view(tdt).cuda()
        self.w = torch.from_numpy(wl.weight.view(np.int16)).view(tdt).cuda()
        self.scale_in = None if self.dynamic else gpu_scale_in(torch, rq, wl, mode, x0, r0, self.w)
        self.x, self.r, self.ro, self.q, self.sc, self.gs, self.ws = [], [], [], [], [], [], []
        for i in range(self.sets):
            self.x.append(x0 if i == 0 else x0.clone())
            if self.res:
                self.r.append(r0 if i == 0 else r0.clone())
                self.ro.append(torch.empty_like(r0))
            else:
                self.r.append(None)
                self.ro.append(None)
            self.q.append(torch.empty(n, H // 2 if qmode == "nvfp4" else H, dtype=torch.uint8, device="cuda"))
            self.sc.append(rq.scales_like(qmode, n, H, "cuda"))
            if self.dynamic:
                self.gs.append(torch.empty(1, dtype=torch.float32, device="cuda"))
                self.ws.append(torch.empty(rq.nvfp4_dynamic_workspace_bytes(n), dtype=torch.uint8,
                                           device="cuda"))

    def launch(self, k, stream):
        """One call of the public API on buffer set k."""
        if self.dynamic:
            self.rq.fused_add_rmsnorm_nvfp4_dynamic(
                self.x[k], self.r[k], self.w, self.wl.eps, out_q=self.q[k], out_scales=self.sc[k],
                out_global_scale=self.gs[k], residual_out=self.ro[k], workspace=self.ws[k],
                stream=stream, variant=VARIANT)
        else:
            self.rq.fused_add_rmsnorm_quant(
                self.x[k], self.r[k], self.w, self.wl.eps, self.mode, self.scale_in,
                out_q=self.q[k], out_scales=self.sc[k], residual_out=self.ro[k], stream=stream,
                variant=VARIANT)


def act_algorithmic_bytes(mode: str, n: int, d: int, es: int) -> int:
    """Bytes the SiLU+Mul + quantisation op must move: gate_up in, codes and
    scales out, scale_in."""
    per_tok = 2 * d * es + (d // 2 if mode == "nvfp4" else d)
    if mode == "fp8_per_token":
        per_tok += 4
    elif mode.startswith("fp8_group"):
        per_tok += 4 * d // (128 if "128" in mode else 64)
    elif mode == "nvfp4":
        per_tok += d // 16
    return n * per_tok + (4 if mode in ("fp8_static", "nvfp4") else 0)


class ActBuffers:
    """Rotating device buffer sets for one SiLU+Mul + quantisation workload."""

    def __init__(self, torch, rq, wl, mode, min_total_bytes):
        tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
        n, d = wl.n_tokens, wl.d
        self.rq, self.mode = rq, mode
        self.bytes = act_algorithmic_bytes(mode, n, d, 2)
        self.sets = max(2, math.ceil(min_total_bytes / self.bytes))
        g0 = torch.from_numpy(wl.gate_up.view(np.int16)).view(tdt).cuda()
        if mode == "fp8_static":
            self.scale_in = torch.tensor([wl.static_scale or 0.05], dtype=torch.float32, device="cuda")
        elif mode == "nvfp4":
            # the workload's rule, gs = 2688 / amax of the activations over the
            # batch: the library's own a = silu(g) * u (its elementwise debug
            # entry), its amax and one fp32 division, outside the timed region
            a = rq.debug_activation("silu_mul", g0[:, :d].float().contiguous(), g0[:, d:].float().contiguous())
            amax = a.abs().max().reshape(1)
            self.scale_in = torch.tensor([2688.0], dtype=torch.float32, device="cuda") / amax
            del a
        else:
            self.scale_in = None
        self.gu, self.q, self.sc = [], [], []
        for i in range(self.sets):
            self.gu.append(g0 if i == 0 else g0.clone())
            self.q.append(torch.empty(n, d // 2 if mode == "nvfp4" else d, dtype=torch.uint8, device="cuda"))
            self.sc.append(rq.scales_like(mode, n, d, "cuda"))
        torch.cuda.synchronize()

    def launch(self, k, stream):
        self.rq.silu_mul_quant(self.gu[k], self.mode, self.scale_in, out_q=self.q[k], out_scales=self.sc[k],
                               stream=stream)


class UnfusedBuffers:
    """Rotating buffer sets for the unfused two-op sequence (add + RMSNorm
    writing y in the activation type, then the quantisation of y): one step
    is both calls.  `bytes` counts what the two ops move, `fused_bytes` what
    the fused op moves for the same result shape."""

    def __init__(self, torch, rq, wl, mode, min_total_bytes):
        tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
        n, H = wl.n_tokens, wl.hidden
        self.rq, self.wl, self.mode = rq, wl, mode
        self.res = wl.residual is not None
        self.fused_bytes = algorithmic_bytes(mode, n, H, 2, self.res)
        self.bytes = self.fused_bytes + 2 * n * H * 2       # y written by the first op, read by the second
        self.sets = max(2, math.ceil(min_total_bytes / self.bytes))
        x0 = torch.from_numpy(wl.x.view(np.int16)).view(tdt).cuda()
        r0 = None if not self.res else torch.from_numpy(wl.residual.view(np.int16)).view(tdt).cuda()
        self.w = torch.from_numpy(wl.weight.view(np.int16)).view(tdt).cuda()
        self.scale_in = gpu_scale_in(torch, rq, wl, mode, x0, r0, self.w)
        self.x, self.r, self.ro, self.y, self.q, self.sc = [], [], [], [], [], []
        for i in range(self.sets):
            self.x.append(x0 if i == 0 else x0.clone())
            self.r.append(None if r0 is None else (r0 if i == 0 else r0.clone()))
            self.ro.append(None if r0 is None else torch.empty_like(r0))
            self.y.append(torch.empty_like(x0))
            self.q.append(torch.empty(n, H // 2 if mode == "nvfp4" else H, dtype=torch.uint8, device="cuda"))
            self.sc.append(rq.scales_like(mode, n, H, "cuda"))

    def launch(self, k, stream):
        self.rq.fused_add_rmsnorm(self.x[k], self.r[k], self.w, self.wl.eps, y_out=self.y[k],
                                  residual_out=self.ro[k], stream=stream)
        self.rq.quant(self.y[k], self.mode, self.scale_in, out_q=self.q[k], out_scales=self.sc[k], stream=stream)


class AllReduceBuffers:
    """Rotating buffer sets for all-reduce + residual add + RMSNorm + quant:
    the ranks' partial tensors are emulated as separate buffers of this
    device (the same loads a multi-GPU node issues to peer memory)."""

    def __init__(self, torch, rq, wl, mode, ranks, min_total_bytes, max_sets=None):
        tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
        n, H = wl.n_tokens, wl.hidden
        self.rq, self.wl, self.mode, self.ranks = rq, wl, mode, ranks
        # each rank's partial row read once, plus what the fused op moves besides x
        self.bytes = algorithmic_bytes(mode, n, H, 2, True) + (ranks - 1) * n * H * 2
        self.sets = max(2, math.ceil(min_total_bytes / self.bytes))
        if max_sets is not None:
            self.sets = min(self.sets, max_sets)
        x0 = torch.from_numpy(wl.x.view(np.int16)).view(tdt).cuda()
        r0 = torch.from_numpy(wl.residual.view(np.int16)).view(tdt).cuda()
        self.w = torch.from_numpy(wl.weight.view(np.int16)).view(tdt).cuda()
        self.scale_in = torch.tensor([0.05 if mode == "fp8_static" else 1000.0], dtype=torch.float32, device="cuda")
        self.parts, self.r, self.ro, self.q, self.sc = [], [], [], [], []
        for i in range(self.sets):
            self.parts.append([x0 * (0.5 + 0.25 * k) for k in range(ranks)])
            self.r.append(r0.clone())
            self.ro.append(torch.empty_like(r0))
            self.q.append(torch.empty(n, H // 2 if mode == "nvfp4" else H, dtype=torch.uint8, device="cuda"))
            self.sc.append(rq.scales_like(mode, n, H, "cuda"))

    def launch(self, k, stream):
        self.rq.allreduce_add_rmsnorm_quant(self.parts[k], self.r[k], self.w, self.wl.eps, self.mode, self.scale_in,
                                            out_q=self.q[k], out_scales=self.sc[k], residual_out=self.ro[k],
                                            stream=stream)


class QkBuffers:
    """Rotating buffer sets for QK-norm + RoPE (in place on qkv)."""

    def __init__(self, torch, rq, wl, min_total_bytes):
        tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
        n, D, nh = wl.n_tokens, wl.head_dim, wl.nq + wl.nkv
        self.rq, self.wl = rq, wl
        # q and k heads read and written, the position, the token's cos / sin row, the weights
        self.bytes = n * (nh * D * 2 * 2 + 8 + D * 4) + 2 * D * 2
        self.sets = max(2, math.ceil(min_total_bytes / self.bytes))
        q0 = torch.from_numpy(wl.qkv.view(np.int16)).view(tdt).cuda()
        self.qkv = [q0 if i == 0 else q0.clone() for i in range(self.sets)]
        self.pos = torch.from_numpy(wl.positions).cuda()
        self.cs = torch.from_numpy(wl.cos_sin).cuda()
        self.qw = torch.from_numpy(wl.q_weight.view(np.int16)).view(tdt).cuda()
        self.kw = torch.from_numpy(wl.k_weight.view(np.int16)).view(tdt).cuda()

    def launch(self, k, stream):
        w = self.wl
        self.rq.qk_norm_rope(self.qkv[k], self.pos, self.cs, self.qw, self.kw, w.eps, w.nq, w.nkv, w.head_dim,
                             w.neox, stream=stream, variant=VARIANT)


class Replayer:
    """The launches of a timed region as CUDA graphs: one graph of one launch
    per buffer set (in rotation order) replayed steps // sets times, plus a
    graph of the remaining launches, so the device runs the K kernels back to
    back instead of waiting on Python between them.  Every launch goes through
    the same public call.  Eager warm-up launches come first (they also fill
    the library's per-function caches before capture)."""

    def __init__(self, torch, bufs, steps, warmup, stream):
        self.torch, self.bufs, self.steps, self.stream = torch, bufs, steps, stream

        def capture(count):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                for i in range(count):
                    bufs.launch(i % bufs.sets, stream)
            return g

        with torch.cuda.stream(stream):
            for i in range(max(warmup, bufs.sets)):
                bufs.launch(i % bufs.sets, stream)
            torch.cuda.synchronize()
            self.reps, rem = divmod(steps, bufs.sets)
            self.g_full = capture(bufs.sets) if self.reps else None
            self.g_rem = capture(rem) if rem else None
            for g in (self.g_full, self.g_rem):          # one untimed replay of each graph
                if g is not None:
                    g.replay()
            torch.cuda.synchronize()

    def timed(self) -> float:
        """Mean device time per launch (ms) over exactly `steps` launches,
        CUDA events on the launching stream."""
        torch = self.torch
        with torch.cuda.stream(self.stream):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            for _ in range(self.reps):
                self.g_full.replay()
            if self.g_rem is not None:
                self.g_rem.replay()
            e1.record(self.stream)
            torch.cuda.synchronize()
        return e0.elapsed_time(e1) / self.steps

    def soak(self, seconds: float) -> int:
        """Untimed replays of the same launches for about `seconds` of wall
        time (the device kept as busy as in the timed region); returns the
        launches run."""
        torch = self.torch
        g = self.g_full or self.g_rem
        per = self.bufs.sets if self.g_full is not None else self.steps
        done, t0 = 0, time.time()
        with torch.cuda.stream(self.stream):
            while time.time() - t0 < seconds:
                for _ in range(16):
                    g.replay()
                done += 16 * per
                torch.cuda.synchronize()
        return done


def time_launches(torch, rq, wl, mode, bufs, steps, warmup, stream):
    """Mean device time per launch (ms) over exactly `steps` launches (see
    Replayer)."""
    return Replayer(torch, bufs, steps, warmup, stream).timed()


def e2e_measure(torch, rq, wl, mode, bufs, steps, stream):
    """Same op through the public API with host buffers: every step copies its
    inputs (x, residual) from pinned host memory to the device, launches, and
    copies its results (codes, scales, residual_out) back to pinned host
    memory, all inside the timed region.  The steps are pipelined the way a
    serving loop would run them: host-to-device copies on one stream, the
    launches on `stream`, device-to-host copies on a third, over two device
    buffer sets ordered by events, so that step k+1's inputs travel while
    step k's results come back (the link is full duplex)."""
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
    hx = torch.from_numpy(wl.x.view(np.int16)).view(tdt).pin_memory()
    hr = None if wl.residual is None else torch.from_numpy(wl.residual.view(np.int16)).view(tdt).pin_memory()
    hq = torch.empty(bufs.q[0].shape, dtype=torch.uint8).pin_memory()
    hs = None if bufs.sc[0] is None else torch.empty(bufs.sc[0].shape, dtype=bufs.sc[0].dtype).pin_memory()
    hro = None if hr is None else torch.empty_like(hr).pin_memory()
    h2d = hx.numel() * 2 + (0 if hr is None else hr.numel() * 2)
    d2h = hq.numel() + (0 if hs is None else hs.numel() * hs.element_size()) + \
        (0 if hro is None else hro.numel() * 2)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    nb = min(2, bufs.sets)
    in_free = [None] * nb    # launch that last read set b's inputs
    out_free = [None] * nb   # copy-out that last read set b's results

    def step(k):
        b = k % nb
        with torch.cuda.stream(s_in):
            if in_free[b] is not None:
                s_in.wait_event(in_free[b])
            bufs.x[b].copy_(hx, non_blocking=True)
            if hr is not None:
                bufs.r[b].copy_(hr, non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
        stream.wait_event(ev_in)
        if out_free[b] is not None:
            stream.wait_event(out_free[b])
        bufs.launch(b, stream)
        ev_k = torch.cuda.Event()
        ev_k.record(stream)
        in_free[b] = ev_k
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_k)
            hq.copy_(bufs.q[b], non_blocking=True)
            if hs is not None:
                hs.copy_(bufs.sc[b], non_blocking=True)
            if hro is not None:
                hro.copy_(bufs.ro[b], non_blocking=True)
            ev_o = torch.cuda.Event()
            ev_o.record(s_out)
        out_free[b] = ev_o

    for k in range(3):
        step(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)              # before the first copy-in: everything timed depends on it
    for k in range(steps):
        step(k)
    e1.record(s_out)             # after the last copy-out, which waits for everything before it
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return ms, h2d, d2h


def _oracle_scale_in(wl, mode, scale_in):
    return scale_in if scale_in is not None else (wl.static_scale if mode == "fp8_static" else 0.0)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(wl, mode, scale_in=None, budget_s: float = 20.0) -> dict:
    """The oracle as it stands, row-parallel over the process's cores, on a
    bounded prefix of the workload's rows; median of 3 runs.  Beside it, the
    same oracle on one thread over a prefix of 1/cores as many rows."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    scale = _oracle_scale_in(wl, mode, scale_in)
    rows = min(wl.n_tokens, 256)

    def run(rows, threads=cores):
        oracle.run(wl.x[:rows], None if wl.residual is None else wl.residual[:rows], wl.weight,
                   eps=wl.eps, mode=mode, scale_in=scale, dtype=wl.dtype, nthreads=threads)

    while True:
        t = time.perf_counter()
        run(rows)
        dt = time.perf_counter() - t
        if rows >= wl.n_tokens or dt * 3 * 4 > budget_s / 2:
            break
        rows = min(wl.n_tokens, rows * 4)
    times = []
    for _ in range(3):
        t = time.perf_counter()
        run(rows)
        times.append(time.perf_counter() - t)
    med = statistics.median(times)
    nbytes = algorithmic_bytes(mode, rows, wl.hidden, 2, wl.residual is not None)
    rows1 = max(1, rows // cores)
    times1 = []
    for _ in range(3):
        t = time.perf_counter()
        run(rows1, 1)
        times1.append(time.perf_counter() - t)
    med1 = statistics.median(times1)
    nbytes1 = algorithmic_bytes(mode, rows1, wl.hidden, 2, wl.residual is not None)
    return {"value": round(nbytes / med / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "tokens_per_s": round(rows / med, 1),
            "sample": f"first {rows} of {wl.n_tokens} rows, median of 3 runs, {cores} threads",
            "cpu": cpu_model(),
            "single_thread": {"value": round(nbytes1 / med1 / 1e9, 4), "unit": "GB/s",
                              "sample": f"first {rows1} rows, median of 3 runs, 1 thread"}}


def parity_vs_oracle(wl, mode, scale_in, got: dict) -> dict:
    """Part of the CPU-baseline leg, run after the timed region: the oracle on
    every row of the workload, compared element by element with the outputs
    of one timed step (`got`: host arrays q, scales, residual_out).  Codes:
    the number of elements that differ and the largest difference in code
    steps; scales and residual_out: whether they are identical bit for bit."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    want = oracle.run(wl.x, wl.residual, wl.weight, eps=wl.eps, mode=mode,
                      scale_in=_oracle_scale_in(wl, mode, scale_in), dtype=wl.dtype, nthreads=cores)
    if mode == "nvfp4":
        g = np.stack([got["q"] & 0xF, got["q"] >> 4], -1).astype(np.int32)
        w = np.stack([want["q"] & 0xF, want["q"] >> 4], -1).astype(np.int32)
        sg, sw, mg, mw = g >> 3, w >> 3, g & 7, w & 7
    else:
        g, w = got["q"].astype(np.int32), want["q"].astype(np.int32)
        sg, sw, mg, mw = g >> 7, w >> 7, g & 0x7F, w & 0x7F
    steps = np.where(sg == sw, np.abs(mg - mw), mg + mw)
    bad = int(np.count_nonzero(steps))
    out = {"elements": int(steps.size), "mismatches": bad, "fraction": bad / max(1, steps.size),
           "max_step": int(steps.max()) if steps.size else 0, "bar": "<= 1 step on <= 1e-4 of the codes"}
    if want["scales"] is not None:
        ws = want["scales"].reshape(-1).view(np.uint8)
        gs = got["scales"].reshape(-1).view(np.uint8)
        out["scales_bitexact"] = bool(np.array_equal(ws, gs))
    if want["residual_out"] is not None:
        out["residual_bitexact"] = bool(np.array_equal(want["residual_out"], got["residual_out"]))
    return out


def workload_config(name: str, wl, mode: str) -> dict:
    """The config object of the JSON line, the same in both arms."""
    return {"workload": name, "n_tokens": wl.n_tokens, "hidden": wl.hidden, "quant_mode": mode,
            "residual": wl.residual is not None, "eps": wl.eps, "act_dtype": wl.dtype,
            "l2": "inputs larger than L2: consecutive GPU steps rotate over buffer sets of > 4x L2"}


# --------------------------------------------------------------------------- arms
def run_reference(args, rank, world):
    """The oracle, timed on the host cores as the reference arm (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    mk, mode = workload_spec(args.workload)
    wl = mk()
    cores = len(os.sched_getaffinity(0))
    scale = wl.static_scale if mode == "fp8_static" else (1000.0 if mode == "nvfp4" else 0.0)
    # size the per-step sample so that warmup + steps fit in about a minute
    probe = 64
    t = time.perf_counter()
    oracle.run(wl.x[:probe], None if wl.residual is None else wl.residual[:probe], wl.weight,
               eps=wl.eps, mode=mode, scale_in=scale, dtype=wl.dtype, nthreads=cores)
    per_row = (time.perf_counter() - t) / probe
    rows = int(max(8, min(wl.n_tokens, 60.0 / max(1, args.steps + args.warmup) / per_row)))

    def step():
        oracle.run(wl.x[:rows], None if wl.residual is None else wl.residual[:rows], wl.weight,
                   eps=wl.eps, mode=mode, scale_in=scale, dtype=wl.dtype, nthreads=cores)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    nbytes = algorithmic_bytes(mode, rows, wl.hidden, 2, wl.residual is not None)
    value = nbytes / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "tokens_per_s": round(rows / dt, 1),
        "config": workload_config(args.workload, wl, mode),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {rows} of {wl.n_tokens} rows per step (host cores, no GPU)",
                         "cpu": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, dist):
    import torch
    import residual_add_rmsnorm_rmsq_gb300 as rq
    from residual_add_rmsnorm_rmsq_gb300 import _build
    _build.build()
    rq.load()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    stream = torch.cuda.Stream()
    if args.sweep_only:
        if rank == 0:
            peak, _ = measured_peak()
            print(json.dumps({"sweep_only": args.sweep_only, "modes": sweep(torch, rq, stream, peak, args)}),
                  flush=True)
        return

    mk, mode = workload_spec(args.workload)
    wl = mk()
    bufs = Buffers(torch, rq, wl, mode, 4 * L2_BYTES + 1)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # warm-up, then the timed region, bracketed by untimed replays of the same
    # launches so that the clock samples cover a window of the same load
    sampler = ClockSampler(int(os.environ.get("LOCAL_RANK", 0))) if rank == 0 else None
    rep = Replayer(torch, bufs, args.steps, args.warmup, stream)
    barrier()
    t_wall0 = time.time()
    soaked = rep.soak(args.clock_window / 2)
    ms = rep.timed()
    soaked += rep.soak(args.clock_window / 2)
    t_wall1 = time.time()
    barrier()
    ms = max_over_ranks(ms, dist, "cuda")
    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None
    if sampler:
        sampler.stop()
        clocks["window"] = (f"{(t_wall1 - t_wall0) * 1e3:.0f} ms of back-to-back replays of the timed launches "
                            f"({soaked} untimed + {args.steps} timed)")

    per_launch = bufs.bytes
    value, tokens_s = whole_job_rates(per_launch, wl.n_tokens, world, ms)

    if rank != 0:
        return
    # outputs of one timed step (buffer set 0), for the parity check below
    got = {"q": bufs.q[0].cpu().numpy(),
           "scales": None if bufs.sc[0] is None else bufs.sc[0].cpu().numpy(),
           "residual_out": None if bufs.ro[0] is None else
           bufs.ro[0].view(torch.int16).cpu().numpy().view(np.uint16)}
    scale_in = None if bufs.scale_in is None else float(bufs.scale_in.cpu().item())
    peak, peak_kind = measured_peak()
    achieved = per_launch / (ms / 1e3) / 1e9
    digest = kernel_digest()
    kname = kernel_name(wl, mode, bufs.res, torch)
    traffic = profiled_traffic(kname, digest)

    e2e_ms, h2d, d2h = e2e_measure(torch, rq, wl, mode, bufs, min(args.steps, 50), stream)
    e2e_val = per_launch * world / (e2e_ms / 1e3) / 1e9

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded splitmix64/Box-Muller, shapes of the pages' workloads)",
        "tokens_per_s": round(tokens_s, 1),
        "config": workload_config(args.workload, wl, mode),
        "launch": {"variant": VARIANT, "kernel": kname, "shape": launch_shape(wl, mode, bufs.res, torch),
                   "buffer_sets": bufs.sets,
                   "bytes_per_step": per_launch,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s", "kernel": kname},
        "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 6)},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if not args.no_sweep:
        line["modes"] = sweep(torch, rq, stream, peak, args)
        line["decode_us_per_call"] = decode_sweep(torch, rq, stream, args)
    if not args.no_cpu and world == 1:
        line["cpu_baseline"] = cpu_baseline(wl, mode, scale_in)
        line["parity"] = parity_vs_oracle(wl, mode, scale_in, got)
    print(json.dumps(line), flush=True)


def eager_us_per_call(torch, bufs, calls, stream) -> float:
    """Microseconds per call when the calls are issued one by one from the
    host on one stream (no graph): what an engine without graph capture sees,
    host launch cost included."""
    with torch.cuda.stream(stream):
        for i in range(5):
            bufs.launch(i % bufs.sets, stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(calls):
            bufs.launch(i % bufs.sets, stream)
        e1.record(stream)
        torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / calls


def decode_sweep(torch, rq, stream, args):
    """Decode batches (fp16, hidden 8192, n = 1 .. 256), every quant mode +-
    residual: microseconds per call replayed back to back from a CUDA graph
    ("graph"), and issued one by one from the host on a stream ("stream").
    Eight buffer sets rotate (at most 15 MB in all), so these inputs are
    L2-resident, as a decode step's activations usually are."""
    import rmsq_inputs as ri
    out = {"graph": {}, "stream": {}}
    for residual in (True, False):
        for n in ri.DECODE_TOKENS:
            wl = ri.decode(n, residual=residual)
            for mode in ("fp8_static", "fp8_per_token", "fp8_group128_row", "nvfp4"):
                key = f"{mode}{'' if residual else '_nores'}"
                bufs = Buffers(torch, rq, wl, mode, 4 * L2_BYTES + 1, max_sets=8)
                ms = time_launches(torch, rq, wl, mode, bufs, args.decode_steps, 5, stream)
                out["graph"].setdefault(key, {})[str(n)] = round(ms * 1e3, 3)
                out["stream"].setdefault(key, {})[str(n)] = round(
                    eager_us_per_call(torch, bufs, args.decode_steps, stream), 3)
                del bufs
    torch.cuda.empty_cache()
    return out


def sweep(torch, rq, stream, peak, args):
    """Every quant mode on its n_tokens >= 4096 workload (GB/s, fraction of
    peak), the unfused two-op sequence beside the fused op on two of them,
    QK-norm + RoPE on a Qwen3-shaped attention input (4096 / 16384 tokens,
    32 + 4 + 4 heads of 128), all-reduce + RMSNorm on the Llama layer (2 and 8
    emulated ranks), and SiLU+Mul + quantisation on a Llama-8B-shaped MLP
    activation (4096 tokens, d = 14336).  With --sweep-only REGEX, only the
    entries whose name matches."""
    import re
    import rmsq_inputs as ri
    out = {}
    want = re.compile(args.sweep_only) if args.sweep_only else None

    def wanted(name):
        return want is None or want.search(name) is not None

    def entry(name, ms, nbytes, tokens, **extra):
        gbs = nbytes / (ms / 1e3) / 1e9
        out[name] = {"us": round(ms * 1e3, 3), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
                     "tokens_per_s": round(tokens / (ms / 1e3), 1), "bytes": nbytes, **extra}

    # The unfused two-op sequence on the same workloads, for the fusion's
    # saving at kernel level: time per step of both ops against the fused op.
    for make, name, mode in ((lambda: ri.llama(4096, True), "llama_fp8_per_token", "fp8_per_token"),
                             (lambda: ri.dsv3(8192), "dsv3_fp8_group128_row", "fp8_group128_row")):
        if not wanted(f"{name}_unfused"):
            continue
        wl = make()
        fb = Buffers(torch, rq, wl, mode, 4 * L2_BYTES + 1)
        fused_ms = time_launches(torch, rq, wl, mode, fb, args.sweep_steps, 5, stream)
        del fb
        ub = UnfusedBuffers(torch, rq, wl, mode, 4 * L2_BYTES + 1)
        ms = time_launches(torch, rq, wl, mode, ub, args.sweep_steps, 5, stream)
        out[f"{name}_unfused"] = {"us": round(ms * 1e3, 3), "fused_us": round(fused_ms * 1e3, 3),
                                  "fusion_speedup": round(ms / fused_ms, 3), "bytes": ub.bytes,
                                  "fused_bytes": ub.fused_bytes,
                                  "GB/s_moved": round(ub.bytes / (ms / 1e3) / 1e9, 1)}
        del ub, wl
        torch.cuda.empty_cache()
    for n_qk in (4096, 16384):
        name = f"qwen_qk_norm_rope_{n_qk}"
        if not wanted(name):
            continue
        qk = ri.qwen_qk(n_qk)
        qb = QkBuffers(torch, rq, qk, 4 * L2_BYTES + 1)
        entry(name, time_launches(torch, rq, qk, None, qb, args.sweep_steps, 5, stream), qb.bytes, qk.n_tokens)
        del qb, qk
        torch.cuda.empty_cache()
    # all-reduce + RMSNorm at the token counts the fusion is meant for (the
    # pages: profitable at small num_tokens), 2 and 8 ranks, on the Llama layer
    for ranks in (2, 8):
        for n_ar in (16, 256, 2048):
            for mode in ("fp8_static", "nvfp4"):
                name = f"allreduce_r{ranks}_{n_ar}x4096_{mode}"
                if not wanted(name):
                    continue
                wl = ri.llama(n_ar, True)
                ab = AllReduceBuffers(torch, rq, wl, mode, ranks, 4 * L2_BYTES + 1, max_sets=64)
                ms = time_launches(torch, rq, wl, mode, ab, args.sweep_steps, 5, stream)
                entry(name, ms, ab.bytes, n_ar,
                      l2="inputs > L2" if ab.sets * ab.bytes > 4 * L2_BYTES else "L2-resident")
                del ab, wl
        torch.cuda.empty_cache()
    act = None
    for mode in ("fp8_static", "fp8_group128_row", "nvfp4"):
        name = f"llama_mlp_silu_mul_{mode}"
        if not wanted(name):
            continue
        act = act or ri.llama_mlp(4096)
        bufs = ActBuffers(torch, rq, act, mode, 4 * L2_BYTES + 1)
        entry(name, time_launches(torch, rq, act, mode, bufs, args.sweep_steps, 5, stream), bufs.bytes,
              act.n_tokens)
        del bufs
        torch.cuda.empty_cache()
    del act
    # Launch time against batch size on the Llama layer (per-token, residual):
    # the slope is the steady-state cost per row, the intercept the fixed cost
    # of a launch (ramp-up of the first copies, the last rows, completion).
    for n_scan in (512, 1024, 2048, 4096, 8192, 16384):
        name = f"scan_llama_fp8_per_token_{n_scan}"
        if not wanted(name):
            continue
        wl = ri.llama(n_scan, True)
        bufs = Buffers(torch, rq, wl, "fp8_per_token", 4 * L2_BYTES + 1)
        entry(name, time_launches(torch, rq, wl, "fp8_per_token", bufs, args.sweep_steps, 5, stream), bufs.bytes,
              n_scan)
        del bufs, wl
        torch.cuda.empty_cache()
    scan = [(int(k.rsplit("_", 1)[1]), v["us"]) for k, v in out.items() if k.startswith("scan_")]
    if len(scan) >= 2:
        xs, ys = np.array([a for a, _ in scan], float), np.array([b for _, b in scan], float)
        slope, icpt = np.polyfit(xs, ys, 1)
        out["scan_llama_fp8_per_token_fit"] = {"ns_per_row": round(slope * 1e3, 3), "intercept_us": round(icpt, 3),
                                               "steady_GB/s": round(28676 / slope / 1e3, 1)}
    groups = [
        (lambda: ri.llama(4096, True), ["llama_fp8_per_token", "llama_fp8_static"]),
        (lambda: ri.llama(4096, False), ["llama_fp8_per_token_nores"]),
        (lambda: ri.dsv3(8192), ["dsv3_fp8_group128_row", "dsv3_fp8_group128_col",
                                 "dsv3_fp8_group64_row", "dsv3_fp8_group64_col"]),
        (lambda: ri.qwen_nvfp4(4096), ["qwen_nvfp4_4096", "qwen_nvfp4_dynamic_4096"]),
        (lambda: ri.qwen_nvfp4(16384), ["qwen_nvfp4_16384", "qwen_nvfp4_dynamic_16384"]),
    ]
    for make, names in groups:
        names = [n for n in names if wanted(n)]
        if not names:
            continue
        wl = make()
        for name in names:
            mode = workload_spec(name)[1]
            bufs = Buffers(torch, rq, wl, mode, 4 * L2_BYTES + 1)
            entry(name, time_launches(torch, rq, wl, mode, bufs, args.sweep_steps, 5, stream), bufs.bytes,
                  wl.n_tokens)
            del bufs
            torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dsv3_fp8_group128_row")
    ap.add_argument("--clock-window", type=float, default=0.4,
                    help="seconds of untimed replays around the timed region, for the clock samples")
    ap.add_argument("--sweep-steps", type=int, default=300)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--sweep-only", default=None,
                    help="regex: run only these sweep entries and print them (no headline line); for profiling")
    ap.add_argument("--decode-steps", type=int, default=200)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--variant", choices=["auto", "direct", "pipelined"], default="auto")
    args = ap.parse_args()
    global VARIANT
    VARIANT = args.variant
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
        dist = tdist
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, dist)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
