#!/usr/bin/env python
"""Throughput of the sparse_attn hot path on GB300, as one JSON line.

A step is one pass of the whole path over one batch of synthetic input:
  1. window_idxs   -- the window columns of idx (the compressed columns are resident input)
  2. act_quant     -- the kv rows this step produces: the chunk's rows (prefill) or one new
                      row per sequence written into its ring slot (decode)
  3. sparse_attn   -- the index-gathered attention with the sink
The metric is query-heads per second (b * s * h per step time).  `value` is device time with
inputs resident in HBM (L2 flushed between steps, each step timed with CUDA events on the
launching stream, and queued whole before its first event fires); `e2e` times the same step through the public API with the step's inputs
copied from pinned host memory and the output read back, the queries in parts (--e2e-chunks)
whose copies in and out overlap the attention of other parts.  `roofline` relates the sparse_attn
launch to the binding roofline (HBM bytes or dense bf16 FLOPs), and `cpu_baseline` times the CPU
oracle on a bounded sample of the same workload.  The headline workload is the largest one that
fits one GPU (the window + compressed prefill); `workloads` adds the device timing and roofline
fraction of every timed workload (sliding-window prefill, window + compressed prefill, batched
decode, fp8-kv long decode), each run the same way.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

N > 1 is launched by torchrun, one rank per GPU; every rank runs its own copy of the workload
(the path has no exchange step: weak scaling) and the slowest rank's time counts.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_latent_attention_gb300 import workloads  # noqa: E402

METRIC = ("sparse_attn query·heads/s and % of roofline (HBM GB/s decode, tensor-pipe "
          "prefill)")
UNIT = "query·heads/s"
DEFAULT_WORKLOAD = "cmp_prefill"  # the largest single-GPU workload (most FLOPs and bytes)
# every workload the line times besides the headline one (the tiny case is parity-only)
TIMED_WORKLOADS = ("swa_prefill", "cmp_prefill", "decode", "fp8_decode")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "source": "fallback"}
HBM_NOMINAL_GBS = 7900.0  # GB300 HBM3e, nominal (the roofline divides by the measured copy rate)
L2_FLUSH_BYTES = 256 << 20  # twice the 129 MB L2
# A GPU-side spin (~0.2 ms at 2 GHz) after each flush, before the step's first event: the host
# enqueues the whole step while the GPU spins, so the events time the step's kernels back to back
# and not the host's argument marshalling between them (the e2e figure keeps the host in).
HEAD_START_CYCLES = 400_000

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant kernel (attn_tc_kernel),
# from the ncu captures summarised under profiles/, keyed by (hash of the files the attention
# kernels are compiled from, workload).  Any change to those files makes the key miss, so a stale
# figure reads as null.
NCU_TRAFFIC = {
    ("a4e14d8a0c3b26e5", "swa_prefill"): 495_975_851,
    ("a4e14d8a0c3b26e5", "cmp_prefill"): 1_061_977_913,
    ("a4e14d8a0c3b26e5", "decode"): 80_171_008,
    # the 4.5 GB workload itself gets a one-pass launch list only: its traffic is that of a
    # 160-sequence capture (unsplit, like the full batch) times 256 / 160
    ("a4e14d8a0c3b26e5", "fp8_decode"): 387_083_494,
}


# The translation units of the attention kernels (attn_tc_kernel, attn_mma_kernel and the split
# merge) and every header they include.
ATTN_SOURCES = ("sparse_latent_attention_gb300/csrc/sa_attn_tc.cu",
                "sparse_latent_attention_gb300/csrc/sa_attn_mma.cu",
                "sparse_latent_attention_gb300/csrc/sa_tc.cuh",
                "sparse_latent_attention_gb300/csrc/sa_fp8.cuh",
                "sparse_latent_attention_gb300/csrc/sa_internal.cuh",
                "include/sparse_attn.h")


def _sha16(paths) -> str:
    import hashlib
    root = os.path.dirname(os.path.abspath(__file__))
    h = hashlib.sha256()
    for rel in sorted(paths):
        h.update(os.path.basename(rel).encode())
        with open(os.path.join(root, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def kernel_source_hash() -> str:
    """First 16 hex digits of the sha256 over the attention kernels' sources (name + bytes)."""
    return _sha16(ATTN_SOURCES)


def library_source_hash() -> str:
    """The same over every CUDA source and header of the library."""
    import glob
    root = os.path.dirname(os.path.abspath(__file__))
    files = glob.glob(os.path.join(root, "sparse_latent_attention_gb300", "csrc", "*")) + glob.glob(
        os.path.join(root, "include", "*.h"))
    return _sha16([os.path.relpath(f, root) for f in files])


# --------------------------------------------------------------------------------------------
# multi-rank plumbing (host side; covered by the gloo tests)
# --------------------------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(backend: str):
    import torch.distributed as dist
    rank, world, local = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over all ranks (x itself at world size 1)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Whole-job throughput: every rank processed units_per_rank in at most seconds_max."""
    return units_per_rank * world / seconds_max


# --------------------------------------------------------------------------------------------
# measured peaks, clocks
# --------------------------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS)


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the benchmark runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.samples = []
        self.proc = None
        self.gpu_id = gpu_id

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id:
            cmd.insert(1, f"--id={self.gpu_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return self
        threading.Thread(target=self._read, daemon=True).start()
        return self

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

    def summary(self, t0: float, t1: float, widen: bool = True):
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        window = "timed region" if widen else "every timed step of every workload"
        if len(inside) < 3 and widen:  # a short timed region: widen to the run around it
            inside = [p for t, p in self.samples]
            window = "warm-up + timed run"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        smax = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4)
                          if p[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(inside), "window": window,
                "power_w_max": max((num(p[2]) or 0.0) for p in inside)}


def gpu_id_of(torch, dev) -> str | None:
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
    except Exception:  # noqa: BLE001
        return None


# --------------------------------------------------------------------------------------------
# the workload's algorithmic bytes and FLOPs
# --------------------------------------------------------------------------------------------

def unique_kv_bytes(wl, idx_np: np.ndarray) -> int:
    total = 0
    for bi in range(wl.b):
        u = np.unique(idx_np[bi])
        total += int((u >= 0).sum())
    return total * wl.kv_row_bytes()


def roofline_terms(wl, idx_np, peaks):
    q_bytes = wl.q_bytes()
    o_bytes = q_bytes
    kv_bytes = unique_kv_bytes(wl, idx_np)
    alg_bytes = q_bytes + o_bytes + kv_bytes
    flops = wl.flops()
    t_hbm = alg_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    return dict(alg_bytes=alg_bytes, kv_bytes=kv_bytes, flops=flops, t_hbm=t_hbm, t_tc=t_tc,
                bound="hbm" if t_hbm >= t_tc else "tensor")


# --------------------------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------------------------

class GpuPath:
    """Device buffers of one workload and its step through the library."""

    def __init__(self, wl, dev, rope_dim=0):
        import torch

        import sparse_latent_attention_gb300 as sa
        self.torch, self.sa, self.wl, self.dev = torch, sa, wl, dev
        bf16 = torch.bfloat16

        def to_dev_bf16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(bf16).to(dev)

        self.fp8 = wl.kv_format == "fp8"
        self.decode = wl.s == 1 and wl.start_pos > 0
        self.q = to_dev_bf16(wl.q)
        self.sink = torch.from_numpy(wl.sink).to(dev)
        self.idx = torch.full((wl.b, wl.s, wl.topk), -1, dtype=torch.int32, device=dev)
        self.idx[:, :, wl.window:] = torch.from_numpy(wl.idx_tail).to(dev)
        # every kv row in raw form, quantised once here; the step re-quantises the rows it owns
        raw = torch.zeros((wl.b, wl.rows, wl.d), dtype=bf16, device=dev)
        rows = torch.from_numpy(wl.kv_rows).to(dev)
        raw[torch.arange(wl.b, device=dev)[:, None].expand_as(rows), rows] = to_dev_bf16(wl.kv_vals)
        d = wl.d
        if self.fp8:
            self.kv = torch.empty((wl.b, wl.rows, d), dtype=torch.uint8, device=dev)
            self.kv_scale = torch.empty((wl.b, wl.rows, d // 32), dtype=torch.uint8, device=dev)
            sa.act_quant_fp8(raw.view(-1, d), codes=self.kv.view(-1, d),
                             scales=self.kv_scale.view(-1, d // 32))
        else:
            self.kv = raw.clone()
            self.kv_scale = None
            sa.act_quant_fp8(self.kv.view(-1, d), out_rt=self.kv.view(-1, d))
        if self.decode:
            self.slot = wl.start_pos % wl.window
            self.new_rows = raw[:, self.slot, :].contiguous()   # this step's latent row per sequence
        else:
            self.new_rows = raw[:, : wl.s, :].contiguous()      # the chunk's latent rows
        del raw
        self.o = torch.empty_like(self.q)
        self.ws = sa.new_workspace(wl.b, wl.s, wl.h, d, wl.rows, wl.topk,
                                   sa.SA_KV_FP8_E4M3 if self.fp8 else sa.SA_KV_BF16, device=dev)
        self.launches_per_step = 2 + (2 if self.ws.numel() > sa.SA_STATUS_BYTES else 1)
        # optional inverse rotation of o's last rope_dim dims, fused into the attention call
        self.rot = None
        if rope_dim:
            self.rot = torch.from_numpy(
                workloads.rope_table(wl.start_pos + wl.s, rope_dim, seed=7)).to(dev)

    def step(self, ev=None):
        """One pass of the path; ev = (start, end) CUDA events bracketing sparse_attn."""
        self.prologue()
        if ev is not None:
            ev[0].record()
        self.attn()
        if ev is not None:
            ev[1].record()

    def chunks(self, n):
        """n contiguous parts of the step's queries: (slice of q / idx / o, slice of kv).  Batched
        decode splits the sequences, a prefill (b = 1) its query tokens."""
        wl = self.wl
        if wl.b > 1:
            edges = np.linspace(0, wl.b, min(n, wl.b) + 1).astype(int)
            return [((slice(a, b),), (slice(a, b),)) for a, b in zip(edges, edges[1:]) if b > a]
        edges = np.linspace(0, wl.s, min(n, wl.s) + 1).astype(int)
        return [((slice(None), slice(a, b)), (slice(None),)) for a, b in zip(edges, edges[1:]) if b > a]

    def attn(self, part=None, workspace=None):
        """sparse_attn over every query, or over one part from chunks() (on the current stream)."""
        wl = self.wl
        qs, ks = part if part is not None else ((slice(None),), (slice(None),))
        rope = None
        if self.rot is not None:  # a part of a prefill starts at its first token's position
            first = (qs[1].start or 0) if len(qs) > 1 else 0
            rope = (self.rot, wl.start_pos + first)
        self.sa.sparse_attn(self.q[qs], self.kv[ks], self.sink, self.idx[qs], wl.scale,
                            kv_scale=None if self.kv_scale is None else self.kv_scale[ks],
                            out=self.o[qs], workspace=self.ws if workspace is None else workspace,
                            rope=rope)

    def workspace_for(self, parts):
        """A workspace large enough for every part (fewer queries can mean more split scratch)."""
        wl, sa = self.wl, self.sa
        fmt = sa.SA_KV_FP8_E4M3 if self.fp8 else sa.SA_KV_BF16
        need = max(sa.workspace_size(*self.q[qs].shape[:2], wl.h, wl.d, wl.rows, wl.topk, fmt)
                   for qs, _ in parts)
        if need <= self.ws.numel():
            return self.ws
        return self.torch.zeros(need, dtype=self.torch.uint8, device=self.dev)

    def prologue(self):
        """The step's window index table and the re-quantisation of the rows it owns."""
        sa, wl, d = self.sa, self.wl, self.wl.d
        sa.window_idxs(wl.start_pos, wl.s, wl.window, out=self.idx[:, :, : wl.window], nbatch=wl.b)
        if self.decode:  # the step's token enters each sequence's ring (its first window rows)
            x = self.new_rows[:, None, :]
            if self.fp8:
                sa.window_write(x, wl.start_pos, codes=self.kv[:, : wl.window],
                                scales=self.kv_scale[:, : wl.window])
            else:
                sa.window_write(x, wl.start_pos, ring_rt=self.kv[:, : wl.window])
        else:
            nr = self.new_rows.view(-1, d)
            sa.act_quant_fp8(nr, out_rt=self.kv[:, : wl.s, :].reshape(-1, d))


COMPRESS_RATIO = 4  # the compressed workloads' ratio
CANDIDATE_TOPK_BLOCKS, CANDIDATE_BLOCK_SIZE = 2048, 8  # the model config's candidate blocks


def time_indexer_topk(wl, dev, steps, warmup, peaks):
    """The indexer's two selection steps at this workload's compressed shape, each timed alone:
    sa_indexer_topk and sa_candidate_blocks (2048 blocks of 8) on index scores
    [b, s, n_comp] f32 drawn N(0, 1), n_comp = (start_pos + s) / 4, -> the workload's compressed
    idx columns (index_topk = its non-window columns, offset = the rows before the compressed
    ones).  Timed alone like the step: L2 flushed, the call queued before its events."""
    import torch

    import sparse_latent_attention_gb300 as sa
    n = (wl.start_pos + wl.s) // COMPRESS_RATIO
    index_topk = wl.topk - wl.window
    if index_topk <= 0 or n == 0 or wl.rows < n:
        return None  # no compressed columns in this workload
    offset = wl.rows - n
    k = min(index_topk, n)
    g = torch.Generator(device=dev).manual_seed(11)
    score = torch.randn((wl.b, wl.s, n), generator=g, device=dev, dtype=torch.float32)
    out = torch.empty((wl.b, wl.s, k), dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    mask = torch.empty((wl.b, wl.s, n), dtype=torch.bool, device=dev)

    def timed(call):
        for _ in range(warmup):
            flush.zero_()
            call()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        torch.cuda.synchronize()
        for a, b in ev:
            flush.zero_()
            torch.cuda._sleep(HEAD_START_CYCLES)
            a.record()
            call()
            b.record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / len(ev)

    def line(kernel, ms, alg, **extra):
        gbs = alg / (ms * 1e-3) / 1e9
        return {"kernel": kernel, "ms": round(ms, 4), "alg_bytes": int(alg), "bound": "hbm",
                "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm_gbs"], 4), "queries": wl.b * wl.s,
                "positions": n, **extra}

    # algorithmic bytes: the scores a query can see (a prefill's hidden positions are never
    # read), plus what is written (the idx, or one mask byte a position)
    if wl.start_pos == 0:
        seen = wl.b * sum((si + 1) // COMPRESS_RATIO for si in range(wl.s))
    else:
        seen = wl.b * wl.s * n
    ms_topk = timed(lambda: sa.indexer_topk(score, wl.start_pos, COMPRESS_RATIO, index_topk,
                                            offset, out=out))
    ms_cand = timed(lambda: sa.candidate_blocks(score, wl.start_pos, COMPRESS_RATIO,
                                                CANDIDATE_TOPK_BLOCKS, CANDIDATE_BLOCK_SIZE,
                                                out=mask))
    return {"indexer_topk": line("indexer_topk_kernel", ms_topk, 4 * seen + 4 * wl.b * wl.s * k,
                                 k=k, score="f32"),
            "candidate_blocks": line("candidate_blocks_kernel", ms_cand,
                                     4 * seen + wl.b * wl.s * n, topk_blocks=CANDIDATE_TOPK_BLOCKS,
                                     block_size=CANDIDATE_BLOCK_SIZE, score="f32")}


HC_TOKENS = 1 << 20  # token rows of the hc_split_sinkhorn timing (201 MB in + out, past L2)


def time_hc_split_sinkhorn(dev, steps, warmup, peaks):
    """hc_split_sinkhorn (hc 4, 20 rounds, eps 1e-6) on 2^20 token rows of N(0, 1) mixes, timed
    alone like the step; algorithmic bytes = the mixes read and pre / post / comb written."""
    import torch

    import sparse_latent_attention_gb300 as sa
    g = torch.Generator(device=dev).manual_seed(12)
    mixes = torch.randn((HC_TOKENS, 24), generator=g, device=dev)
    scale = torch.ones(3, device=dev)
    base = torch.zeros(24, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        sa.hc_split_sinkhorn(mixes, scale, base)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        flush.zero_()
        torch.cuda._sleep(HEAD_START_CYCLES)
        a.record()
        sa.hc_split_sinkhorn(mixes, scale, base)
        b.record()
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in ev) / len(ev)
    alg = HC_TOKENS * (24 + 24) * 4
    gbs = alg / (ms * 1e-3) / 1e9
    return {"kernel": "hc_split_sinkhorn_kernel", "ms": round(ms, 4), "alg_bytes": int(alg),
            "bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(gbs / peaks["hbm_gbs"], 4), "tokens": HC_TOKENS, "hc": 4, "iters": 20}


def roofline_line(terms, peaks, ms_attn, traffic):
    """The JSON line's roofline object for the sparse_attn call: the achieved rate against the
    binding measured peak (HBM bytes or dense bf16 FLOPs), the other roofline beside it, and the
    sustained-bf16 and nominal-HBM figures as context."""
    t_attn = ms_attn / 1e3
    gbs = terms["alg_bytes"] / t_attn / 1e9
    tfs = terms["flops"] / t_attn / 1e12
    hbm = {"unit": "GB/s", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
           "frac": round(gbs / peaks["hbm_gbs"], 4)}
    tc = {"unit": "TFLOP/s", "achieved": round(tfs, 1), "peak": peaks["bf16_tflops"],
          "frac": round(tfs / peaks["bf16_tflops"], 4)}
    binding, other = (hbm, tc) if terms["bound"] == "hbm" else (tc, hbm)
    roof = {"bound": terms["bound"], "achieved": binding["achieved"], "peak": binding["peak"],
            "unit": binding["unit"], "frac": binding["frac"], "traffic": traffic,
            "kernel": "sa_sparse_attn", "ms": round(ms_attn, 4), "alg_bytes": terms["alg_bytes"],
            "alg_flops": terms["flops"], "peak_source": peaks["source"] + " (burst)",
            "other": other,
            "roofline_ms": round(max(terms["t_hbm"], terms["t_tc"]) * 1e3, 4),
            "frac_of_roofline_time": round(max(terms["t_hbm"], terms["t_tc"]) / t_attn, 4)}
    # context beside the binding measured peak: the sustained bf16 figure (a long GEMM under the
    # power cap) and the nominal HBM3e bandwidth
    sustained = peaks.get("bf16_tflops_sustained")
    roof["context"] = {
        "bf16_tflops_sustained": sustained,
        "tensor_frac_of_sustained": round(tfs / sustained, 4) if sustained else None,
        "hbm_nominal_gbs": HBM_NOMINAL_GBS,
        "hbm_frac_of_nominal": round(gbs / HBM_NOMINAL_GBS, 4)}
    return roof


def time_device_steps(torch, path, flush, steps, warmup):
    """warmup + steps passes of the path, each timed on the device with CUDA events (the step, and
    the sparse_attn call inside it); the L2 is flushed before every step and the step is queued
    whole behind an untimed GPU spin, so the events time the kernels back to back."""
    for _ in range(warmup):
        flush.zero_()
        torch.cuda._sleep(HEAD_START_CYCLES)
        path.step()
    torch.cuda.synchronize()
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(steps)]
    for e in ev:
        flush.zero_()
        torch.cuda._sleep(HEAD_START_CYCLES)  # not timed: lets the host queue the step first
        e[0].record()
        path.step(ev=(e[2], e[3]))
        e[1].record()
    torch.cuda.synchronize()
    return ([a.elapsed_time(b) for a, b, _, _ in ev], [c.elapsed_time(d) for _, _, c, d in ev])


def config_of(wl, world, rope=0):
    """The workload's config object; the GPU arm and the reference arm print the same one."""
    return {"workload": wl.name, "b": wl.b, "s": wl.s, "h": wl.h, "d": wl.d,
            "rows": wl.rows, "topk": wl.topk, "window": wl.window,
            "start_pos": wl.start_pos, "kv_format": wl.kv_format,
            "l2": "flushed between timed steps (256 MB write, outside the step events)",
            "launch": "each step fully queued before its first event (a 0.2 ms GPU spin "
                      "after the flush, outside the events)",
            "parallelism": f"replica x{world}" if world > 1 else "1 GPU",
            **({"inverse_rope_dims": rope} if rope else {})}


def workload_line(wl, terms, peaks, step_ms, attn_ms, traffic):
    """One workload's device timing: the step and its sparse_attn call, the binding roofline's
    fraction, the other roofline, and the ncu traffic for the current kernel sources (or null)."""
    ms_step = sum(step_ms) / len(step_ms)
    ms_attn = sum(attn_ms) / len(attn_ms)
    roof = roofline_line(terms, peaks, ms_attn, traffic)
    return {"ms_per_step": round(ms_step, 4), "ms_attn": round(ms_attn, 4),
            "value": round(wl.n_tokens * wl.h / (ms_step / 1e3), 1), "unit": UNIT,
            "bound": roof["bound"], "frac": roof["frac"], "achieved": roof["achieved"],
            "peak": roof["peak"], "roof_unit": roof["unit"], "other": roof["other"],
            "roofline_ms": roof["roofline_ms"], "traffic": traffic,
            "traffic_key": [kernel_source_hash(), wl.name], "steps": len(step_ms)}


def host_link_rates(torch, dev, nbytes=256 << 20, reps=5):
    """Pinned host <-> device copy rates (GB/s, best of reps), each direction alone and both at
    once on two streams: the floor of the end-to-end step's copies."""
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h2 = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d2 = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def best(fn):
        t = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            t.append(a.elapsed_time(b) / 1e3)
        return min(t)

    def both():
        cur = torch.cuda.current_stream()
        s1.wait_stream(cur)
        s2.wait_stream(cur)
        with torch.cuda.stream(s1):
            d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s2):
            h2.copy_(d2, non_blocking=True)
        cur.wait_stream(s1)
        cur.wait_stream(s2)

    t_h2d = best(lambda: d.copy_(h, non_blocking=True))
    t_d2h = best(lambda: h2.copy_(d2, non_blocking=True))
    t_both = best(both)
    return {"h2d_gbs": round(nbytes / t_h2d / 1e9, 1), "d2h_gbs": round(nbytes / t_d2h / 1e9, 1),
            "duplex_gbs": round(2 * nbytes / t_both / 1e9, 1), "bytes": nbytes}


def e2e_link_floor_ms(link, h2d_bytes, d2h_bytes):
    """The end-to-end step's copies alone at the measured pinned rates, the two directions
    overlapped (as the step's parts overlap them): max of each direction alone and of the total
    at the duplex rate."""
    t = max(h2d_bytes / (link["h2d_gbs"] * 1e9), d2h_bytes / (link["d2h_gbs"] * 1e9),
            (h2d_bytes + d2h_bytes) / (link["duplex_gbs"] * 1e9))
    return t * 1e3


def run_gpu(args, rank, world, local):
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rank0 = rank == 0
    peaks = load_peaks()
    wl = workloads.make_named(args.workload, batch=args.batch)
    path = GpuPath(wl, dev, rope_dim=args.rope)
    path.step()
    torch.cuda.synchronize()
    idx_np = path.idx.cpu().numpy()
    terms = roofline_terms(wl, idx_np, peaks)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    sampler = ClockSampler(gpu_id_of(torch, dev)).start() if rank0 else None
    time_device_steps(torch, path, flush, 0, args.warmup)

    # timed region: K steps, each bracketed by events; L2 flushed between steps (not timed)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    step_ms, attn_ms = time_device_steps(torch, path, flush, args.steps, 0)
    barrier(world)
    t1 = time.time()
    assert path.sa.read_status(path.ws) == 0, "kernel reported an out-of-range index"

    # end to end through the public API: host inputs in, host output out, every step
    pin = dict(q=path.q.cpu().pin_memory(), rows=path.new_rows.cpu().pin_memory(),
               sink=path.sink.cpu().pin_memory(),
               idx=path.idx.cpu().pin_memory() if wl.topk > wl.window else None,
               o=torch.empty(path.o.shape, dtype=path.o.dtype).pin_memory())
    h2d = (pin["q"].numel() * 2 + pin["rows"].numel() * 2 + pin["sink"].numel() * 4 +
           (pin["idx"].numel() * 4 if pin["idx"] is not None else 0))
    d2h = pin["o"].numel() * 2

    # The queries go in, are attended and come back out in parts, on three streams, so that the
    # copies of one part overlap the compute of another (every byte still crosses the link every
    # step, and every output is computed); --e2e-chunks 1 is the plain serial step.
    # (default: one part per 256 query tokens, at most 16 -- parts large enough to fill the GPU
    # without splitting their index columns; a decode batch stays whole)
    n_parts = args.e2e_chunks if args.e2e_chunks > 0 else max(1, min(16, wl.n_tokens // 256))
    parts = path.chunks(n_parts)
    ws_parts = path.workspace_for(parts)
    s_in, s_cmp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))

    def e2e_step_serial():
        path.q.copy_(pin["q"], non_blocking=True)
        path.new_rows.copy_(pin["rows"], non_blocking=True)
        path.sink.copy_(pin["sink"], non_blocking=True)
        if pin["idx"] is not None:
            path.idx.copy_(pin["idx"], non_blocking=True)
        path.step()
        pin["o"].copy_(path.o, non_blocking=True)

    ev_cmp_all = torch.cuda.Event()                        # every compute of a step is done
    ev_out = [torch.cuda.Event() for _ in parts]           # part i's copy out is done
    ev_q = [torch.cuda.Event() for _ in parts]             # part i's queries are in
    ev_in, ev_pro = torch.cuda.Event(), torch.cuda.Event()
    started = [False]

    def e2e_step_parts():
        """One step: the step's inputs in (idx, sink, the new kv rows, then the queries part by
        part), the prologue, each part's attention and its copy out, on three streams.  A step's
        copies in wait only for the previous step's computes (which read q, idx and kv), so they
        overlap the previous step's last copies out; a part's attention also waits for that
        part's previous copy out (o is reused)."""
        cur = torch.cuda.current_stream()
        s_in.wait_stream(cur)  # after the timing event and the previous step's prologue
        if started[0]:
            s_in.wait_event(ev_cmp_all)
        with torch.cuda.stream(s_in):
            if pin["idx"] is not None:
                path.idx.copy_(pin["idx"], non_blocking=True)
            path.sink.copy_(pin["sink"], non_blocking=True)
            path.new_rows.copy_(pin["rows"], non_blocking=True)
            ev_in.record()
        cur.wait_event(ev_in)
        path.prologue()
        ev_pro.record(cur)
        for i, part in enumerate(parts):
            qs = part[0]
            with torch.cuda.stream(s_in):
                path.q[qs].copy_(pin["q"][qs], non_blocking=True)
                ev_q[i].record()
            s_cmp.wait_event(ev_pro)
            s_cmp.wait_event(ev_q[i])
            if started[0]:
                s_cmp.wait_event(ev_out[i])
            with torch.cuda.stream(s_cmp):
                path.attn(part, ws_parts)
            s_out.wait_stream(s_cmp)
            with torch.cuda.stream(s_out):
                pin["o"][qs].copy_(path.o[qs], non_blocking=True)
                ev_out[i].record()
        ev_cmp_all.record(s_cmp)
        started[0] = True

    e2e_step = e2e_step_parts if len(parts) > 1 else e2e_step_serial

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 20))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record()
    for _ in range(e2e_steps):
        e2e_step()
    # the last step's copies out (on their own stream) are inside the timed region
    torch.cuda.current_stream().wait_stream(s_out)
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    # the overlapped end-to-end step read back what a plain step computes, bit for bit
    path.step()
    torch.cuda.synchronize()
    assert torch.equal(pin["o"].view(torch.int16), path.o.cpu().view(torch.int16)), \
        "end-to-end output differs from the device step"

    # the other workloads, each timed alone the same way (device time only; rank 0's GPU line
    # carries them, every rank runs them so the ranks stay in step)
    others = {}
    if not args.headline_only and args.batch is None:
        del flush
        for name in TIMED_WORKLOADS:
            if name == wl.name:
                continue
            wl_o = workloads.make_named(name)
            path_o = GpuPath(wl_o, dev)
            path_o.step()
            torch.cuda.synchronize()
            terms_o = roofline_terms(wl_o, path_o.idx.cpu().numpy(), peaks)
            flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
            time_device_steps(torch, path_o, flush, 0, args.warmup)
            sm_o, am_o = time_device_steps(torch, path_o, flush, args.steps, 0)
            assert path_o.sa.read_status(path_o.ws) == 0, f"{name}: kernel status"
            others[name] = workload_line(wl_o, terms_o, peaks, sm_o, am_o,
                                         NCU_TRAFFIC.get((kernel_source_hash(), name)))
            del path_o, flush
            torch.cuda.empty_cache()
    t2 = time.time()
    if sampler:
        sampler.stop()
    link = host_link_rates(torch, dev) if rank0 else None

    units = wl.n_tokens * wl.h
    ms_step = max_over_ranks(sum(step_ms) / len(step_ms), world, dev)
    ms_attn = max_over_ranks(sum(attn_ms) / len(attn_ms), world, dev)
    ms_e2e = max_over_ranks(e2e_ms, world, dev)
    if not rank0:
        return None
    value = job_value(units, world, ms_step / 1e3)
    lib_version = path.sa._lib.version()
    src_hash = kernel_source_hash()
    roof = roofline_line(terms, peaks, ms_attn, NCU_TRAFFIC.get((src_hash, wl.name)))
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8-e4m3 kv, bf16 q/o, f32 accumulate" if path.fp8 else
                 "bf16 (f32 accumulate)",
        "data": "synthetic (seeded N(0,1) inputs with the workload's index structure)",
        "config": config_of(wl, world, args.rope),
        "roofline": roof,
        "e2e": {"value": round(job_value(units, world, ms_e2e / 1e3), 1), "unit": UNIT,
                "ms_per_step": round(ms_e2e, 4), "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "parts": len(parts),
                "link": link,
                "link_floor_ms": round(e2e_link_floor_ms(link, h2d, d2h), 4),
                "frac_of_link_floor": round(e2e_link_floor_ms(link, h2d, d2h) / ms_e2e, 4)},
        "gpu_launches": path.launches_per_step * args.steps,
        "clocks": sampler.summary(t0, t1) if sampler else None,
        "clocks_all_timing": sampler.summary(t0, t2, widen=False) if sampler else None,
        "workloads": dict(others, **{wl.name: workload_line(
            wl, terms, peaks, step_ms, attn_ms, NCU_TRAFFIC.get((src_hash, wl.name)))}),
        "lib_version": lib_version,
        "kernel_source_hash": src_hash,
        "library_source_hash": library_source_hash(),
    }
    if args.indexer_topk:
        out["next_rows"] = time_indexer_topk(wl, dev, args.steps, args.warmup, peaks)
    if args.hc_sinkhorn:
        out.setdefault("next_rows", {})
        out["next_rows"] = dict(out["next_rows"] or {},
                                hc_split_sinkhorn=time_hc_split_sinkhorn(dev, args.steps,
                                                                         args.warmup, peaks))
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_budget)
    return out


# --------------------------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# --------------------------------------------------------------------------------------------

class OracleStep:
    """The path's step on the CPU oracle, on a sample of the workload's query tokens."""

    def __init__(self, wl, seed=0):
        import oracle
        self.oracle, self.wl = oracle, wl
        oracle.build()
        self.threads = os.cpu_count() or 1
        rng = np.random.default_rng(seed)
        self.order = rng.permutation(wl.n_tokens)
        self.pos = 0
        # resident state prepared outside any timing: quantised cache rows and the idx tail
        zrt, zc, zs = oracle.act_quant(np.zeros((1, wl.d), np.uint16))
        self.zero_row = (zrt, zc, zs)
        self.idx = np.full((wl.b, wl.s, wl.topk), -1, np.int32)
        self.idx[:, :, wl.window:] = wl.idx_tail
        self._cache = {}

    def _seq_state(self, bi):
        """Quantised kv of one sequence (rows that hold values quantised once, cached)."""
        if bi not in self._cache:
            wl, o = self.wl, self.oracle
            rt_u, codes_u, sc_u = o.act_quant(wl.kv_vals[bi])
            zrt, zc, zs = self.zero_row
            if wl.kv_format == "fp8":
                codes = np.broadcast_to(zc, (wl.rows, wl.d)).copy()
                scales = np.broadcast_to(zs, (wl.rows, wl.d // 32)).copy()
                codes[wl.kv_rows[bi]] = codes_u
                scales[wl.kv_rows[bi]] = sc_u
                self._cache[bi] = (codes, scales)
            else:
                rt = np.broadcast_to(zrt, (wl.rows, wl.d)).copy()
                rt[wl.kv_rows[bi]] = rt_u
                self._cache[bi] = (rt, None)
        return self._cache[bi]

    def prepare(self, tokens):
        for bi in sorted(set((np.asarray(tokens) // self.wl.s).tolist())):
            self._seq_state(bi)

    def next_tokens(self, n):
        if self.pos + n > len(self.order):
            self.pos = 0
        t = self.order[self.pos:self.pos + n]
        self.pos += n
        return np.sort(t)

    def run(self, tokens):
        """window_idxs + act_quant of the rows this step owns + attention for `tokens`."""
        wl, o = self.wl, self.oracle
        win = o.window_idxs(wl.start_pos, wl.s, wl.window)
        self.idx[:, :, : wl.window] = win[None]
        if wl.s == 1 and wl.start_pos > 0:
            # one new row per sequence, in its ring slot (rows 0..window-1 lead kv_vals)
            o.act_quant(wl.kv_vals[:, wl.start_pos % wl.window, :])
        else:
            o.act_quant(wl.kv_vals[0, : wl.s])  # the chunk's rows
        by_seq = {}
        for t in tokens:
            by_seq.setdefault(int(t) // wl.s, []).append(int(t) % wl.s)
        for bi, sl in by_seq.items():
            kv, sc = self._seq_state(bi)
            o.sparse_attn(wl.q[bi:bi + 1], kv[None], wl.sink, self.idx[bi:bi + 1], wl.scale,
                          kv_scales=None if sc is None else sc[None], tokens=np.array(sl),
                          nthreads=self.threads)


def cpu_baseline(wl, budget_s=12.0):
    """The oracle step timed on the host's cores over chunks of the workload's query tokens
    (wrapping around the workload when it is shorter than the budget) until ~budget_s of CPU
    work has been timed."""
    step = OracleStep(wl)
    probe = step.next_tokens(min(64, wl.n_tokens))
    step.prepare(probe)
    t = time.perf_counter()
    step.run(probe)
    per_tok = (time.perf_counter() - t) / len(probe)
    # chunks of ~1/4 of the budget (at least the probe's size), capped at the workload
    chunk = int(max(len(probe), min(wl.n_tokens, 0.25 * budget_s / max(per_tok, 1e-9))))
    done, total = 0, 0.0
    while total < budget_s:
        tokens = step.next_tokens(chunk)
        step.prepare(tokens)  # quantised cache rows: setup, outside the timing
        t = time.perf_counter()
        step.run(tokens)
        total += time.perf_counter() - t
        done += len(tokens)
    return {"value": round(done * wl.h / total, 1), "unit": UNIT, "cores": step.threads,
            "kind": "oracle",
            "sample": f"{done} query tokens (all {wl.h} heads) of {wl.name} in chunks of {chunk} "
                      f"(the workload has {wl.n_tokens}; chunks wrap around it), plus each chunk's "
                      f"window_idxs and act_quant; {total:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    wl = workloads.make_named(args.workload, batch=args.batch)
    step = OracleStep(wl)
    probe = step.next_tokens(min(8, wl.n_tokens))
    step.prepare(probe)
    t = time.perf_counter()
    step.run(probe)
    per_tok = (time.perf_counter() - t) / len(probe)
    per_step_budget = args.ref_budget / max(1, args.steps + args.warmup)
    n = int(max(1, min(wl.n_tokens, per_step_budget / max(per_tok, 1e-9))))
    for _ in range(args.warmup):
        tk = step.next_tokens(n)
        step.prepare(tk)
        step.run(tk)
    times = []
    for _ in range(args.steps):
        tk = step.next_tokens(n)
        step.prepare(tk)  # cache preparation is setup, outside the timed step
        t = time.perf_counter()
        step.run(tk)
        times.append(time.perf_counter() - t)
    total = sum(times)
    value = n * wl.h * args.steps / total
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (CPU oracle)",
        "data": "synthetic (seeded N(0,1) inputs with the workload's index structure)",
        "config": config_of(wl, world),
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "kind": "oracle",
                         "cores": step.threads,
                         "sample": f"{n} query tokens per step (all heads) of {wl.name}, "
                                   "with the step's window_idxs and act_quant"},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=[n for n in workloads.NAMED])
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work")
    ap.add_argument("--ref-budget", type=float, default=90.0,
                    help="seconds of oracle work for the whole --impl reference run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="time only --workload (skip the line's other workloads)")
    ap.add_argument("--batch", type=int, default=None,
                    help="sequences of a decode workload (a smaller case for profiler captures)")
    ap.add_argument("--e2e-chunks", type=int, default=0,
                    help="parts the end-to-end step's queries are copied and attended in "
                         "(0: one per 256 query tokens, at most 16)")
    ap.add_argument("--indexer-topk", action="store_true",
                    help="also time the indexer's selection and candidate blocks at the "
                         "workload's compressed shape")
    ap.add_argument("--hc-sinkhorn", action="store_true",
                    help="also time hc_split_sinkhorn on 2^20 token rows")
    ap.add_argument("--rope", type=int, default=0, metavar="DIMS",
                    help="also rotate o's last DIMS dims back (inverse RoPE fused into the call; "
                         "the layer uses 64); 0 = off")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = dist_env()
    if world != args.gpus:
        if world == 1 and args.gpus > 1:
            ap.error("--gpus N > 1 is launched with torchrun (one rank per GPU)")
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        dist_init("nccl")
        out = run_gpu(args, rank, world, local)
    if out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
