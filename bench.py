#!/usr/bin/env python
"""Benchmark of the tensor-parallel sharded projection on one GB300.

Default workload: a stack of 8 SwiGLU MLP blocks (hidden 6144, ffn 18432,
tokens 4608, tp_degree 4, all four ranks on this GPU), loaded shard-on-read
from a page-locked host state dict of 5.44 GB of bf16.

* ``value`` -- the sharded blocks' throughput: the forward pass through all 8
  blocks (per block: tp_linear_colwise with the fused SwiGLU epilogue, then
  tp_linear_rowwise with the ranks' partials summed on chip) is one step; value
  = its FLOPs (2*T*K*N per projection, summed over ranks) per second of device
  time, the shards and the input already resident in HBM.  Every step reads
  5.44 GB of weights, far more than L2, so no flush is needed between steps.
* ``roofline`` -- the dominant kernel, the gate/up GEMM with the SwiGLU
  epilogue: its FLOPs per launch over its mean launch time (each launch timed
  alone with CUDA events), against the measured sustained bf16 peak (the
  launches run back to back inside a 14 ms pass).
* ``shard_load`` -- shard-extract GB/s: every rank's slice of all 16 weights
  read from the page-locked state dict straight into device shards
  (tp_plan_shard_ranks), against a plain host-to-device copy of 1 GiB measured
  in the same run (the link, not HBM, bounds it).
* ``e2e`` -- the same metric through the C-ABI with host buffers: each step
  reads every rank's slice of every weight from host memory, copies the input
  in and the output back, pipelined (block b computes while later blocks'
  slices arrive).
* ``cpu_baseline`` -- the float64 numpy oracle on a seeded sample of token
  rows through all 8 blocks (all shards extracted), on the host's cores.
* ``attn_proj_tp4`` and ``block_tp4`` -- per-kernel figures of the attention
  projections (tokens 4096, hidden 3072, 24 heads) and of the full attention +
  SwiGLU MLP block (hidden 6144, 48 heads, tp 4), each step timed with L2
  flushed between steps (a 256 MiB write, then a 256 MiB read), including the
  rowwise projection in both join forms (on-chip sum, fp32 partials summed in
  the GEMM epilogue through an HBM workspace) and the device-to-device
  extraction GB/s against HBM.

``--workload`` runs one of the other workloads alone with the same machinery.
``--impl reference`` times the CPU oracle on the default workload, each step a
bounded sample (one block on sampled token rows).

The library simulates every rank on one GPU; it is a single-GPU library (its
GEMMs multicast operand tiles inside a thread-block cluster of this GPU), so
this benchmark refuses to run under torchrun with more than one process.
"""
from __future__ import annotations

import os

# The CPU baseline uses every host core through BLAS; fix the thread count
# before numpy loads so it can be reported.
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))

import argparse
import hashlib
import json
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import tp_inputs  # noqa: E402

METRIC = "sharded-block TFLOP/s & % bf16 tensor peak on 1 GB300; shard-extract GB/s % HBM"
UNIT = "TFLOP/s"
WORKLOAD = "stack8_swiglu_tp4"
ATTN_PROJ = "attn_proj_tp4"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """Empties L2 between timed steps: a write larger than L2 evicts whatever the
    last step left there, and a read of another buffer as large then evicts the
    write's own dirty lines, so the next step starts from a cold, clean L2 (the
    state a profiler's cache flush gives) and pays for none of the flush's
    write-backs."""

    def __init__(self, torch, device):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.amax()


def refuse_multi_gpu(args) -> None:
    """One process, one GPU: the library is a single-GPU library; more GPUs are refused."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1 or args.gpus != 1:
        msg = (f"single-GPU benchmark: libtp simulates every tensor-parallel rank on one GPU and its GEMMs "
               f"multicast operand tiles within a cluster of that GPU; refusing WORLD_SIZE={world}, --gpus {args.gpus}")
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps({"metric": METRIC, "value": None, "n_gpus": max(world, args.gpus), "error": msg}))
        print(msg, file=sys.stderr)
        sys.exit(2)


# ----------------------------------------------------------------------------- peaks, clocks, traffic

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS)


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def source_digest(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


KERNEL_SOURCES = {
    "gemm": ["tensor_sharded_linear_tp_gb300/csrc/tp_gemm.cu", "tensor_sharded_linear_tp_gb300/csrc/tp_ptx.cuh",
             "tensor_sharded_linear_tp_gb300/csrc/tp_internal.h"],
    "copy": ["tensor_sharded_linear_tp_gb300/csrc/tp_copy.cu", "tensor_sharded_linear_tp_gb300/csrc/tp_internal.h"],
}


def recorded_traffic(kernel: str, kind: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernel source.

    profiles/dram_traffic.txt lines: <kernel> <source-digest> <dram-bytes-per-launch> <note...>
    """
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    digest = source_digest(KERNEL_SOURCES[kind])
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel and parts[1] == digest:
                    return float(parts[2])
    except FileNotFoundError:
        pass
    return None


# ----------------------------------------------------------------------------- workload

class AttnProjWorkload:
    """Attention projections, tp_degree 4: fused QKV colwise + gather, out-projection rowwise (fused sum)."""

    def __init__(self, tp, torch, device, reduce_mode="accum", fused_gather=True):
        cfg = tp_inputs.WORKLOADS[ATTN_PROJ]
        self.tp, self.torch, self.device = tp, torch, device
        self.fused_gather = fused_gather
        self.p, self.T, self.H = cfg["tp"], cfg["tokens"], cfg["hidden"]
        self.heads, self.hd = cfg["heads"], cfg["head_dim"]
        self.mode = reduce_mode
        p, T, H = self.p, self.T, self.H
        w_qkv, w_out, x, a = tp_inputs.attn_proj_inputs(cfg["seed"], T, H)
        self.host = dict(w_qkv=w_qkv, w_out=w_out, x=x, a=a)
        bf = lambda b: tp.bf16_from_bits(b, device)  # noqa: E731
        self.w_qkv = bf(w_qkv)
        self.w_out = bf(w_out)
        self.x = bf(x)
        Kr = H // p
        self.a_sh = [bf(np.ascontiguousarray(a[:, r * Kr:(r + 1) * Kr])) for r in range(p)]
        e = lambda *s: torch.empty(s, dtype=torch.bfloat16, device=device)  # noqa: E731
        self.qkv_sh = [e(3 * H // p, H) for _ in range(p)]
        self.out_sh = [e(H, Kr) for _ in range(p)]
        self.y_sh = [e(T, 3 * H // p) for _ in range(p)]
        self.y = e(T, 3 * H)
        # The AllGather fused into the colwise store: rank r writes columns [r*3H/p, (r+1)*3H/p)
        # of the gathered output directly (row stride 3H).
        self.y_cols = [self.y[:, r * 3 * H // p:(r + 1) * 3 * H // p] for r in range(p)]
        self.z = e(T, H)
        ws = tp.tp_rowwise_workspace_bytes(p, T, H, reduce_mode)
        self.ws = torch.empty(max(ws, 1), dtype=torch.uint8, device=device)
        self.z_part = torch.empty((p, T, H), dtype=torch.float32, device=device) if reduce_mode == "none" else None
        # Algorithmic work per step.
        self.flops_qkv = 2.0 * T * H * 3 * H
        self.flops_out = 2.0 * T * H * H
        self.flops = self.flops_qkv + self.flops_out
        self.extract_bytes = 2.0 * 2 * (3 * H * H + H * H)   # read + write of every shard
        self.gather_bytes = 2.0 * 2 * T * 3 * H
        # The timed step (step()): two extraction launches (the out-projection weight's ranks,
        # then the QKV weight's on a side stream), rowwise, colwise.  Otherwise the phases: one
        # extraction launch, colwise, gather unless fused, rowwise (+ the counter clear of the
        # workspace mode, or the separate reduce of the unfused mode).
        if fused_gather and reduce_mode == "accum":
            self.launches_per_step = 4
        else:
            self.launches_per_step = (3 if fused_gather else 4) + (1 if reduce_mode in ("workspace", "none") else 0)
        # Pinned host copies for the end-to-end measurement.
        self.pin = None

    def config(self):
        return {"workload": ATTN_PROJ, "tokens": self.T, "hidden": self.H, "heads": self.heads, "head_dim": self.hd,
                "tp_degree": self.p, "rowwise_reduce": self.mode,
                "gather": "fused into the colwise store (ldy)" if self.fused_gather else "tp_combine kernel",
                "step": "tp_plan_shard_many (out-projection weight, 4 ranks, from device memory) + "
                        "tp_linear_rowwise, with tp_plan_shard_many (fused QKV weight, 4 ranks) + tp_linear_colwise "
                        "writing the gathered QKV [T, 3H] on a side stream beside it"
                        if self.fused_gather and self.mode == "accum" else
                        "tp_plan_shard_many (both weights, 4 ranks each) + tp_linear_colwise "
                        + ("" if self.fused_gather else "+ tp_combine(gather) ") + "+ tp_linear_rowwise"}

    def phases(self):
        """(label, enqueue function, roofline kind, algorithmic work per step: FLOPs or bytes)."""
        if self.fused_gather:
            return [("extract", self.phase_extract, "hbm", self.extract_bytes),
                    ("colwise_qkv", self.phase_colwise, "tensor", self.flops_qkv),
                    ("rowwise_out", self.phase_rowwise, "tensor", self.flops_out)]
        return [("extract", self.phase_extract, "hbm", self.extract_bytes),
                ("colwise_qkv", self.phase_colwise, "tensor", self.flops_qkv),
                ("gather", self.phase_gather, "hbm", self.gather_bytes),
                ("rowwise_out", self.phase_rowwise, "tensor", self.flops_out)]

    def oracle_step(self, rows):
        return oracle_sample_step(self.host, rows, self.p, self.H, self.heads, self.hd)

    # The four phases of a step, each enqueued on `stream`.
    def _extract_requests(self):
        p, H = self.p, self.H
        return (dict(weight=self.w_qkv, style="colwise", tp_degree=p, fused_splits=[H] * 3, num_heads=self.heads,
                     head_dim=self.hd, outs=self.qkv_sh),
                dict(weight=self.w_out, style="rowwise", tp_degree=p, num_heads=self.heads, head_dim=self.hd,
                     outs=self.out_sh))

    def phase_extract(self, stream):
        # Both weights' shards, every rank, in one launch.
        self.tp.tp_plan_shard_many(list(self._extract_requests()), stream=stream)

    def step(self, stream):
        """One timed step: the phases' work in another order.  The two projections are
        independent here (the out-projection's input is its own activation), so the smaller
        weight's shards are extracted first and its rowwise projection runs while the QKV
        weight's shards are extracted on a side stream, launched after it: the copy runs on
        the SMs that the projection's clusters and its last, partial wave of tiles leave
        idle.  The QKV projection follows its extraction on the side stream, so its CTAs
        take SMs as the out-projection's leave them; the step ends when both are done."""
        if not (self.fused_gather and self.mode == "accum"):
            return run_step(self, stream)
        if getattr(self, "side_stream", None) is None:
            self.side_stream = self.torch.cuda.Stream(self.device)
        side = self.side_stream
        req_qkv, req_out = self._extract_requests()
        self.tp.tp_plan_shard_many([req_out], stream=stream)
        side.wait_stream(stream)
        self.phase_rowwise(stream)
        with self.torch.cuda.stream(side):
            self.tp.tp_plan_shard_many([req_qkv], stream=side)
            self.phase_colwise(side)
        stream.wait_stream(side)

    def phase_colwise(self, stream, x=None):
        x = self.x if x is None else x
        if self.fused_gather:
            self.tp.tp_linear_colwise(x, self.qkv_sh, "none", y_shards=self.y_cols, ldy=3 * self.H, stream=stream)
        else:
            self.tp.tp_linear_colwise(x, self.qkv_sh, "none", y_shards=self.y_sh, stream=stream)

    def phase_gather(self, stream):
        self.tp.tp_combine("gather", self.y_sh, out=self.y, stream=stream)

    def phase_rowwise(self, stream):
        self._rowwise(self.a_sh, stream)

    def join_phases(self):
        """The two joins as separate kernels, timed beside the step: the AllGather of the QKV
        slices and the AllReduce of fp32 rowwise partials (the unfused forms)."""
        torch, p, T, H = self.torch, self.p, self.T, self.H
        if getattr(self, "_join_parts", None) is None:
            self._join_parts = torch.zeros((p, T, H), dtype=torch.float32, device=self.device)
            self._join_out = torch.empty((T, H), dtype=torch.bfloat16, device=self.device)
        parts, out = self._join_parts, self._join_out
        return [("gather", lambda st: self.tp.tp_combine("gather", self.y_sh, out=self.y, stream=st),
                 self.gather_bytes),
                ("reduce", lambda st: self.tp.tp_combine("reduce", list(parts), out=out, stream=st),
                 4.0 * p * T * H + 2.0 * T * H)]

    def reference_points(self):
        """Library and framework equivalents of the step's kernels, timed beside it (reference
        points, not targets): cuBLAS (torch.matmul) on the unsharded projections and torch's
        strided copy for the rowwise extraction."""
        torch, p, H = self.torch, self.p, self.H
        if getattr(self, "_ref_bufs", None) is None:
            a_full = torch.cat(self.a_sh, dim=1)
            self._ref_bufs = (a_full, torch.empty_like(self.y), torch.empty_like(self.z))
        a_full, y_ref, z_ref = self._ref_bufs
        Kr = H // p
        return [
            ("cublas_colwise_qkv", lambda st: torch.matmul(self.x, self.w_qkv.t(), out=y_ref), "tensor",
             self.flops_qkv),
            ("cublas_rowwise_out", lambda st: torch.matmul(a_full, self.w_out.t(), out=z_ref), "tensor",
             self.flops_out),
            ("torch_rowwise_extract", lambda st: [self.out_sh[r].copy_(self.w_out[:, r * Kr:(r + 1) * Kr])
                                                  for r in range(p)], "hbm", 2.0 * 2 * H * H),
        ]

    def _rowwise(self, a_sh, stream):
        tp = self.tp
        if self.mode == "none":
            tp.tp_linear_rowwise(a_sh, self.out_sh, mode="none", out=self.z_part, stream=stream)
            tp.tp_combine("reduce", list(self.z_part), out=self.z, stream=stream)
        else:
            tp.tp_linear_rowwise(a_sh, self.out_sh, mode=self.mode, workspace=self.ws, out=self.z, stream=stream)

    # -- end to end: host buffers in, result out --------------------------------------------------
    def setup_e2e(self):
        torch = self.torch
        pin = lambda b: torch.empty(b.shape, dtype=torch.bfloat16, pin_memory=True).copy_(  # noqa: E731
            self.tp.bf16_from_bits(b))
        Kr = self.H // self.p
        self.pin = dict(
            w_qkv=pin(self.host["w_qkv"]), w_out=pin(self.host["w_out"]), x=pin(self.host["x"]),
            a_sh=[pin(np.ascontiguousarray(self.host["a"][:, r * Kr:(r + 1) * Kr])) for r in range(self.p)],
            a=pin(self.host["a"]),
            z=torch.empty((self.T, self.H), dtype=torch.bfloat16, pin_memory=True))
        self.x_in = torch.empty_like(self.x)
        self.a_in = [torch.empty_like(t) for t in self.a_sh]
        # The pipelined step keeps every rank's A_r side by side in one [T, H] buffer (rank r's
        # columns [r*H/p, (r+1)*H/p)), so a block of rows of all ranks is one copy.
        self.a_in_cat = torch.empty((self.T, self.H), dtype=torch.bfloat16, device=self.device)
        # The step's inputs are its activations; its result is Z.
        self.h2d_bytes = self.pin["x"].numel() * 2 + sum(t.numel() * 2 for t in self.pin["a_sh"])
        self.d2h_bytes = self.pin["z"].numel() * 2
        # Variant: the weights too come from host memory every step (shard-on-read).
        self.h2d_bytes_weights = (self.pin["w_qkv"].numel() + self.pin["w_out"].numel()) * 2

    def step_e2e(self, stream, weights_from_host=False):
        """One step through the public calls: activations in from page-locked host memory, Z out.

        The weights stay in device memory (a serving process loads them once) and every rank's
        shard is extracted from them as in the device-timed step; with weights_from_host, each
        rank's slice is read from page-locked host memory instead (shard-on-read every step).
        """
        tp, p, H, torch = self.tp, self.p, self.H, self.torch
        if getattr(self, "copy_stream", None) is None:
            self.copy_stream = torch.cuda.Stream(self.device)
        # X first on the compute stream (the QKV projection needs it); the rowwise inputs A_r on a
        # second stream, overlapping the extraction and the QKV projection.
        with torch.cuda.stream(stream):
            self.x_in.copy_(self.pin["x"], non_blocking=True)
        self.copy_stream.wait_stream(stream)
        with torch.cuda.stream(self.copy_stream):
            for dst, src in zip(self.a_in, self.pin["a_sh"]):
                dst.copy_(src, non_blocking=True)
        w_qkv = self.pin["w_qkv"] if weights_from_host else self.w_qkv
        w_out = self.pin["w_out"] if weights_from_host else self.w_out
        tp.tp_plan_shard_many([
            dict(weight=w_qkv, style="colwise", tp_degree=p, fused_splits=[H] * 3, num_heads=self.heads,
                 head_dim=self.hd, outs=self.qkv_sh),
            dict(weight=w_out, style="rowwise", tp_degree=p, num_heads=self.heads, head_dim=self.hd,
                 outs=self.out_sh)], stream=stream)
        self.phase_colwise(stream, self.x_in)
        if not self.fused_gather:
            tp.tp_combine("gather", self.y_sh, out=self.y, stream=stream)
        stream.wait_stream(self.copy_stream)
        self._rowwise(self.a_in, stream)
        with torch.cuda.stream(stream):
            self.pin["z"].copy_(self.z, non_blocking=True)

    def step_e2e_chunked(self, stream, a_rows=(4096,), x_rows=(2048, 2048)):
        """The e2e step pipelined over token row blocks, so that the copies overlap the compute.

        A copy stream moves A in (every rank's A_r side by side, blocks of `a_rows` rows), then X
        (blocks of `x_rows` rows); the compute stream runs the out-projection of each A block as
        soon as it has landed (tp_linear_rowwise_split_input: rank r's slice is its columns) and
        a third stream reads that block of Z back at once, while X is still on the way; then the
        QKV projection of each X block.  The gathered QKV stays on the device, so once the last,
        small X block has landed only its projection is left.  The same public calls on row
        blocks of the same buffers; Z is bit-identical to the device-resident step's."""
        tp, p, H, T, torch = self.tp, self.p, self.H, self.T, self.torch
        if getattr(self, "copy_stream", None) is None:
            self.copy_stream = torch.cuda.Stream(self.device)
        if getattr(self, "d2h_stream", None) is None:
            self.d2h_stream = torch.cuda.Stream(self.device)
        cs, ds = self.copy_stream, self.d2h_stream

        def blocks(rows):
            assert sum(rows) == T and min(rows) > 0
            ends = np.cumsum(rows).tolist()
            return [(e - r, e) for r, e in zip(rows, ends)]
        ab, xb = blocks(a_rows), blocks(x_rows)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        ea, ez, ex = [ev() for _ in ab], [ev() for _ in ab], [ev() for _ in xb]
        cs.wait_stream(stream)
        with torch.cuda.stream(cs):
            for i, (r0, r1) in enumerate(ab):
                self.a_in_cat[r0:r1].copy_(self.pin["a"][r0:r1], non_blocking=True)
                ea[i].record(cs)
            for i, (r0, r1) in enumerate(xb):
                self.x_in[r0:r1].copy_(self.pin["x"][r0:r1], non_blocking=True)
                ex[i].record(cs)
        tp.tp_plan_shard_many([
            dict(weight=self.w_qkv, style="colwise", tp_degree=p, fused_splits=[H] * 3, num_heads=self.heads,
                 head_dim=self.hd, outs=self.qkv_sh),
            dict(weight=self.w_out, style="rowwise", tp_degree=p, num_heads=self.heads, head_dim=self.hd,
                 outs=self.out_sh)], stream=stream)
        ds.wait_stream(stream)
        for i, (r0, r1) in enumerate(ab):
            stream.wait_event(ea[i])
            tp.tp_linear_rowwise_split_input(self.a_in_cat[r0:r1], self.out_sh, mode="accum", out=self.z[r0:r1],
                                             stream=stream)
            ez[i].record(stream)
            ds.wait_event(ez[i])
            with torch.cuda.stream(ds):
                self.pin["z"][r0:r1].copy_(self.z[r0:r1], non_blocking=True)
        for i, (r0, r1) in enumerate(xb):
            stream.wait_event(ex[i])
            tp.tp_linear_colwise(self.x_in[r0:r1], self.qkv_sh, "none", y_shards=[y[r0:r1] for y in self.y_cols],
                                 ldy=3 * H, stream=stream)
        stream.wait_stream(ds)


def side_stream(wl):
    """The workload's second stream (for work that overlaps the main stream's within a step)."""
    if getattr(wl, "side_stream", None) is None:
        wl.side_stream = wl.torch.cuda.Stream(wl.device)
    return wl.side_stream


def whole_step(wl, stream):
    """Enqueue one timed step of `wl`: its own step() where it has one, else its phases in order."""
    if hasattr(wl, "step"):
        wl.step(stream)
    else:
        run_step(wl, stream)


def run_step(wl, stream, marks=None):
    """Enqueue one step of `wl` on `stream`; `marks` (one more event than phases) bracket the phases."""
    for i, (_, fn, _, _) in enumerate(wl.phases()):
        if marks:
            marks[i].record(stream)
        fn(stream)
    if marks:
        marks[-1].record(stream)


class MlpWorkload:
    """One MLP block: colwise in-projection with its activation, rowwise out-projection summed on chip.

    tiny_mlp_tp2: hidden 256, ffn 1024, 64 tokens, GELU(tanh), tp 2.
    swiglu_mlp_tp4: hidden 6144, ffn 18432 (fused gate/up [36864, 6144]), 4608 tokens, SwiGLU, tp 4.
    """

    def __init__(self, tp, torch, device, name):
        cfg = tp_inputs.WORKLOADS[name]
        self.name, self.tp, self.torch, self.device = name, tp, torch, device
        self.p, self.T, self.H, self.F = cfg["tp"], cfg["tokens"], cfg["hidden"], cfg["ffn"]
        self.heads, self.act = cfg["heads"], cfg["act"]
        p, T, H, F = self.p, self.T, self.H, self.F
        if self.act == "swiglu":
            w_in, w_out, x = tp_inputs.swiglu_mlp_inputs(cfg["seed"], T, H, F)
            self.splits, n_in = [F, F], 2 * F
        else:
            w_in, w_out, x = tp_inputs.tiny_mlp_inputs(cfg["seed"], T, H, F)
            self.splits, n_in = None, F
        self.host = dict(w_in=w_in, w_out=w_out, x=x)
        bf = lambda b: tp.bf16_from_bits(b, device)  # noqa: E731
        self.w_in, self.w_out, self.x = bf(w_in), bf(w_out), bf(x)
        e = lambda *sh: torch.empty(sh, dtype=torch.bfloat16, device=device)  # noqa: E731
        self.in_sh = [e(n_in // p, H) for _ in range(p)]
        self.out_sh = [e(H, F // p) for _ in range(p)]
        self.h_sh = [e(T, F // p) for _ in range(p)]
        self.z = e(T, H)
        self.flops_in = 2.0 * T * H * n_in
        self.flops_out = 2.0 * T * F * H
        self.flops = self.flops_in + self.flops_out
        self.extract_bytes = 2.0 * 2 * (n_in * H + H * F)
        self.launches_per_step = 4  # two extraction launches in the timed step (step()), two projections

    def config(self):
        return {"workload": self.name, "tokens": self.T, "hidden": self.H, "ffn": self.F, "act": self.act,
                "tp_degree": self.p, "rowwise_reduce": "accum",
                "step": "tp_plan_shard_many (in-projection weight, device) + tp_linear_colwise (act), with "
                        "tp_plan_shard_many (down-projection weight) on a side stream beside it + tp_linear_rowwise"}

    def _extract_requests(self):
        p = self.p
        return [dict(weight=self.w_in, style="colwise", tp_degree=p, fused_splits=self.splits, num_heads=self.heads,
                     outs=self.in_sh),
                dict(weight=self.w_out, style="rowwise", tp_degree=p, num_heads=self.heads, outs=self.out_sh)]

    def phase_extract(self, stream):
        self.tp.tp_plan_shard_many(self._extract_requests(), stream=stream)

    def step(self, stream):
        """One timed step: the phases' work, with the down-projection weight's shards extracted on
        a side stream launched after the in-projection (the copy, bound by HBM, runs beside it);
        the down-projection waits for them."""
        side = side_stream(self)
        req_in, req_out = self._extract_requests()
        self.tp.tp_plan_shard_many([req_in], stream=stream)
        side.wait_stream(stream)
        self.phase_colwise(stream)
        with self.torch.cuda.stream(side):
            self.tp.tp_plan_shard_many([req_out], stream=side)
        stream.wait_stream(side)
        self.phase_rowwise(stream)

    def phase_colwise(self, stream):
        self.tp.tp_linear_colwise(self.x, self.in_sh, self.act, y_shards=self.h_sh, stream=stream)

    def phase_rowwise(self, stream):
        self.tp.tp_linear_rowwise(self.h_sh, self.out_sh, mode="accum", out=self.z, stream=stream)

    def phases(self):
        return [("extract", self.phase_extract, "hbm", self.extract_bytes),
                ("colwise_" + self.act, self.phase_colwise, "tensor", self.flops_in),
                ("rowwise_down", self.phase_rowwise, "tensor", self.flops_out)]

    def reference_points(self):
        """cuBLAS (torch.matmul) on the unsharded in- and out-projections: the same FLOPs as the
        two projection phases (reference points, not targets: no activation, no sharding)."""
        torch = self.torch
        if getattr(self, "_ref_bufs", None) is None:
            y = torch.empty((self.T, self.w_in.shape[0]), dtype=torch.bfloat16, device=self.device)
            h = torch.empty((self.T, self.F), dtype=torch.bfloat16, device=self.device).normal_()
            z = torch.empty((self.T, self.H), dtype=torch.bfloat16, device=self.device)
            self._ref_bufs = (y, h, z)
        y, h, z = self._ref_bufs
        return [("cublas_colwise", lambda st: torch.matmul(self.x, self.w_in.t(), out=y), "tensor", self.flops_in),
                ("cublas_rowwise_down", lambda st: torch.matmul(h, self.w_out.t(), out=z), "tensor",
                 self.flops_out)]

    def oracle_step(self, rows):
        from oracle import tp_oracle as O
        p, h = self.p, self.host
        w_in = [O.shard(h["w_in"], "colwise", p, r, self.splits) for r in range(p)]
        w_out = [O.shard(h["w_out"], "rowwise", p, r) for r in range(p)]
        return O.mlp_forward(h["x"][rows], w_in, w_out, self.act)[1]


class BlockWorkload:
    """The full attention + SwiGLU MLP block (hidden 6144, 48 heads x 128, ffn 18432, 4608 tokens) at one tp."""

    def __init__(self, tp, torch, device, p):
        cfg = tp_inputs.WORKLOADS["block_sweep"]
        self.tp, self.torch, self.device = tp, torch, device
        self.p, self.T, self.H, self.F = p, cfg["tokens"], cfg["hidden"], cfg["ffn"]
        self.heads, self.hd = cfg["heads"], cfg["head_dim"]
        tp.tp_validate(3 * self.H, self.H, "colwise", p, self.heads, self.hd, [self.H] * 3)  # 5 and 7 raise here
        T, H, F, hl = self.T, self.H, self.F, self.heads // p
        wqkv, wout, wgu, wdown, x = tp_inputs.block_inputs(cfg["seed"], T, H, F)
        self.host = dict(wqkv=wqkv, wout=wout, wgu=wgu, wdown=wdown, x=x)
        bf = lambda b: tp.bf16_from_bits(b, device)  # noqa: E731
        self.w = {k: bf(v) for k, v in self.host.items() if k != "x"}
        self.x = bf(x)
        e = lambda *sh: torch.empty(sh, dtype=torch.bfloat16, device=device)  # noqa: E731
        self.qkv_sh = [e(3 * H // p, H) for _ in range(p)]
        self.out_sh = [e(H, H // p) for _ in range(p)]
        self.gu_sh = [e(2 * F // p, H) for _ in range(p)]
        self.dn_sh = [e(H, F // p) for _ in range(p)]
        self.y_sh = [e(T, 3 * H // p) for _ in range(p)]
        self.o_sh = [e(T, H // p) for _ in range(p)]
        self.z1 = e(T, H)
        self.h_sh = [e(T, F // p) for _ in range(p)]
        self.z = e(T, H)
        self.attn_ws = torch.empty(tp.tp_attention_ranks_workspace_bytes(p, T, hl, self.hd), dtype=torch.uint8,
                                   device=device)
        self.fl = dict(qkv=2.0 * T * H * 3 * H, attn=4.0 * T * T * self.hd * self.heads, out=2.0 * T * H * H,
                       gu=2.0 * T * H * 2 * F, down=2.0 * T * F * H)
        self.flops = sum(self.fl.values())
        self.extract_bytes = 2.0 * 2 * (4 * H * H + 3 * H * F)
        # Two extraction launches in the timed step (step()), the QKV projection, the attention,
        # three more projections.
        self.launches_per_step = 2 + 1 + attention_launches(p, hl, self.hd) + 3

    def config(self):
        return {"workload": "block_sweep", "tokens": self.T, "hidden": self.H, "ffn": self.F, "heads": self.heads,
                "head_dim": self.hd, "tp_degree": self.p, "rowwise_reduce": "accum",
                "flops": "projections + attention core (4*T^2*head_dim per head)",
                "step": "tp_plan_shard_many (QKV weight) + QKV colwise, with tp_plan_shard_many (the other 3 weights) "
                        "on a side stream beside it + tp_attention_heads_ranks (every rank) + out rowwise + "
                        "gate/up colwise SwiGLU + down rowwise"}

    def _extract_requests(self):
        p, H, F = self.p, self.H, self.F
        return [dict(weight=self.w["wqkv"], style="colwise", tp_degree=p, fused_splits=[H] * 3, num_heads=self.heads,
                     head_dim=self.hd, outs=self.qkv_sh),
                dict(weight=self.w["wout"], style="rowwise", tp_degree=p, num_heads=self.heads, head_dim=self.hd,
                     outs=self.out_sh),
                dict(weight=self.w["wgu"], style="colwise", tp_degree=p, fused_splits=[F, F], num_heads=self.heads,
                     outs=self.gu_sh),
                dict(weight=self.w["wdown"], style="rowwise", tp_degree=p, num_heads=self.heads, outs=self.dn_sh)]

    def phase_extract(self, stream):
        # The block's four weights, every rank, in one launch.
        self.tp.tp_plan_shard_many(self._extract_requests(), stream=stream)

    def step(self, stream):
        """One timed step: the phases' work, with only the QKV weight's shards extracted before
        the QKV projection; the other three weights' shards are extracted on a side stream
        launched after it, so the copy (bound by HBM) runs beside the projection (bound by the
        tensor cores) and the attention; the out-projection waits for it."""
        side = side_stream(self)
        reqs = self._extract_requests()
        self.tp.tp_plan_shard_many(reqs[:1], stream=stream)
        side.wait_stream(stream)
        self.phase_qkv(stream)
        with self.torch.cuda.stream(side):
            self.tp.tp_plan_shard_many(reqs[1:], stream=side)
        self.phase_attention(stream)
        stream.wait_stream(side)
        self.phase_out(stream)
        self.phase_gate_up(stream)
        self.phase_down(stream)

    def phase_qkv(self, stream):
        # Q, K and V feed the softmax: chunked fp32 accumulation (TP_ACCUM_CHUNKED).
        self.tp.tp_linear_colwise(self.x, self.qkv_sh, "none", y_shards=self.y_sh, stream=stream, chunked=True)

    def phase_attention(self, stream):
        self.tp.tp_attention_heads_ranks(self.y_sh, self.heads // self.p, self.hd, outs=self.o_sh,
                                         workspace=self.attn_ws, stream=stream)

    def phase_out(self, stream):
        self.tp.tp_linear_rowwise(self.o_sh, self.out_sh, mode="accum", out=self.z1, stream=stream)

    def phase_gate_up(self, stream):
        self.tp.tp_linear_colwise(self.z1, self.gu_sh, "swiglu", y_shards=self.h_sh, stream=stream)

    def phase_down(self, stream):
        self.tp.tp_linear_rowwise(self.h_sh, self.dn_sh, mode="accum", out=self.z, stream=stream)

    def phases(self):
        return [("extract", self.phase_extract, "hbm", self.extract_bytes),
                ("colwise_qkv", self.phase_qkv, "tensor", self.fl["qkv"]),
                ("attention", self.phase_attention, "tensor", self.fl["attn"]),
                ("rowwise_out", self.phase_out, "tensor", self.fl["out"]),
                ("colwise_swiglu", self.phase_gate_up, "tensor", self.fl["gu"]),
                ("rowwise_down", self.phase_down, "tensor", self.fl["down"])]

    def oracle_step(self, rows):
        from oracle import tp_oracle as O
        p, h, H, F = self.p, self.host, self.H, self.F
        return O.transformer_block_forward(
            h["x"], [O.shard(h["wqkv"], "colwise", p, r, [H] * 3) for r in range(p)],
            [O.shard(h["wout"], "rowwise", p, r) for r in range(p)],
            [O.shard(h["wgu"], "colwise", p, r, [F, F]) for r in range(p)],
            [O.shard(h["wdown"], "rowwise", p, r) for r in range(p)],
            n_local_heads=self.heads // p, head_dim=self.hd, q_rows=rows)["z"]


def attention_launches(ranks, local_heads, head_dim):
    """Kernels one tp_attention_heads_ranks call launches: one fused kernel for every rank at
    head_dim 64 or 128, else per rank V^T plus scores / softmax / PV per 16 heads."""
    if head_dim in (64, 128):
        return 1
    return ranks * (1 + 3 * ((local_heads + 15) // 16))


class SingleStreamWorkload:
    """The single-stream block (hidden 6144, 48 heads x 128, mlp_ratio 3, 4608 tokens): one fused
    [1,1,1,3,3] in-projection (colwise) and the packed [inner, mlp] out-projection (rowwise)."""

    def __init__(self, tp, torch, device, p=None):
        cfg = tp_inputs.WORKLOADS["single_stream_tp4"]
        self.tp, self.torch, self.device = tp, torch, device
        self.p = p = p or cfg["tp"]
        self.T, self.H, self.heads, self.hd = cfg["tokens"], cfg["hidden"], cfg["heads"], cfg["head_dim"]
        self.F = F = cfg["mlp_ratio"] * self.H
        T, H = self.T, self.H
        self.splits_in, self.splits_out = [H, H, H, F, F], [H, F]
        tp.tp_validate(3 * H + 2 * F, H, "colwise", p, self.heads, 0, self.splits_in)
        w_in, w_out, x = tp_inputs.single_stream_inputs(cfg["seed"], T, H, cfg["mlp_ratio"])
        self.host = dict(w_in=w_in, w_out=w_out, x=x)
        bf = lambda b: tp.bf16_from_bits(b, device)  # noqa: E731
        self.w_in, self.w_out, self.x = bf(w_in), bf(w_out), bf(x)
        e = lambda *sh: torch.empty(sh, dtype=torch.bfloat16, device=device)  # noqa: E731
        w, f = H // p, F // p
        self.w, self.f = w, f
        self.in_sh = [e(3 * w + 2 * f, H) for _ in range(p)]
        self.out_sh = [e(H, w + f) for _ in range(p)]
        self.qkv = [e(T, 3 * w) for _ in range(p)]
        self.cat = [e(T, w + f) for _ in range(p)]      # [attention_r, mlp_r]: rank r's out-projection input
        self.z = e(T, H)
        self.attn_ws = torch.empty(tp.tp_attention_ranks_workspace_bytes(p, T, self.heads // p, self.hd),
                                   dtype=torch.uint8, device=device)
        self.fl = dict(qkv=2.0 * T * H * 3 * H, gu=2.0 * T * H * 2 * F, attn=4.0 * T * T * H,
                       out=2.0 * T * (H + F) * H)
        self.flops = sum(self.fl.values())
        self.extract_bytes = 2.0 * 2 * ((3 * H + 2 * F) * H + H * (H + F))
        # Two extraction launches in the timed step (step()), two colwise launches, the attention,
        # the rowwise out-projection.
        self.launches_per_step = 2 + 2 + attention_launches(p, self.heads // p, self.hd) + 1

    def config(self):
        return {"workload": "single_stream_tp4", "tokens": self.T, "hidden": self.H, "mlp_hidden": self.F,
                "heads": self.heads, "head_dim": self.hd, "tp_degree": self.p, "rowwise_reduce": "accum",
                "flops": "projections + attention core (4*T^2*head_dim per head)",
                "step": "tp_plan_shard_many (Q/K/V blocks of the packed [1,1,1,3,3] colwise weight) + colwise "
                        "Q/K/V rows, with tp_plan_shard_many (its gate/up blocks, packed [inner, mlp] rowwise) on a "
                        "side stream beside it + tp_attention_heads_ranks into [attention, mlp] + colwise SwiGLU "
                        "gate/up rows into [attention, mlp] + packed rowwise to_out"}

    def phase_extract(self, stream):
        # Both packed weights, every rank, in one launch.
        tp, p = self.tp, self.p
        tp.tp_plan_shard_many([
            dict(weight=self.w_in, style="colwise", tp_degree=p, fused_splits=self.splits_in, num_heads=self.heads,
                 outs=self.in_sh),
            dict(weight=self.w_out, style="rowwise", tp_degree=p, fused_splits=self.splits_out, num_heads=self.heads,
                 outs=self.out_sh)], stream=stream)

    def step(self, stream):
        """One timed step: the phases' work, with only the Q/K/V blocks of the packed in-projection
        weight extracted before the Q/K/V projection.  Its gate/up blocks and the out-projection
        weight are extracted on a side stream launched after that projection (the copy, bound by
        HBM, runs beside it and the attention, which needs only Q/K/V); the gate/up projection
        waits for them.  A rank's packed shard is
        its Q/K/V rows followed by its gate/up rows, so the two partial plans (blocks [H, H, H]
        of rows [0, 3H), blocks [F, F] of the rest) fill the same shard buffers, bit for bit."""
        tp, p, H, w = self.tp, self.p, self.H, self.w
        side = side_stream(self)
        tp.tp_plan_shard_many([
            dict(weight=self.w_in[:3 * H], style="colwise", tp_degree=p, fused_splits=[H] * 3, num_heads=self.heads,
                 outs=[s[:3 * w] for s in self.in_sh])], stream=stream)
        side.wait_stream(stream)
        self.phase_qkv(stream)
        with self.torch.cuda.stream(side):
            tp.tp_plan_shard_many([
                dict(weight=self.w_in[3 * H:], style="colwise", tp_degree=p, fused_splits=self.splits_in[3:],
                     num_heads=self.heads, outs=[s[3 * w:] for s in self.in_sh]),
                dict(weight=self.w_out, style="rowwise", tp_degree=p, fused_splits=self.splits_out,
                     num_heads=self.heads, outs=self.out_sh)], stream=side)
        self.phase_attention(stream)
        stream.wait_stream(side)
        self.phase_gate_up(stream)
        self.phase_out(stream)

    def phase_qkv(self, stream):
        # Q, K and V feed the softmax: chunked fp32 accumulation (TP_ACCUM_CHUNKED).
        self.tp.tp_linear_colwise(self.x, [s[:3 * self.w] for s in self.in_sh], "none", y_shards=self.qkv,
                                  stream=stream, chunked=True)

    def phase_gate_up(self, stream):
        self.tp.tp_linear_colwise(self.x, [s[3 * self.w:] for s in self.in_sh], "swiglu",
                                  y_shards=[c[:, self.w:] for c in self.cat], ldy=self.w + self.f, stream=stream)

    def phase_attention(self, stream):
        self.tp.tp_attention_heads_ranks(self.qkv, self.heads // self.p, self.hd, outs=[c[:, :self.w] for c in self.cat],
                                         workspace=self.attn_ws, stream=stream)

    def phase_out(self, stream):
        self.tp.tp_linear_rowwise(self.cat, self.out_sh, mode="accum", out=self.z, stream=stream)

    def phases(self):
        return [("extract", self.phase_extract, "hbm", self.extract_bytes),
                ("colwise_qkv", self.phase_qkv, "tensor", self.fl["qkv"]),
                ("colwise_swiglu", self.phase_gate_up, "tensor", self.fl["gu"]),
                ("attention", self.phase_attention, "tensor", self.fl["attn"]),
                ("rowwise_out", self.phase_out, "tensor", self.fl["out"])]

    def oracle_step(self, rows):
        from oracle import tp_oracle as O
        p, h = self.p, self.host
        return O.single_stream_block_forward(
            h["x"], [O.shard(h["w_in"], "colwise", p, r, self.splits_in) for r in range(p)],
            [O.shard(h["w_out"], "rowwise", p, r, self.splits_out) for r in range(p)],
            n_local_heads=self.heads // p, head_dim=self.hd, q_rows=rows)["z"]


class StackWorkload:
    """Eight SwiGLU MLP blocks (hidden 6144, ffn 18432, tp 4) from a page-locked host state dict.

    The shards are loaded once (shard-on-read, every rank's slice of every weight
    straight from host memory); a step is the forward pass through the 8 blocks.
    Block b reads the previous block's output (x for block 0) and writes one of two
    ping-pong buffers.
    """

    def __init__(self, tp, torch, device):
        cfg = tp_inputs.WORKLOADS[WORKLOAD]
        self.tp, self.torch, self.device = tp, torch, device
        self.p, self.nb, self.T, self.H, self.F = cfg["tp"], cfg["blocks"], cfg["tokens"], cfg["hidden"], cfg["ffn"]
        self.heads, self.seed = cfg["heads"], cfg["seed"]
        p, H, F, T = self.p, self.H, self.F, self.T
        # The seeded state dict: 16 tensors, generated side by side (numpy releases the GIL).
        jobs = [(b, which) for b in range(self.nb) for which in ("gate_up", "down")]
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            bits = list(ex.map(lambda j: tp_inputs.stack_weight(self.seed, j[0], j[1], H, F), jobs))
        self.host_bits = [(bits[2 * b], bits[2 * b + 1]) for b in range(self.nb)]
        pin = lambda b: torch.empty(b.shape, dtype=torch.bfloat16, pin_memory=True).copy_(  # noqa: E731
            tp.bf16_from_bits(b))
        self.host = [(pin(gu), pin(dn)) for gu, dn in self.host_bits]
        self.x_bits = tp_inputs.stack_input(self.seed, self.nb, T, H)
        self.x_pin = pin(self.x_bits)
        self.x = tp.bf16_from_bits(self.x_bits, device)
        self.z_pin = torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True)
        e = lambda *sh: torch.empty(sh, dtype=torch.bfloat16, device=device)  # noqa: E731
        self.shards = [([e(2 * F // p, H) for _ in range(p)], [e(H, F // p) for _ in range(p)])
                       for _ in range(self.nb)]
        self.h = [e(T, F // p) for _ in range(p)]
        self.zbuf = [e(T, H), e(T, H)]
        self.z = self.zbuf[(self.nb - 1) % 2]          # the last block's output
        self.x_in = e(T, H)
        self.shard_bytes = self.nb * (2 * F * H + H * F) * 2
        self.fl_gu = 2.0 * T * H * 2 * F
        self.fl_dn = 2.0 * T * F * H
        self.flops = self.nb * (self.fl_gu + self.fl_dn)
        self.launches_per_step = 2 * self.nb
        self.copy_stream = None

    def config(self):
        return {"workload": WORKLOAD, "blocks": self.nb, "tokens": self.T, "hidden": self.H, "ffn": self.F,
                "heads": self.heads, "tp_degree": self.p, "rowwise_reduce": "accum",
                "weights": f"{self.shard_bytes / 1e9:.2f} GB of bf16 shards (2.72B parameters)",
                "step": "8 x (tp_linear_colwise SwiGLU + tp_linear_rowwise accum), shards resident in HBM"}

    # -- shard-on-read ----------------------------------------------------------------------------
    def load_block(self, b, stream, after_gate_up=None):
        """Every rank's slices of block b's two weights, gate/up first (`after_gate_up`, an
        event, is recorded between the two)."""
        tp, p, F = self.tp, self.p, self.F
        gu, dn = self.host[b]
        gu_sh, dn_sh = self.shards[b]
        tp.tp_plan_shard_ranks(gu, "colwise", p, 0, p, [F, F], self.heads, 0, outs=gu_sh, stream=stream)
        if after_gate_up is not None:
            after_gate_up.record(stream)
        tp.tp_plan_shard_ranks(dn, "rowwise", p, 0, p, None, self.heads, 0, outs=dn_sh, stream=stream)

    def load(self, stream):
        for b in range(self.nb):
            self.load_block(b, stream)

    # -- the forward pass -------------------------------------------------------------------------
    def block_input(self, b, x=None):
        if b == 0:
            return self.x if x is None else x
        return self.zbuf[(b - 1) % 2]

    def gate_up(self, b, stream, x=None):
        self.tp.tp_linear_colwise(self.block_input(b, x), self.shards[b][0], "swiglu", y_shards=self.h,
                                  stream=stream)

    def down(self, b, stream):
        self.tp.tp_linear_rowwise(self.h, self.shards[b][1], mode="accum", out=self.zbuf[b % 2], stream=stream)

    def forward(self, stream, x=None):
        for b in range(self.nb):
            self.gate_up(b, stream, x)
            self.down(b, stream)
        return self.z

    def step(self, stream):
        self.forward(stream)

    def phases(self):
        out = []
        for b in range(self.nb):
            out.append(("colwise_swiglu", lambda st, b=b: self.gate_up(b, st), "tensor", self.fl_gu))
            out.append(("rowwise_down", lambda st, b=b: self.down(b, st), "tensor", self.fl_dn))
        return out

    def reference_points(self):
        """cuBLAS (torch.matmul) on block 0's unsharded projections, the same FLOPs as the two
        phases (a reference point, not a target: no SwiGLU, no sharding, no join)."""
        torch = self.torch
        if getattr(self, "_ref_bufs", None) is None:
            gu, dn = self.host[0]
            w_gu, w_dn = gu.to(self.device), dn.to(self.device)
            y = torch.empty((self.T, 2 * self.F), dtype=torch.bfloat16, device=self.device)
            h = torch.empty((self.T, self.F), dtype=torch.bfloat16, device=self.device).normal_()
            z = torch.empty((self.T, self.H), dtype=torch.bfloat16, device=self.device)
            self._ref_bufs = (w_gu, w_dn, y, h, z)
        w_gu, w_dn, y, h, z = self._ref_bufs
        return [("cublas_gate_up", lambda st: torch.matmul(self.x, w_gu.t(), out=y), "tensor", self.fl_gu),
                ("cublas_down", lambda st: torch.matmul(h, w_dn.t(), out=z), "tensor", self.fl_dn)]

    # -- end to end: every step from host memory ----------------------------------------------------
    def step_e2e(self, stream, pipelined=True):
        """One step through the public calls with host buffers: every rank's slice of every weight
        read from the page-locked state dict (shard-on-read), the input copied in, the 8 blocks,
        the output copied back.  Pipelined: the input and the blocks' slices arrive in block order
        on a copy stream; block b's gate/up projection starts as soon as its gate/up slices
        have landed and its down-projection once its down slices have, so the compute overlaps
        the transfer of the later slices (the last block's gate/up, that of its own down
        weight).  Unpipelined: the same calls one after another on one stream."""
        torch = self.torch
        if not pipelined:
            self.load(stream)
            with torch.cuda.stream(stream):
                self.x_in.copy_(self.x_pin, non_blocking=True)
            self.forward(stream, self.x_in)
            with torch.cuda.stream(stream):
                self.z_pin.copy_(self.z, non_blocking=True)
            return
        if self.copy_stream is None:
            self.copy_stream = torch.cuda.Stream(self.device)
        cs = self.copy_stream
        ex = torch.cuda.Event()
        egu = [torch.cuda.Event() for _ in range(self.nb)]
        edn = [torch.cuda.Event() for _ in range(self.nb)]
        cs.wait_stream(stream)
        with torch.cuda.stream(cs):
            self.x_in.copy_(self.x_pin, non_blocking=True)
            ex.record(cs)
            for b in range(self.nb):
                self.load_block(b, cs, after_gate_up=egu[b])
                edn[b].record(cs)
        stream.wait_event(ex)
        for b in range(self.nb):
            stream.wait_event(egu[b])
            self.gate_up(b, stream, self.x_in)
            stream.wait_event(edn[b])
            self.down(b, stream)
        with torch.cuda.stream(stream):
            self.z_pin.copy_(self.z, non_blocking=True)

    def step_e2e_resident(self, stream):
        """One serving step through the public calls with the shards already loaded: the input
        copied in from page-locked host memory, the 8 blocks, the output copied back."""
        torch = self.torch
        with torch.cuda.stream(stream):
            self.x_in.copy_(self.x_pin, non_blocking=True)
        self.forward(stream, self.x_in)
        with torch.cuda.stream(stream):
            self.z_pin.copy_(self.z, non_blocking=True)

    # -- the oracle on sampled rows -----------------------------------------------------------------
    def oracle_block(self, b, x_bits):
        """The oracle's block b on the given input rows: every rank's shards extracted from the
        host state dict, then the SwiGLU MLP block.  Returns the output's bf16 bits."""
        from oracle import tp_oracle as O
        p, F = self.p, self.F
        gu, dn = self.host_bits[b]
        with np.errstate(all="ignore"):   # the stacked values leave the bf16 range after block 4
            _, z = O.mlp_forward(x_bits, [O.shard(gu, "colwise", p, r, [F, F]) for r in range(p)],
                                 [O.shard(dn, "rowwise", p, r) for r in range(p)], "swiglu")
            return O.f64_to_bf16(z)


# ----------------------------------------------------------------------------- CPU oracle timing

def stack_cpu_baseline(wl, n_rows=512):
    """The oracle through all 8 blocks on a seeded sample of token rows (exact for those rows)."""
    rows = tp_inputs.sample_rows(12, wl.T, n_rows)
    t0 = time.perf_counter()
    z = wl.x_bits[rows]
    for b in range(wl.nb):
        z = wl.oracle_block(b, z)
    dt = time.perf_counter() - t0
    flops = wl.flops * n_rows / wl.T
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": int(os.environ["OPENBLAS_NUM_THREADS"]),
            "kind": "oracle",
            "sample": f"{n_rows} of {wl.T} token rows through all {wl.nb} blocks, every rank's shards of all "
                      f"{2 * wl.nb} weights extracted (float64 numpy oracle), {dt:.1f} s; TFLOP/s = the sample's "
                      f"FLOPs (the step's scaled by rows) / its time",
            "per_row_s": dt / n_rows, "extrapolated_full_step_s": dt / n_rows * wl.T,
            "extrapolation": "per-row time x all token rows (extrapolated, not run; the shard extraction it "
                             "includes would not grow with the rows)"}


def generic_cpu_baseline(wl, target_s=12.0):
    """The oracle on a bounded sample of the workload's token rows, scaled to TFLOP/s."""
    T = wl.T
    n = 16
    t0 = time.perf_counter()
    wl.oracle_step(tp_inputs.sample_rows(11, T, n))
    dt = time.perf_counter() - t0
    while dt < target_s / 4 and n < T:
        n = min(T, n * 4)
        t0 = time.perf_counter()
        wl.oracle_step(tp_inputs.sample_rows(11, T, n))
        dt = time.perf_counter() - t0
    reps = max(1, int(round(target_s / max(dt, 1e-3)))) if n == T else 1
    t0 = time.perf_counter()
    for _ in range(reps):
        wl.oracle_step(tp_inputs.sample_rows(12, T, n))
    dt = time.perf_counter() - t0
    flops = wl.flops * n / T * reps
    what = f"{reps} repetitions of the whole step" if n == T else f"{n} of {T} token rows of one step"
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": int(os.environ["OPENBLAS_NUM_THREADS"]),
            "kind": "oracle", "sample": f"{what} (float64 numpy oracle), {dt:.1f} s; TFLOP/s = the sample's "
                                        f"FLOPs (the step's FLOPs scaled by rows) / its time"}


def oracle_sample_step(host, rows, p, H, heads, hd):
    """The oracle's attention-projection step, restricted to the given token rows (exact for those rows)."""
    from oracle import tp_oracle as O
    qkv = [O.shard(host["w_qkv"], "colwise", p, r, [H] * 3, num_heads=heads, head_dim=hd) for r in range(p)]
    wo = [O.shard(host["w_out"], "rowwise", p, r, num_heads=heads, head_dim=hd) for r in range(p)]
    ys = [O.f64_to_bf16(y) for y in O.colwise_forward(host["x"][rows], qkv, "none")]
    O.combine_gather(ys)
    a = host["a"][rows]
    z = O.rowwise_forward([O.shard(a, "rowwise", p, r) for r in range(p)], wo)
    return O.f64_to_bf16(z)


# ----------------------------------------------------------------------------- measurement

def make_workload(name, args, tp, torch, device):
    if name == WORKLOAD:
        return StackWorkload(tp, torch, device)
    if name == ATTN_PROJ:
        return AttnProjWorkload(tp, torch, device, args.reduce_mode, fused_gather=not args.unfused_gather)
    if name in ("tiny_mlp_tp2", "swiglu_mlp_tp4"):
        return MlpWorkload(tp, torch, device, name)
    if name == "block_sweep":
        return BlockWorkload(tp, torch, device, args.tp)
    if name == "single_stream_tp4":
        return SingleStreamWorkload(tp, torch, device, args.tp)
    raise ValueError(name)


def time_events(torch, stream, fn, reps, before=None):
    """Mean CUDA-event time (ms) of fn(stream) over reps runs, each alone (before() outside the events)."""
    ms = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            if before is not None:
                before()
            a.record(stream)
            fn(stream)
            b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    return float(np.mean(ms))


def measure(wl, args, tp, torch, device, stream, peaks, flush=None, steps=None, with_refs=True, sampler=None):
    """Time `wl`: warm-up, then `steps` whole steps each replayed as one CUDA graph (flush() between
    them, outside the events, when given), then a per-phase pass (each phase its own graph with
    events between them).  Returns the figures as a dict."""
    steps = args.steps if steps is None else steps
    phases = wl.phases()
    nph = len(phases)
    noop = (lambda: None)
    fl = flush or noop
    for _ in range(args.warmup):
        whole_step(wl, stream)
    stream.synchronize()
    tp.tp_device_status(stream)

    # Eager launches: host enqueue cost per step and a per-phase cross-check.
    n_eager = min(steps, 20)
    eager_marks = [[torch.cuda.Event(enable_timing=True) for _ in range(nph + 1)] for _ in range(n_eager)]
    torch.cuda.synchronize()
    host_s = 0.0
    for k in range(n_eager):
        with torch.cuda.stream(stream):
            fl()
        t0 = time.perf_counter()
        run_step(wl, stream, eager_marks[k])
        host_s += time.perf_counter() - t0
    torch.cuda.synchronize()
    eager_phase = np.array([[m[i].elapsed_time(m[i + 1]) for i in range(nph)] for m in eager_marks])

    # The timed steps replay the whole step as one captured CUDA graph (the launches a serving
    # loop would replay); the per-phase breakdown replays each phase as its own graph.
    graphs, step_graph = [], None
    if not args.eager:
        for _, fn, _, _ in phases:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn(stream)
            graphs.append(g)
        step_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(step_graph, stream=stream):
            whole_step(wl, stream)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                step_graph.replay()
                for g in graphs:
                    g.replay()
        stream.synchronize()
        tp.tp_device_status(stream)

    bounds = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if sampler is not None:
        sampler.start()
        time.sleep(0.3)
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for k in range(steps):
        with torch.cuda.stream(stream):
            fl()
            bounds[k][0].record(stream)
            if step_graph is not None:
                step_graph.replay()
            else:
                whole_step(wl, stream)
            bounds[k][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop() if sampler is not None else None
    tp.tp_device_status(stream)
    step_ms = float(np.mean([a.elapsed_time(b) for a, b in bounds]))

    # The timed step (which may reorder or overlap independent work) against the phases run one
    # after another: the same output, bit for bit.
    step_matches_phases = None
    if hasattr(wl, "step") and hasattr(wl, "z"):
        run_step(wl, stream)
        stream.synchronize()
        z_phases = wl.z.clone()
        with torch.cuda.stream(stream):
            wl.z.zero_()
        whole_step(wl, stream)
        stream.synchronize()
        step_matches_phases = bool(torch.equal(wl.z.view(torch.int16), z_phases.view(torch.int16)))

    # Per-phase breakdown (not the timed region): each phase alone between events.
    n_phase_steps = min(steps, 50)
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(nph + 1)] for _ in range(n_phase_steps)]
    for k in range(n_phase_steps):
        with torch.cuda.stream(stream):
            fl()
            if graphs:
                for i, g in enumerate(graphs):
                    marks[k][i].record(stream)
                    g.replay()
                marks[k][nph].record(stream)
            else:
                run_step(wl, stream, marks[k])
    torch.cuda.synchronize()
    tp.tp_device_status(stream)
    phase = np.array([[m[i].elapsed_time(m[i + 1]) for i in range(nph)] for m in marks])  # ms
    ph = phase.mean(axis=0)

    # Kernels by label: phases that share a label (the stack's 8 blocks) are pooled.
    agg = {}
    for (label, _, kind, work), ms in zip(phases, ph):
        a = agg.setdefault(label, [kind, 0.0, 0.0, 0])
        a[1] += work
        a[2] += float(ms)
        a[3] += 1
    kernels = {}
    for label, (kind, work, ms, n) in agg.items():
        rec = {"ms": round(ms / n, 5)}
        if n > 1:
            rec["launches_per_step"] = n
        if kind == "tensor":
            v = work / (ms * 1e-3) / 1e12
            rec.update({"TFLOP/s": v, "frac_tensor": v / peaks["bf16_tflops"],
                        "frac_tensor_sustained": v / peaks["bf16_tflops_sustained"]})
        else:
            v = work / (ms * 1e-3) / 1e9
            rec.update({"GB/s": v, "frac_hbm": v / peaks["hbm_gbs"]})
        kernels[label] = rec
    dominant = max(agg, key=lambda k: agg[k][2])

    res = {"ms_per_step": step_ms, "value": wl.flops / (step_ms * 1e-3) / 1e12, "kernels": kernels,
           "dominant": dominant, "phase_sum_ms": float(phase.sum(axis=1).mean()),
           "step_output_bit_identical_to_phases": step_matches_phases,
           "eager_ms_per_step": float(eager_phase.sum(axis=1).mean()),
           "host_enqueue_ms_per_step": host_s / n_eager * 1e3, "bracket_s": t_wall, "clocks": clocks,
           "launch": "eager" if args.eager else "cuda_graph_per_step"}

    # Reference points (cuBLAS / torch on the same work) and the join kernels alone, L2 flushed.
    if with_refs and hasattr(wl, "reference_points"):
        refs = {}
        for label, fn, kind, work in wl.reference_points():
            fn(stream)
            t = time_events(torch, stream, fn, 20, fl)
            if kind == "tensor":
                v = work / (t * 1e-3) / 1e12
                refs[label] = {"ms": round(t, 5), "TFLOP/s": v, "frac_tensor": v / peaks["bf16_tflops"]}
            else:
                v = work / (t * 1e-3) / 1e9
                refs[label] = {"ms": round(t, 5), "GB/s": v, "frac_hbm": v / peaks["hbm_gbs"]}
        if hasattr(wl, "phase_extract"):
            wl.phase_extract(stream)   # the shards the reference copy overwrote (same bytes) -- keep them exact
        stream.synchronize()
        res["reference_points"] = refs
    if with_refs and hasattr(wl, "join_phases"):
        joins = {}
        for label, fn, nbytes in wl.join_phases():
            fn(stream)
            t = time_events(torch, stream, fn, 20, fl)
            joins[label] = {"ms": round(t, 5), "GB/s": nbytes / (t * 1e-3) / 1e9,
                            "frac_hbm": nbytes / (t * 1e-3) / 1e9 / peaks["hbm_gbs"]}
        tp.tp_device_status(stream)
        res["join_kernels"] = joins
    return res


def roofline_of(res, workload, peaks, sustained):
    """The roofline object for the dominant kernel of a measure() result."""
    label = res["dominant"]
    k = res["kernels"][label]
    if "TFLOP/s" in k:
        peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
        return {"bound": "tensor", "achieved": k["TFLOP/s"], "peak": peak, "unit": "TFLOP/s",
                "frac": k["TFLOP/s"] / peak, "frac_of_burst": k["TFLOP/s"] / peaks["bf16_tflops"],
                "kernel": f"tp_gemm_kernel ({label})" if label != "attention" else "tp_flash_kernel",
                "peak_source": peaks["source"] + (" sustained" if sustained else " burst"),
                "launch_ms": k["ms"], "traffic": recorded_traffic(f"{workload}:{label}", "gemm")}
    return {"bound": "hbm", "achieved": k["GB/s"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": k["GB/s"] / peaks["hbm_gbs"], "kernel": label, "peak_source": peaks["source"],
            "launch_ms": k["ms"], "traffic": recorded_traffic(f"{workload}:{label}", "copy")}


def time_e2e(torch, tp, stream, fn, warmup, reps, flush=None, runs=None):
    """Median CUDA-event time (ms) of `reps` end-to-end steps, each alone: a step crosses the
    CPU-GPU link, whose copies now and then stall for tens of milliseconds on this machine.
    The single times go to `runs` when given."""
    for _ in range(max(1, warmup)):
        with torch.cuda.stream(stream):
            fn(stream)
    stream.synchronize()
    ts = [time_events(torch, stream, fn, 1, flush) for _ in range(reps)]
    tp.tp_device_status(stream)
    if runs is not None:
        runs.extend(round(t, 3) for t in ts)
    return float(np.median(ts))


def attn_proj_extras(args, tp, torch, device, stream, peaks, flush):
    """Per-kernel figures of the attention projections (tokens 4096, hidden 3072, tp 4), both join
    forms of the rowwise out-projection, and the end-to-end step with host buffers."""
    wl = AttnProjWorkload(tp, torch, device, "accum", fused_gather=True)
    res = measure(wl, args, tp, torch, device, stream, peaks, flush=flush, steps=args.steps)
    # The rowwise out-projection in its other join form: fp32 partials through an HBM workspace,
    # summed in the GEMM epilogue (the counters' clear and the GEMM, one phase).
    ws_bytes = tp.tp_rowwise_workspace_bytes(wl.p, wl.T, wl.H, "workspace")
    wsbuf = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    z_ws = torch.empty_like(wl.z)
    fn = lambda st: tp.tp_linear_rowwise(wl.a_sh, wl.out_sh, mode="workspace", workspace=wsbuf, out=z_ws,  # noqa
                                         stream=st)
    fn(stream)
    t = time_events(torch, stream, fn, 20, flush)
    tp.tp_device_status(stream)
    v = wl.flops_out / (t * 1e-3) / 1e12
    extra = 2.0 * wl.p * wl.T * wl.H * 4
    res["kernels"]["rowwise_out_workspace"] = {
        "ms": round(t, 5), "TFLOP/s": v, "frac_tensor": v / peaks["bf16_tflops"],
        "workspace_bytes_per_launch": extra,
        "traffic": recorded_traffic(f"{ATTN_PROJ}:rowwise_out_workspace", "gemm"),
        "what": "TP_REDUCE_WORKSPACE: every rank's fp32 partial tile written to the workspace and summed back in "
                "rank order by the tile's CTAs (2*p*T*N*4 bytes more than the on-chip sum)"}
    # End to end (host buffers): activations in, Z out, pipelined over row blocks, one graph.
    wl.setup_e2e()
    step = lambda st: wl.step_e2e_chunked(st)  # noqa: E731
    step(stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step(stream)
    e2e_ms = time_e2e(torch, tp, stream, lambda st: g.replay(), args.warmup, min(args.steps, 50), flush)
    res["e2e"] = {"value": wl.flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": e2e_ms,
                  "h2d_bytes_per_step": int(wl.h2d_bytes), "d2h_bytes_per_step": int(wl.d2h_bytes)}
    res["config"] = wl.config()
    res["flops_per_step"] = wl.flops
    return res


def block_extras(args, tp, torch, device, stream, peaks, flush):
    """Per-kernel figures of the full attention + SwiGLU MLP block at tp 4."""
    saved = args.tp
    args.tp = 4
    try:
        wl = BlockWorkload(tp, torch, device, 4)
    finally:
        args.tp = saved
    res = measure(wl, args, tp, torch, device, stream, peaks, flush=flush, steps=args.steps, with_refs=False)
    res["config"] = wl.config()
    res["flops_per_step"] = wl.flops
    add_attention_issued(res, peaks)
    return res


def add_attention_issued(res, peaks):
    """The attention phase's issued tensor work beside its algorithmic figure: P enters P.V as
    two bf16 terms, so the tensor core runs 1.5 times the 4*T^2*d FLOPs credited per head."""
    k = res.get("kernels", {}).get("attention")
    if k and "TFLOP/s" in k:
        k["issued_TFLOP/s"] = 1.5 * k["TFLOP/s"]
        k["issued_frac_tensor"] = k["issued_TFLOP/s"] / peaks["bf16_tflops"]
        k["issued_note"] = "S = Q K^T plus P_hi V and P_lo V: 1.5 x the credited FLOPs"


def run_ours(args):
    refuse_multi_gpu(args)
    import torch
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    from __graft_entry__ import build
    build()
    import tensor_sharded_linear_tp_gb300 as tp
    stream = torch.cuda.Stream(device)
    peaks = load_peaks()
    if args.workload == WORKLOAD:
        return run_stack(args, tp, torch, device, stream, peaks)
    flush = L2Flush(torch, device)
    wl = make_workload(args.workload, args, tp, torch, device)
    res = measure(wl, args, tp, torch, device, stream, peaks, flush=flush, sampler=ClockSampler(0))
    add_attention_issued(res, peaks)
    cpu = None if args.no_cpu_baseline else generic_cpu_baseline(wl)
    cfg = wl.config()
    cfg.update({"parallelism": f"tp{wl.p} simulated on one GPU", "l2": "flushed between steps "
                "(256 MiB write, then 256 MiB read)", "sms": torch.cuda.get_device_properties(device).multi_processor_count})
    line = {"metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,0.02) weights, N(0,1) activations)",
            "config": cfg, "roofline": roofline_of(res, args.workload, peaks, sustained=False),
            "cpu_baseline": cpu, "gpu_launches": wl.launches_per_step * args.steps, "peaks": peaks}
    line.update({k: v for k, v in res.items() if k not in ("value", "ms_per_step")})
    print(json.dumps(line))


def run_stack(args, tp, torch, device, stream, peaks):
    """The default line: the 8-block stack, shard-on-read, with the other workloads' kernels beside it."""
    wl = StackWorkload(tp, torch, device)

    # Shard-on-read of the whole state dict, against a plain page-locked copy of 1 GiB: two
    # untimed loads, then the median of nine (each alone between events).  The host link
    # stalls now and then for tens of milliseconds; nine runs keep up to four such runs out
    # of the median.
    for _ in range(2):
        wl.load(stream)
    stream.synchronize()
    tp.tp_device_status(stream)
    load_runs = [time_events(torch, stream, wl.load, 1) for _ in range(9)]
    load_ms = float(np.median(load_runs))
    probe_n = 1 << 30
    src = torch.empty(probe_n, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(probe_n, dtype=torch.uint8, device=device)

    def link_copy(st):
        with torch.cuda.stream(st):
            dst.copy_(src, non_blocking=True)
    link_copy(stream)
    copy_ms = float(np.median([time_events(torch, stream, link_copy, 1) for _ in range(9)]))
    del dst, src
    load_gbs = wl.shard_bytes / (load_ms * 1e-3) / 1e9
    link_gbs = probe_n / (copy_ms * 1e-3) / 1e9

    # The forward pass (the timed steps), clocks sampled during it.
    sampler = ClockSampler(0)
    res = measure(wl, args, tp, torch, device, stream, peaks, flush=None, sampler=sampler)
    roof = roofline_of(res, WORKLOAD, peaks, sustained=True)

    # End to end with host buffers (every weight slice, the input and the output cross the link).
    e2e_runs, serial_runs, resident_runs = [], [], []
    e2e_ms = time_e2e(torch, tp, stream, lambda st: wl.step_e2e(st, pipelined=True), 1, 5, runs=e2e_runs)
    e2e_serial_ms = time_e2e(torch, tp, stream, lambda st: wl.step_e2e(st, pipelined=False), 1, 5,
                             runs=serial_runs)
    wl.load(stream)
    e2e_resident_ms = time_e2e(torch, tp, stream, wl.step_e2e_resident, 2, 9, runs=resident_runs)
    # The pipelined step's output against the device-resident forward's, bit for bit.
    wl.forward(stream)
    stream.synchronize()
    z_dev = wl.z.clone()
    wl.step_e2e(stream, pipelined=True)
    stream.synchronize()
    e2e_same = bool(torch.equal(wl.z_pin.to(device).view(torch.int16), z_dev.view(torch.int16)))
    h2d = wl.shard_bytes + wl.T * wl.H * 2
    d2h = wl.T * wl.H * 2

    flush = L2Flush(torch, device)
    extras = {}
    if not args.no_extras:
        extras[ATTN_PROJ] = attn_proj_extras(args, tp, torch, device, stream, peaks, flush)
        extras["block_tp4"] = block_extras(args, tp, torch, device, stream, peaks, flush)
    cpu = None if args.no_cpu_baseline else stack_cpu_baseline(wl)

    cfg = wl.config()
    cfg.update({"parallelism": f"tp{wl.p} simulated on one GPU",
                "l2": "inputs larger than L2: every step reads 5.44 GB of weight shards (no flush)",
                "sms": torch.cuda.get_device_properties(device).multi_processor_count})
    line = {
        "metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,0.02) weights, N(0,1) activations)",
        "config": cfg, "roofline": roof, "kernels": res["kernels"],
        "reference_points": res.get("reference_points"),
        "shard_load": {"bytes": wl.shard_bytes, "ms": load_ms, "ms_runs": [round(v, 3) for v in load_runs],
                       "GB/s": load_gbs, "link_copy_GB/s": link_gbs,
                       "frac_of_link_copy": load_gbs / link_gbs, "frac_hbm": load_gbs / peaks["hbm_gbs"],
                       "what": "every rank's slice of all 16 weights from page-locked host memory into device "
                               "shards (tp_plan_shard_ranks: copy-engine transfers, one per packed block and rank), "
                               "median of 9, against a 1 GiB page-locked host-to-device copy (median of 9)"},
        "e2e": {"value": wl.flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": e2e_ms,
                "ms_runs": e2e_runs, "timing": "median of 5 steps, each alone between events",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "inputs": "every rank's weight slices (shard-on-read, 5.44 GB) and X from page-locked host memory "
                          "every step; Z read back",
                "pipelining": "X and the blocks' slices arrive in block order on a copy stream; each projection "
                              "starts as soon as its own weight's slices have landed",
                "output_bit_identical_to_device_step": e2e_same,
                "unpipelined": {"value": wl.flops / (e2e_serial_ms * 1e-3) / 1e12, "ms_per_step": e2e_serial_ms,
                                "ms_runs": serial_runs},
                "weights_resident": {"value": wl.flops / (e2e_resident_ms * 1e-3) / 1e12, "ms_per_step": e2e_resident_ms,
                                     "ms_runs": resident_runs,
                                     "h2d_bytes_per_step": wl.T * wl.H * 2, "d2h_bytes_per_step": d2h,
                                     "what": "a serving step with the shards loaded once: X in from page-locked "
                                             "host memory, the 8 blocks, Z back"}},
        "cpu_baseline": cpu,
        "gpu_launches": wl.launches_per_step * args.steps,
        "clocks": res["clocks"], "peaks": peaks,
    }
    for k in ("phase_sum_ms", "step_output_bit_identical_to_phases", "eager_ms_per_step", "host_enqueue_ms_per_step",
              "bracket_s", "launch"):
        line[k] = res[k]
    for name, r in extras.items():
        line[name] = {k: v for k, v in r.items() if k not in ("clocks", "dominant")}
        line[name]["roofline"] = roofline_of(r, ATTN_PROJ if name == ATTN_PROJ else "block_sweep", peaks,
                                             sustained=False)
    if ATTN_PROJ in extras:
        ex = extras[ATTN_PROJ]["kernels"]["extract"]
        line["extract_gbs"] = ex["GB/s"]
        line["extract_frac_hbm"] = ex["frac_hbm"]
    print(json.dumps(line))


def run_reference(args):
    """The CPU oracle as the reference arm, on the default workload: each step one block of the stack
    (blocks in turn) on a seeded sample of token rows, every rank's shards of its two weights extracted."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    cfg = tp_inputs.WORKLOADS[WORKLOAD]
    p, nb, T, H, F, seed = cfg["tp"], cfg["blocks"], cfg["tokens"], cfg["hidden"], cfg["ffn"], cfg["seed"]
    from oracle import tp_oracle as O
    jobs = [(b, which) for b in range(nb) for which in ("gate_up", "down")]
    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        bits = list(ex.map(lambda j: tp_inputs.stack_weight(seed, j[0], j[1], H, F), jobs))
    x = tp_inputs.stack_input(seed, nb, T, H)
    n_rows = 64
    flops_block = 2.0 * n_rows * (H * 2 * F + F * H)

    def one(k):
        b = k % nb
        gu, dn = bits[2 * b], bits[2 * b + 1]
        rows = tp_inputs.sample_rows(40 + k, T, n_rows)
        t0 = time.perf_counter()
        O.mlp_forward(x[rows], [O.shard(gu, "colwise", p, r, [F, F]) for r in range(p)],
                      [O.shard(dn, "rowwise", p, r) for r in range(p)], "swiglu")
        return time.perf_counter() - t0
    for w in range(args.warmup):
        one(w)
    times = [one(args.warmup + k) for k in range(args.steps)]
    value = flops_block / float(np.mean(times)) / 1e12
    cores = int(os.environ["OPENBLAS_NUM_THREADS"])
    sample = (f"one block per step (blocks in turn) on {n_rows} of {T} token rows, every rank's shards of the "
              f"block's two weights extracted (float64 numpy oracle)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": float(np.mean(times)) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "blocks": nb, "tokens": T, "hidden": H, "ffn": F, "tp_degree": p},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def _status_bytes(key):
    """A size line of /proc/self/status (VmHWM, RssAnon, ...) in bytes, or None."""
    try:
        with open("/proc/self/status") as fh:
            for line in fh:
                if line.startswith(key + ":"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def _vm_hwm_bytes():
    return _status_bytes("VmHWM")


def run_st_load(args):
    """Shard-on-read of single-stream blocks (hidden 6144, mlp_ratio 3, tp 4) from a safetensors file.

    A synthetic checkpoint of 4 blocks (the fused [1,1,1,3,3] in-projection and the packed
    to_out of each, 3.93 GB of bf16) is written to a temporary directory, read once untimed
    (the page cache is then warm: this measures the loader, not the disk), then every rank's
    shard of every tensor is loaded with tp_st_plan_shard_ranks.  Beside it: a plain
    page-locked host-to-device copy of 1 GiB (the link ceiling) and the peak host memory the
    loads add (the page's "peak CPU/rank" column).
    """
    import shutil
    import tempfile

    refuse_multi_gpu(args)
    import torch
    from __graft_entry__ import build
    build()
    import tensor_sharded_linear_tp_gb300 as tp
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    cfg = tp_inputs.WORKLOADS["single_stream_tp4"]
    H, p, heads, seed = cfg["hidden"], cfg["tp"], cfg["heads"], cfg["seed"]
    F = cfg["mlp_ratio"] * H
    nb = 4
    total = nb * ((3 * H + 2 * F) * H + H * (H + F)) * 2
    tmp = tempfile.mkdtemp(prefix="tp_st_bench_")
    try:
        if shutil.disk_usage(tmp).free < total + (2 << 30):
            print(json.dumps({"metric": "shard-on-read load GB/s from a safetensors file", "value": None,
                              "unavailable": f"not enough free space in {tmp} for a {total / 1e9:.1f} GB file"}))
            return
        path = os.path.join(tmp, "single_stream_blocks.safetensors")
        tensors = []
        for b in range(nb):
            w_in = tp_inputs.weight_bf16(seed, 10 + 2 * b, (3 * H + 2 * F, H))
            w_out = tp_inputs.weight_bf16(seed, 11 + 2 * b, (H, H + F))
            tensors += [(f"single_transformer_blocks.{b}.attn.to_qkv_mlp_proj.weight", "BF16", w_in),
                        (f"single_transformer_blocks.{b}.attn.to_out.weight", "BF16", w_out)]
        tp_inputs.write_safetensors(path, tensors, metadata={"format": "pt"})
        del tensors
        e = lambda *sh: torch.empty(sh, dtype=torch.bfloat16, device=device)  # noqa: E731
        outs = [([e((3 * H + 2 * F) // p, H) for _ in range(p)], [e(H, (H + F) // p) for _ in range(p)])
                for _ in range(nb)]
        stream = torch.cuda.Stream(device)
        f = tp.SafetensorsFile(path)
        read_mode = f.read_mode_on_device()

        def load():
            for b, (o_in, o_out) in enumerate(outs):
                f.shard_ranks(f"single_transformer_blocks.{b}.attn.to_qkv_mlp_proj.weight", "colwise", p,
                              fused_splits=[H, H, H, F, F], num_heads=heads, outs=o_in, stream=stream)
                f.shard_ranks(f"single_transformer_blocks.{b}.attn.to_out.weight", "rowwise", p,
                              fused_splits=[H, F], num_heads=heads, outs=o_out, stream=stream)
            stream.synchronize()

        with open(path, "rb") as fh:              # warm the page cache
            while fh.read(64 << 20):
                pass
        load()
        hwm_reset = True
        try:
            with open("/proc/self/clear_refs", "w") as fh:
                fh.write("5")
        except OSError:
            hwm_reset = False
        hwm0, anon0 = _vm_hwm_bytes(), _status_bytes("RssAnon")
        reps = max(1, min(args.steps, 5))

        def timed_loads():
            times = []
            for _ in range(reps):
                t0 = time.perf_counter()
                load()
                times.append(time.perf_counter() - t0)
            return times

        load_runs = timed_loads()
        load_s = statistics.median(load_runs)
        hwm1, anon1 = _vm_hwm_bytes(), _status_bytes("RssAnon")
        # The other way of reading, for comparison: staged through page-locked buffers by host
        # threads (bounded by the host's file-read rate), where the default maps the file.
        other = "staged" if read_mode == "mapped" else None
        other_s = None
        if other is not None:
            f.close()
            f = tp.SafetensorsFile(path, read_mode=other)
            load()
            other_s = statistics.median(timed_loads())
        f.close()
        tp.tp_device_status(stream)

        probe_n = 1 << 30
        src = torch.empty(probe_n, dtype=torch.uint8, pin_memory=True)
        dst = torch.empty(probe_n, dtype=torch.uint8, device=device)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        with torch.cuda.stream(stream):
            dst.copy_(src, non_blocking=True)
            ev[0].record(stream)
            for _ in range(3):
                dst.copy_(src, non_blocking=True)
            ev[1].record(stream)
        stream.synchronize()
        link_gbs = 3 * probe_n / (ev[0].elapsed_time(ev[1]) * 1e-3) / 1e9
        value = total / load_s / 1e9
        line = {
            "metric": "shard-on-read load GB/s from a safetensors file", "value": value, "unit": "GB/s",
            "n_gpus": 1, "steps": reps, "warmup": 1, "ms_per_step": load_s * 1e3, "higher_is_better": True,
            "ms_runs": [round(t * 1e3, 2) for t in load_runs], "timing": "median of the loads",
            "dtype": "bf16", "data": "synthetic (seeded N(0,0.02) weights)",
            "config": {"workload": "st_load_single_stream", "blocks": nb, "hidden": H, "mlp_hidden": F,
                       "tp_degree": p, "ranks_loaded": p, "file_bytes": total,
                       "staging_bytes": 2 * (64 << 20), "page_cache": "warm",
                       "step": "every rank's shard of every tensor: packed [1,1,1,3,3] colwise in-projection "
                               "and packed [inner, mlp] rowwise to_out, 4 blocks"},
            "read_mode": read_mode,
            "link_copy_GB/s": link_gbs, "frac_of_link_copy": value / link_gbs,
            "peak_host_rss_growth_bytes": (hwm1 - hwm0) if (hwm_reset and hwm0 is not None) else None,
            "host_anon_growth_bytes": (anon1 - anon0) if (anon0 is not None and anon1 is not None) else None,
            "host_memory_note": "mapped reads keep the file's pages mapped (page cache, shared, reclaimable) "
                                "until the file is closed, so the peak resident size counts them; anonymous "
                                "memory is what the loader itself holds",
            "gpu_launches": nb * (-(-((H + F) * 2 * H) // (64 << 20))) * reps,
        }
        if other_s is not None:
            line[f"{other}_GB/s"] = total / other_s / 1e9
            line[f"{other}_ms_per_step"] = other_s * 1e3
        print(json.dumps(line))
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1, help="must be 1: the library runs every rank on one GPU")
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--reduce-mode", choices=["accum", "workspace", "none"], default="accum",
                    help="rowwise join of --workload attn_proj_tp4")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--no-extras", action="store_true",
                    help="default workload: skip the attention-projection and block figures beside the stack")
    ap.add_argument("--eager", action="store_true", help="launch the timed steps eagerly instead of as graphs")
    ap.add_argument("--unfused-gather", action="store_true",
                    help="attention projections: gather the QKV slices with a separate tp_combine kernel instead "
                         "of writing the gathered layout from the colwise GEMM")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=[WORKLOAD, ATTN_PROJ, "tiny_mlp_tp2", "swiglu_mlp_tp4", "block_sweep",
                             "single_stream_tp4", "st_load_single_stream"],
                    help="the 8-block stack loaded shard-on-read (default), the attention projections, the tiny "
                         "or SwiGLU MLP block, the full block (with --tp), the single-stream block, or "
                         "shard-on-read from a safetensors file")
    ap.add_argument("--tp", type=int, default=4, help="tp_degree of --workload block_sweep / single_stream_tp4")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)   # at least three untimed warm-up steps, whatever was asked
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "st_load_single_stream":
        run_st_load(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
