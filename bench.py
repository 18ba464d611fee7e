"""Benchmark of the AttnRes depth-wise aggregation on GB300.

One step = one pass of the aggregation hot path over one batch of synthetic
inputs already resident in HBM. The default (headline) workload is the
long-context prefill Block AttnRes pass: T = 131072 tokens (128K), d = 2048,
48 sublayers in 8 blocks of 6, bf16 storage with fp32 arithmetic; every
sublayer's read runs by the two-stage computation (stage 1 per block, one
online-softmax merge per later sublayer, a freeze per block summary, in the
order a layer-by-layer forward runs them). This is
the largest single-GPU footprint of the standard workloads (about 60 GB
resident). The other bench workloads are measured in the same run and
reported under "extras": the deep-narrow Full pass (141 reads, 32768 x 640),
the 400M Full pass (64 reads, 8192 x 896) and the 8 x 8 Block pass (16384 x
1024).

Prints one JSON line (rank 0). Metric: tokens/s (higher is better), with the
HBM roofline of the dominant kernel. The K timed steps follow the benchmark
contract; a separate "sustained" measurement replays the same step for at
least 2 s with its own clock samples. ``--impl reference`` times the fp64 CPU
oracle on the same workload instead (a bounded sample of token rows per step).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME] [--op OP] [--no-e2e] [--no-extras]
                       [--no-cpu-baseline] [--no-sustained]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from depth_wise_attention_attnres_gb300 import inputs  # noqa: E402

METRIC = "AttnRes aggregation tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
DEFAULT_WORKLOAD = "block_pass_8x6x131072x2048_bf16"
NOMINAL_HBM_GBS = 8000.0  # the nominal HBM bandwidth the target is stated against
# Measured in the same run as the headline (when it is not one of them).
EXTRA_WORKLOADS = ["full_pass_141x32768x640_bf16", "full_pass_64x8192x896_bf16",
                   "block_pass_8x8x16384x1024_bf16"]
SUSTAINED_S = 2.0  # length of the separate sustained measurement


# ----------------------------------------------------------------- bytes ----

def full_pass_bytes(R: int, T: int, d: int, es: int) -> int:
    """Algorithmic bytes of a Full pass: read r moves r+1 source rows and
    writes one output row per token: sum_r (r + 2) * T * d * es."""
    return sum(r + 2 for r in range(R)) * T * d * es


def block_pass_bytes(N: int, S: int, T: int, d: int, es: int, plan=None, freeze_last: bool = False,
                     fused_freeze: bool = False) -> dict:
    """Algorithmic bytes per kernel of the two-stage Block pass.

    stage 1 of block n (n+1 sources): reads (n+1) rows, writes S output rows
    and S lse values per token. Merge j (1 <= j < S): reads O_j, lse_j and its
    running sum P_j as the last kept sum P_m (fp32, if m > 0) plus the j - m
    outputs since, writes out_j and, if the plan keeps P_j, P_j (fp32). The
    freeze reads P_S the same way and writes the summary (attnres_block_pass,
    in the order of a layer-by-layer forward). With fused_freeze the block's
    last merge freezes instead (attnres_block_merge_parts' summary_out, for
    callers holding every output): it reads f_{S-1} more and writes the
    summary. plan[j] = 1 where the pass keeps P_j
    (attnres_block_running_sum_plan); None keeps every sum (the one-step
    merges).
    """
    if plan is None:
        plan = [0] + [1] * (S - 1) + [0]
    E = T * d
    st1 = merge = freeze = 0
    for n in range(N):
        st1 += (n + 1) * E * es + S * E * es + S * T * 4
        m = 0
        for j in range(1, S):
            merge += 2 * E * es + T * 4 + (j - m) * E * es + (4 * E if m > 0 else 0) + (4 * E if plan[j] else 0)
            if plan[j]:
                m = j
        if n + 1 < N or freeze_last:
            if S > 1 and fused_freeze:
                merge += 2 * E * es
            else:
                freeze += (S - m) * E * es + (4 * E if m > 0 else 0) + E * es
    return {"stage1": st1, "merge": merge, "freeze": freeze, "total": st1 + merge + freeze}


DSPLIT_SHARDS = 4
E2E_COPY_STREAMS = 4  # streams per copy direction in the e2e loop


def block_bwd_bytes(N: int, S: int, T: int, d: int, es: int) -> dict:
    """Algorithmic bytes of the Block pass backward with all S reads of a block
    in one pass (the batched kernel: d a multiple of 128 up to 1024, N <= 8,
    S <= 8). Per block n: the n + 1 sources, the block's outputs but its last
    (for the running sums) and the S gradients dL/dout read once, the gradient
    of the block's summary read (n + 1 < N), the sources' fp32 gradient rows
    and the S outputs' fp32 gradient rows read and written once. Once: those
    rows zeroed; the embedding's gradient added at the end."""
    E = T * d
    read = route = 0
    for n in range(N):
        read += (n + 1) * E * es + (S - 1) * E * es + S * E * es + (4 * E if n + 1 < N else 0)
        route += (n + 1) * 8 * E + S * 8 * E
    route += N * 4 * E + 12 * E
    return {"read": read, "route": route, "total": read + route}


def block_bwd_bytes_per_read(N: int, S: int, T: int, d: int, es: int) -> dict:
    """Algorithmic bytes of the Block pass backward read by read (the fallback).

    Per read k = nS + j over n_src = n + 1 (+ 1 for the running sum when j >= 1)
    fp32 sources: the read backward moves n_src rows (read) and their fp32
    gradient rows (read and written) and dL/dout_k ("read"); with j >= 1 the
    running sum is copied into its source slot and its gradient routed (G,
    the slot and dF_{k-1} read and written: "route"). Per block: the running
    sums rebuilt, and the gradient of the block's summary added to its S
    members ("route"). Once: the sources widened to fp32 and their gradients
    zeroed; the embedding's gradient added at the end ("route").
    """
    E = T * d
    read = route = 0
    for n in range(N):
        for j in range(S):
            n_src = n + 1 + (1 if j >= 1 else 0)
            read += n_src * E * (4 + 8) + E * es
            if j >= 1:
                route += 8 * E + 24 * E
        route += E * (es + 4) + max(S - 2, 0) * E * (4 + es + 4) + 4 * E  # running sums, G zeroed
        if n + 1 < N:
            route += 4 * E + S * 8 * E + 4 * E
    route += (N + 1) * 4 * E + N * E * (es + 4) + 12 * E
    return {"read": read, "route": route, "total": read + route}


def dsplit_stage1_bytes(N: int, S: int, T: int, d: int, es: int, P: int) -> dict:
    """Algorithmic bytes of the Block pass's N stage-1 reads taken as a d-split
    over P feature shards. Block n (n+1 sources): the partials kernels read
    every source row once and write the fp32 sums [T, n+1, S+1] (the first
    shard writes them, the others read and write them); the finish kernels
    read every source row once more and the sums once per shard, and write S
    output rows and S lse values per token."""
    E = T * d
    part = fin = 0
    for n in range(N):
        sums = (n + 1) * T * (S + 1) * 4
        part += (n + 1) * E * es + sums * (2 * P - 1)
        fin += (n + 1) * E * es + sums * P + S * E * es + S * T * 4
    return {"partials": part, "finish": fin, "total": part + fin}


# ---------------------------------------------------------------- clocks ----

class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="attnres_clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self) -> dict:
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- peaks ----

def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) over algorithmic
# bytes, from one ncu capture of the kernel, keyed by the sha256 prefix of the
# kernel source it was taken with: reported as null once the source changes.
# full_bwd_bulk_kernel: all 64 launches of the 8192 x 896 pass backward
# without ncu's cache flush between launches, 103100.1 MB read + 60938.3 MB
# written for 153612.2 MB algorithmic (the second pass over a tile's sources
# re-reads part of them from DRAM).
# block_bwd_batched_kernel: all 8 launches of one 8x8 Block backward at 2048
# tokens, 1554.1 MB read + 420.6 MB written for the step's 2483.0 MB
# algorithmic (reads equal the algorithmic reads; the rest of the writes were
# still in L2 when ncu flushed it between launches). The per-launch traffic
# grows with the tokens.
# full_fwd_bulk_kernel (source 664fdb90f174cfdb): all 64 launches of the 8192 x
# 896 pass without ncu's cache flush between launches, 30289.2 MB read +
# 1033.1 MB written for 31474.1 MB algorithmic.
NCU_TRAFFIC = {("full_fwd_bulk_kernel", "664fdb90f174cfdb"): (30289.201664 + 1033.079552) / 31474.057216,
               ("full_bwd_bulk_kernel", "bd0791324025b552"): (103100.1 + 60938.3) / 153612.2,
               ("block_bwd_batched_kernel", "cb4b0fb7ff058c27"): (1554.098176 + 420.645888) / 2483.027968}


# Block-pass kernels: DRAM bytes / algorithmic bytes over all launches of one
# kind in one pass, captured without ncu's cache flush between launches
# (steady-state write-backs counted), keyed by (kernel, source digest) and then
# by workload. The 128K prefill's ratios come from the same blocks at 8192
# tokens (profiles/block_pass_kernels_8x6x131072x2048_bf16.md).
NCU_TRAFFIC_BLOCK = {
    ("stage1_tc_kernel", "424235d9916c799e"): {
        "block_pass_8x6x131072x2048_bf16": (1144.0 + 1357.6) / 2820.1,
        "block_pass_8x8x16384x1024_bf16": (1143.2 + 1871.4) / 3359.6},
    ("merge_tile_kernel", "0eb18c612a846d80"): {
        "block_pass_8x6x131072x2048_bf16": (4676.6 + 2071.9) / 6712.2,
        "block_pass_8x8x16384x1024_bf16": (7003.8 + 3135.3) / 10204.2},
    ("accum_fast_kernel", "0eb18c612a846d80"): {
        "block_pass_8x6x131072x2048_bf16": (838.3 + 289.7) / 1174.4,
        "block_pass_8x8x16384x1024_bf16": (838.7 + 303.9) / 1174.4},
}

KERNEL_FILES = {"full_fwd_bulk_kernel": "full_fwd.cu", "full_bwd_bulk_kernel": "full_bwd.cu",
                "block_bwd_batched_kernel": "block_bwd.cu", "stage1_tc_kernel": "stage1_tc.cu",
                "merge_tile_kernel": "merge.cu", "accum_fast_kernel": "merge.cu"}


def kernel_digest(name: str) -> str:
    path = os.path.join(ROOT, "depth_wise_attention_attnres_gb300", "csrc", name)
    with open(path, "rb") as fh:
        return hashlib.sha256(fh.read()).hexdigest()[:16]


# ------------------------------------------------------------ distributed ----

def dist_setup(n_gpus: int, backend: str | None = None):
    """Join the process group torchrun set up (one rank per GPU; NCCL on GPUs,
    gloo otherwise). Returns (rank, world, local_rank)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = backend or ("nccl" if torch.cuda.is_available() else "gloo")
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest per-rank value (the job's step time is its slowest rank's)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank processes its own batch (weak scaling)."""
    return tokens_per_rank * world / (ms_per_step / 1e3)


# ---------------------------------------------------------------- our arm ----

class FullPassStep:
    """One Full pass. op "read": the reads alone; "prenorm": each read emits
    the sublayer pre-norm of its result instead of the result (the same bytes);
    "prenorm_both": the result and its pre-norm (one more row write per read)."""

    def __init__(self, wl, dev, op="read"):
        from depth_wise_attention_attnres_gb300 import binding
        self.ar = binding
        self.wl = wl
        self.op = op
        self.V, self.W, self.G = inputs.full_inputs(wl, dev)
        dt = inputs.DTYPES[wl.dtype]
        self.out = torch.empty(wl.R, wl.T, wl.d, device=dev, dtype=dt)
        es = 2 if wl.dtype == "bf16" else 4
        self.bytes = full_pass_bytes(wl.R, wl.T, wl.d, es)
        if op in ("prenorm", "prenorm_both"):
            g = inputs.generator(wl.seed + 1, dev)
            self.Gpre = 1 + 0.1 * inputs.queries(wl.R, wl.d, 1.0, g, dev)
            self.normed = torch.empty(wl.R, wl.T, wl.d, device=dev, dtype=dt)
            if op == "prenorm_both":
                self.bytes += wl.R * wl.T * wl.d * es
        if op == "dynq":
            # Input-dependent query: read r's query projected from its newest
            # source V[r] by its own Wq[r] (tensor-core GEMM), then the read.
            g = inputs.generator(wl.seed + 3, dev)
            self.Wq = (inputs.randn((wl.R, wl.d, wl.d), "f32", g, dev) / wl.d ** 0.5).to(torch.bfloat16)
            self.Q = torch.empty(wl.T, wl.d, device=dev)
            E = wl.T * wl.d
            # per read: the GEMM reads V[r] and Wq[r] and writes Q; the read adds Q
            self.bytes += sum(E * es + wl.d * wl.d * 2 + E * 4 + E * 4 for _ in range(wl.R))
            self.flops = 2 * wl.T * wl.d * wl.d * wl.R
        if op == "bwd":
            # The pass backward: reads in reverse order, each adding its share
            # into fp32 dV (read-modify-write), dW and dGamma.
            g = inputs.generator(wl.seed + 2, dev)
            self.dZ = inputs.randn((wl.R, wl.T, wl.d), wl.dtype, g, dev)
            self.dV = torch.zeros(wl.R, wl.T, wl.d, device=dev)
            self.dW = torch.zeros(wl.R, wl.d, device=dev)
            self.dG = torch.zeros(wl.R, wl.d, device=dev)
            E = wl.T * wl.d
            self.bytes = sum((r + 1) * E * (es + 8) + E * es for r in range(wl.R))
        self.launches = wl.R * (2 if op == "dynq" else 1)

    def __call__(self):
        if self.op == "read":
            self.ar.attnres_full_pass(self.V, self.W, self.G, self.wl.eps, self.out)
        elif self.op == "dynq":
            for r in range(self.wl.R):
                self.ar.attnres_query_projection(self.V[r], self.Wq[r], self.Q)
                self.ar.attnres_full_fwd_dynq(self.V, r + 1, self.Q, self.G[r], self.wl.eps, self.out[r])
        elif self.op == "bwd":
            for r in reversed(range(self.wl.R)):
                self.ar.attnres_full_bwd(self.V, r + 1, self.W[r], self.G[r], self.wl.eps, self.dZ[r], self.dV,
                                         self.dW[r], self.dG[r])
        else:
            self.ar.attnres_full_pass_prenorm(self.V, self.W, self.G, self.wl.eps, self.Gpre, self.wl.eps,
                                              self.out if self.op == "prenorm_both" else None, self.normed)


class BlockPassStep:
    def __init__(self, wl, dev):
        from depth_wise_attention_attnres_gb300 import binding
        self.ar = binding
        self.wl = wl
        dt = inputs.DTYPES[wl.dtype]
        emb, self.F, self.W, self.G = inputs.block_inputs(wl, dev)
        self.Src = torch.empty(wl.N, wl.T, wl.d, device=dev, dtype=dt)
        self.Src[0].copy_(emb)
        del emb
        self.O = torch.empty(max(wl.S - 1, 1), wl.T, wl.d, device=dev, dtype=dt)
        self.lse = torch.empty(wl.S, wl.T, device=dev)
        self.P = torch.empty(wl.T, wl.d, device=dev)
        self.out = torch.empty(wl.N * wl.S, wl.T, wl.d, device=dev, dtype=dt)
        self.launches = wl.N + wl.N * (wl.S - 1) + (wl.N - 1)
        es = 2 if wl.dtype == "bf16" else 4
        self.plan = binding.attnres_block_running_sum_plan(wl.S, binding.BF16 if es == 2 else binding.F32)
        self.byte_parts = block_pass_bytes(wl.N, wl.S, wl.T, wl.d, es, self.plan)
        self.bytes = self.byte_parts["total"]

    def __call__(self):
        self.ar.attnres_block_pass(self.F, self.wl.N, self.wl.S, self.W, self.G, self.wl.eps,
                                   self.Src, self.O, self.lse, self.P, self.out)

    def launch_groups(self):
        """The pass's launches by kernel kind, each as the per-sublayer API
        call that makes it (for graph-timing one kind at a time)."""
        ar, wl, plan = self.ar, self.wl, self.plan
        groups = {"stage1": [], "merge": [], "freeze": []}
        for n in range(wl.N):
            k0 = n * wl.S
            O = [self.out[k0]] + [self.O[j - 1] for j in range(1, wl.S)]
            groups["stage1"].append(lambda n=n, k0=k0, O=O: ar.attnres_block_stage1(
                self.Src, n + 1, self.W[k0:k0 + wl.S], self.G[k0:k0 + wl.S], wl.eps, O, self.lse))
            m = 0
            for j in range(1, wl.S):
                groups["merge"].append(lambda k0=k0, j=j, m=m: ar.attnres_block_merge_parts(
                    self.O[j - 1], self.lse[j], self.P if m > 0 else None, self.F[k0 + m:], j - m,
                    self.P if plan[j] else None, self.W[k0 + j], self.G[k0 + j], wl.eps, self.out[k0 + j]))
                if plan[j]:
                    m = j
            if n + 1 < wl.N:
                groups["freeze"].append(lambda n=n, k0=k0, m=m: ar.attnres_block_summary_parts(
                    self.P if m > 0 else None, self.F[k0 + m:], wl.S - m, summary_out=self.Src[n + 1]))
        return groups


class DsplitStep:
    """The Block pass's N stage-1 reads (block n: the embedding and n block
    summaries as sources, the block's S queries) with the features split over
    P shards, as a tensor-parallel prefill lays them out: per block, every
    shard's partial score sums (added in turn, where devices would all-reduce
    them), then every shard's finish."""

    def __init__(self, wl, dev, P=DSPLIT_SHARDS):
        from depth_wise_attention_attnres_gb300 import binding
        self.ar = binding
        self.wl = wl
        self.P = P
        dt = inputs.DTYPES[wl.dtype]
        ds = wl.d // P
        g = inputs.generator(wl.seed, dev)
        src = inputs.history(wl.N, wl.T, wl.d, wl.dtype, g, dev, wl.depth_scaled)
        W = inputs.queries(wl.N * wl.S, wl.d, wl.w_std, g, dev)
        G = torch.ones((wl.N * wl.S, wl.d), dtype=torch.float32, device=dev)
        self.Src = [src[:, :, p * ds:(p + 1) * ds].contiguous() for p in range(P)]
        self.Wp = [W[:, p * ds:(p + 1) * ds].contiguous() for p in range(P)]
        self.Gp = [G[:, p * ds:(p + 1) * ds].contiguous() for p in range(P)]
        del src
        self.parts = [torch.empty(wl.T, n + 1, wl.S + 1, device=dev) for n in range(wl.N)]
        self.outs = [[torch.empty(wl.T, ds, device=dev, dtype=dt) for _ in range(wl.S)] for _ in range(P)]
        self.lse = torch.empty(wl.S, wl.T, device=dev)
        self.launches = wl.N * 2 * P
        es = 2 if wl.dtype == "bf16" else 4
        self.byte_parts = dsplit_stage1_bytes(wl.N, wl.S, wl.T, wl.d, es, P)
        self.bytes = self.byte_parts["total"]

    def partials(self, n, stream=None):
        S = self.wl.S
        for p in range(self.P):
            self.ar.attnres_stage1_dsplit_partials(self.Src[p], n + 1, self.Wp[p][n * S:(n + 1) * S],
                                                   self.Gp[p][n * S:(n + 1) * S], self.parts[n], p > 0,
                                                   stream=stream)

    def finish(self, n, stream=None):
        for p in range(self.P):
            self.ar.attnres_stage1_dsplit_finish(self.Src[p], n + 1, self.wl.d, self.parts[n], self.wl.eps,
                                                 self.outs[p], self.lse if p == 0 else None, stream=stream)

    def __call__(self):
        for n in range(self.wl.N):
            self.partials(n)
            self.finish(n)


class BlockBwdStep:
    """The Block pass backward: the forward pass runs once at set-up (its
    frozen summaries are what the backward reads); a step is one
    attnres_block_bwd over all N*S reads with seeded dL/dout."""

    def __init__(self, wl, dev):
        from depth_wise_attention_attnres_gb300 import binding
        self.ar = binding
        self.wl = wl
        fwd = BlockPassStep(wl, dev)
        fwd()
        self.Src, self.F, self.W, self.G = fwd.Src, fwd.F, fwd.W, fwd.G
        del fwd
        torch.cuda.empty_cache()
        g = inputs.generator(wl.seed + 4, dev)
        self.dOut = inputs.randn((wl.N * wl.S, wl.T, wl.d), wl.dtype, g, dev)
        self.dEmb = torch.zeros(wl.T, wl.d, device=dev)
        self.dF = torch.zeros(wl.N * wl.S, wl.T, wl.d, device=dev)
        self.dW = torch.zeros(wl.N * wl.S, wl.d, device=dev)
        self.dGamma = torch.zeros(wl.N * wl.S, wl.d, device=dev)
        self.scratch = torch.empty(binding.attnres_block_bwd_scratch_floats(wl.N, wl.S, wl.T, wl.d), device=dev)
        L = wl.N * wl.S
        self.launches = L + (L - wl.N) + wl.N * max(wl.S - 1, 0) + (wl.N - 1) + 2
        es = 2 if wl.dtype == "bf16" else 4
        batched = wl.d % 128 == 0 and wl.d <= 1024 and wl.N <= 8 and wl.S <= 8
        self.byte_parts = (block_bwd_bytes if batched else block_bwd_bytes_per_read)(wl.N, wl.S, wl.T, wl.d, es)
        self.bytes = self.byte_parts["total"]
        if batched:
            self.launches = wl.N + 1

    def __call__(self):
        self.ar.attnres_block_bwd(self.Src, self.F, self.wl.N, self.wl.S, self.W, self.G, self.wl.eps, self.dOut,
                                  self.dEmb, self.dF, self.dW, self.dGamma, self.scratch)


def time_dsplit_kernels(step, reps, stream):
    """Device time of the partials and finish launches of a d-split step."""
    acc = {"partials": 0.0, "finish": 0.0}
    marks = []
    with torch.cuda.stream(stream):
        for _ in range(reps):
            for n in range(step.wl.N):
                for kind in ("partials", "finish"):
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    getattr(step, kind)(n, stream=stream)
                    b.record(stream)
                    marks.append((kind, a, b))
    torch.cuda.synchronize()
    for kind, a, b in marks:
        acc[kind] += a.elapsed_time(b)
    return {k: v / reps for k, v in acc.items()}


def make_step(name, dev, op="read"):
    wl = inputs.WORKLOADS[name]
    if wl.kind == "full_pass":
        if op == "dsplit":
            raise ValueError("--op dsplit applies to Block-pass workloads")
        return FullPassStep(wl, dev, op)
    if wl.kind == "block_pass" and op == "dsplit":
        return DsplitStep(wl, dev)
    if wl.kind == "block_pass" and op == "bwd":
        return BlockBwdStep(wl, dev)
    if op != "read":
        raise ValueError("--op applies to Full-pass workloads (dsplit: Block-pass workloads)")
    if wl.kind == "block_pass":
        return BlockPassStep(wl, dev)
    raise ValueError(f"{name} is a parity case, not a benchmark workload")


def time_graph(step, steps, warmup, world, stream):
    """Capture one step in a CUDA graph; time `steps` replays with events."""
    with torch.cuda.stream(stream):
        step()  # first call outside capture (one-time attribute setup)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = start.elapsed_time(end) / steps
    return ms, graph


def time_block_kernels(step, reps, stream):
    """Device time per kernel kind of the Block pass, measured the way the
    step is: each kind's launches of one pass (its stage-1 reads, its merges,
    its freezes) are captured in a CUDA graph of their own and replayed `reps`
    times between CUDA events on the launching stream. Returns ms per pass
    and launches per pass for each kind. The kinds' sum differs from the
    step's own graph time by the overlap of neighbouring launches."""
    out = {}
    for kind, calls in step.launch_groups().items():
        if not calls:
            out[kind] = {"ms": 0.0, "launches": 0}
            continue
        with torch.cuda.stream(stream):
            for c in calls:
                c()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for c in calls:
                c()
        with torch.cuda.stream(stream):
            for _ in range(2):
                graph.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(reps):
                graph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        out[kind] = {"ms": a.elapsed_time(b) / reps, "launches": len(calls)}
        del graph
    # Leave the pass's buffers as a full pass leaves them.
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    return out


def block_roofline(step, ms_step, stream, peaks, reps=3):
    """Roofline block of a Block-pass line: the kernel kind with the largest
    share of the step, its algorithmic bytes per launch over its average
    launch duration (graph-timed), and every kind's time and share."""
    times = time_block_kernels(step, reps, stream)
    parts = step.byte_parts
    total = sum(v["ms"] for v in times.values()) or 1.0
    kernels = {}
    for k, v in times.items():
        if not v["launches"]:
            continue
        kernels[k] = {"ms": v["ms"], "launches": v["launches"],
                      "gbs": parts[k] / (v["ms"] / 1e3) / 1e9 if v["ms"] else None,
                      "share": v["ms"] / total,
                      "ms_in_step": v["ms"] / total * ms_step}
    top = max(kernels, key=lambda k: kernels[k]["ms"])
    g = kernels[top]["gbs"]
    name = {"stage1": "stage1_tc_kernel", "merge": "merge_tile_kernel", "freeze": "accum_fast_kernel"}[top]
    ratio = NCU_TRAFFIC_BLOCK.get((name, kernel_digest(KERNEL_FILES[name])), {}).get(step.wl.name)
    per_launch = parts[top] / kernels[top]["launches"]
    return {"kernel": name, "bound": "hbm", "achieved": g, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": g / peaks["hbm_gbs"], "frac_of_nominal_8000": g / NOMINAL_HBM_GBS,
            "peak_source": peaks["source"], "per_launch_bytes": per_launch,
            "traffic": None if ratio is None else ratio * per_launch,
            "per_kernel": kernels, "kinds_sum_over_step": total / ms_step,
            "note": "each kernel kind's launches of one pass graph-timed on their own; 'share' is of the "
                    "kinds' sum, 'ms_in_step' that share of the step's own graph time"}


def _device_tensors(step):
    return {k: v for k, v in vars(step).items() if isinstance(v, torch.Tensor) and v.is_cuda}


def _input_names(step):
    return ["F", "W", "G", "Src"] if isinstance(step, BlockPassStep) else ["V", "W", "G"]


def run_e2e(step, steps, warmup, stream):
    """The same metric through the public API with host buffers, as a serving
    loop runs it: every step copies its inputs host -> device from pinned
    memory, runs the pass, and copies its outputs device -> host, all inside
    the timed region. The three parts of consecutive steps overlap on three
    streams (step k's upload, step k-1's pass, step k-2's download), with two
    device buffer sets and events ordering every reuse."""
    import copy
    sets = [step, copy.copy(step)]
    for name, t in _device_tensors(step).items():
        setattr(sets[1], name, torch.empty_like(t))
    names = _input_names(step)

    def pinned_copy(t):
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        return h
    if isinstance(step, BlockPassStep):
        host_in = {"F": pinned_copy(step.F), "W": pinned_copy(step.W), "G": pinned_copy(step.G),
                   "Src": pinned_copy(step.Src[0])}
    else:
        host_in = {n: pinned_copy(getattr(step, n)) for n in names}
    host_out = [torch.empty(step.out.shape, dtype=step.out.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_out[0].numel() * host_out[0].element_size()

    dev = step.out.device
    # Large copies go out in slices on several streams per direction (one
    # stream per direction reached about 155 GB/s each way with both running,
    # several about 170).
    n_cs = E2E_COPY_STREAMS
    ups = [torch.cuda.Stream(device=dev) for _ in range(n_cs)]
    downs = [torch.cuda.Stream(device=dev) for _ in range(n_cs)]
    s_up, s_down = ups[0], downs[0]

    def sliced_copy(dst, src, streams):
        """dst.copy_(src) in slices along dim 0, slice c on streams[c]; the
        first stream waits for the others before it returns."""
        lead = streams[0]
        k = min(len(streams), dst.shape[0]) if dst.dim() > 0 and dst.numel() * dst.element_size() > (1 << 30) else 1
        if k == 1:
            dst.copy_(src, non_blocking=True)
            return
        start = torch.cuda.Event()
        start.record(lead)
        bounds = [dst.shape[0] * c // k for c in range(k + 1)]
        done = []
        for c in range(k):
            sc = streams[c]
            if c:
                sc.wait_event(start)
            with torch.cuda.stream(sc):
                dst[bounds[c]:bounds[c + 1]].copy_(src[bounds[c]:bounds[c + 1]], non_blocking=True)
            if c:
                e = torch.cuda.Event()
                e.record(sc)
                done.append(e)
        for e in done:
            lead.wait_event(e)

    def upload(st):
        for n in names:
            dst = st.Src[0] if n == "Src" else getattr(st, n)
            sliced_copy(dst, host_in[n], ups)
    graphs = []
    for st in sets:
        upload(st)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            st()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            st()
        graphs.append(g)
    torch.cuda.synchronize()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    computed = [ev(), ev()]
    downloaded = [ev(), ev()]
    uploaded = [ev(), ev()]
    for e in computed + downloaded:
        e.record(stream)

    def run(k):
        i = k % 2
        with torch.cuda.stream(s_up):
            s_up.wait_event(computed[i])          # set i's inputs no longer in use
            upload(sets[i])
            uploaded[i].record(s_up)
        with torch.cuda.stream(stream):
            stream.wait_event(uploaded[i])
            stream.wait_event(downloaded[i])      # set i's outputs already copied out
            graphs[i].replay()
            computed[i].record(stream)
        with torch.cuda.stream(s_down):
            s_down.wait_event(computed[i])
            sliced_copy(host_out[i], sets[i].out, downs)
            downloaded[i].record(s_down)

    for k in range(warmup):
        run(k)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(s_up)
    for k in range(steps):
        run(k)
    end.record(s_down)
    torch.cuda.synchronize()
    del graphs
    return start.elapsed_time(end) / steps, h2d, d2h


MAX_ORACLE_ROWS = 8192  # token rows gathered for the oracle at most


def oracle_inputs(name, device, rows_cap=MAX_ORACLE_ROWS, step=None):
    """The workload's stored inputs restricted to a stride sample of at most
    rows_cap token rows, as CPU tensors. They are drawn where the bench draws
    them (on the GPU when there is one, so the oracle sees the same bits) and
    only the sampled rows are copied back; `step` reuses tensors already on
    the device. Returns (kind-specific inputs, rows)."""
    wl = inputs.WORKLOADS[name]
    rows = inputs.sample_rows(wl.T, rows_cap)
    if wl.kind == "full_pass":
        V, W, G = (step.V, step.W, step.G) if step is not None else inputs.full_inputs(wl, device)
        r = rows.to(V.device)
        got = (V[:, r].cpu(), W.cpu().double(), G.cpu().double())
    else:
        if step is not None:
            emb, F, W, G = step.Src[0], step.F, step.W, step.G
        else:
            emb, F, W, G = inputs.block_inputs(wl, device)
        r = rows.to(F.device)
        got = (emb[r].cpu(), F[:, r].cpu(), W.cpu().double(), G.cpu().double())
    return got, rows


def cpu_baseline(name, target_s=12.0, device="cpu", step=None):
    """The fp64 oracle, as it stands, on a bounded sample of token rows (at
    most MAX_ORACLE_ROWS, sized to take about target_s seconds)."""
    import oracle
    oracle.build()
    wl = inputs.WORKLOADS[name]
    data, all_rows = oracle_inputs(name, device, step=step)
    if wl.kind == "full_pass":
        V, W64, G64 = data

        def run(sel):
            oracle.full_pass(V[:, sel], wl.R, W64, G64, wl.eps)
    else:
        emb, F, W64, G64 = data

        def run(sel):
            oracle.block_pass(emb[sel], F[:, sel, :], wl.N, wl.S, W64, G64, wl.eps)
    m = len(all_rows)
    probe = torch.linspace(0, m - 1, min(16, m)).round().long().unique()
    t0 = time.perf_counter()
    run(probe)
    dt = max(time.perf_counter() - t0, 1e-6)
    nrows = int(min(m, max(16, len(probe) * target_s / dt)))
    sel = torch.linspace(0, m - 1, nrows).round().long().unique()
    t0 = time.perf_counter()
    run(sel)
    dt = time.perf_counter() - t0
    cores = oracle.threads()
    # The same oracle on one thread, on a smaller sample (about 1/8 of the time).
    one = sel[:max(16, len(sel) // (8 * max(cores, 1)) + 1)]
    oracle.set_threads(1)
    try:
        t1 = time.perf_counter()
        run(one)
        dt1 = time.perf_counter() - t1
    finally:
        oracle.set_threads(cores)
    return {"value": len(sel) / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(sel)} of {wl.T} token rows (stride-sampled) of {name}, fp64, "
                      f"{dt:.1f} s; tokens are independent so tokens/s scales",
            "single_thread": {"value": len(one) / dt1, "unit": "tokens/s",
                              "sample": f"{len(one)} token rows, {dt1:.1f} s"}}, (run, sel)


def time_sustained(graph, ms_probe, seconds, stream):
    """Replays an already captured step graph for at least `seconds` between
    CUDA events (after the regular timing, which warmed it up)."""
    steps = max(1, int(math.ceil(seconds * 1e3 / max(ms_probe, 1e-3))))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(steps):
            graph.replay()
        b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps, steps


def full_roofline(step, ms, peaks, op):
    kname = "full_bwd_bulk_kernel" if op == "bwd" else "full_fwd_bulk_kernel"
    gbs = step.bytes / (ms / 1e3) / 1e9
    traffic = NCU_TRAFFIC.get((kname, kernel_digest(KERNEL_FILES[kname])))
    return {"kernel": kname, "bound": "hbm", "achieved": gbs,
            "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
            "frac_of_nominal_8000": gbs / NOMINAL_HBM_GBS,
            "peak_source": peaks["source"],
            "traffic": None if traffic is None else traffic * step.bytes / step.launches,
            "per_launch_bytes": step.bytes / step.launches,
            "note": "the step is R launches of this one kernel back to back in a CUDA graph; "
                    "average launch duration = step time / R (gaps included)"}


def measure_extra(name, dev, steps, warmup, world, stream, peaks):
    """One more bench workload in the same run: its step graph-timed like the
    headline (K steps after W warm-up replays); Block passes add their
    per-kernel roofline."""
    step = make_step(name, dev)
    ms, graph = time_graph(step, steps, warmup, world, stream)
    del graph
    ms = max_over_ranks(ms, world)
    gbs = step.bytes / (ms / 1e3) / 1e9
    wl = step.wl
    rec = {"ms_per_step": ms, "steps": steps, "tokens_per_s": wl.T * world / (ms / 1e3),
           "algorithmic_gbs": gbs, "frac": gbs / peaks["hbm_gbs"], "frac_of_nominal_8000": gbs / NOMINAL_HBM_GBS,
           "gpu_launches": step.launches * steps}
    if isinstance(step, BlockPassStep):
        rec["roofline"] = block_roofline(step, ms, stream, peaks)
    else:
        rec["roofline"] = full_roofline(step, ms, peaks, "read")
    del step
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def ours(args):
    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    barrier(world)
    __graft_entry__.build()
    peaks = measured_peaks()
    stream = torch.cuda.Stream(device=dev)
    wl = inputs.WORKLOADS[args.workload]
    step = make_step(args.workload, dev, args.op)

    with ClockSampler(local) as clocks:
        ms, graph = time_graph(step, args.steps, args.warmup, world, stream)
    ms = max_over_ranks(ms, world)
    tokens = wl.T * world
    value = job_throughput(wl.T, world, ms)
    gbs = step.bytes / (ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "kind": wl.kind, "T": wl.T, "d": wl.d,
                   "reads" if wl.kind == "full_pass" else "blocks": wl.R if wl.kind == "full_pass" else wl.N,
                   **({"S": wl.S} if wl.kind == "block_pass" else {}),
                   **({"op": args.op} if args.op != "read" else {}),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (129 MB); no flush",
                   "timing": "CUDA graph of one step, CUDA events on the launching stream"},
        "algorithmic_gbs": gbs,
        "timed_region_s": ms * args.steps / 1e3,
        "gpu_launches": step.launches * args.steps,
    }
    line["clocks"] = clocks.summary()
    if not args.no_sustained:
        with ClockSampler(local) as sclocks:
            sms, ssteps = time_sustained(graph, ms, SUSTAINED_S, stream)
        sms = max_over_ranks(sms, world)
        line["sustained"] = {"ms_per_step": sms, "steps": ssteps, "timed_region_s": sms * ssteps / 1e3,
                             "value": job_throughput(wl.T, world, sms), "unit": "tokens/s",
                             "algorithmic_gbs": step.bytes / (sms / 1e3) / 1e9,
                             "clocks": sclocks.summary(),
                             "note": "the same step graph replayed back to back for at least "
                                     f"{SUSTAINED_S:.0f} s after the K timed steps"}
    del graph
    torch.cuda.synchronize()

    if wl.kind == "full_pass":
        line["roofline"] = full_roofline(step, ms, peaks, args.op)
    elif isinstance(step, BlockBwdStep):
        g = step.byte_parts["total"] / (ms / 1e3) / 1e9
        batched = step.launches == step.wl.N + 1
        ratio = NCU_TRAFFIC.get(("block_bwd_batched_kernel", kernel_digest("block_bwd.cu"))) if batched else None
        line["roofline"] = {
            "kernel": "block_bwd_batched_kernel" if batched else "full_bwd_bulk_kernel", "bound": "hbm",
            "achieved": g, "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": g / peaks["hbm_gbs"], "frac_of_nominal_8000": g / NOMINAL_HBM_GBS,
            "peak_source": peaks["source"],
            "traffic": None if ratio is None else ratio * step.byte_parts["total"] / step.wl.N,
            "byte_parts": step.byte_parts,
            "note": "whole step: one batched launch per block (all S reads)" if batched else
                    "whole step: the per-read backward launches carry "
                    f"{step.byte_parts['read'] / step.byte_parts['total']:.0%} of the algorithmic bytes"}
    elif isinstance(step, DsplitStep):
        times = time_dsplit_kernels(step, 3, stream)
        parts = step.byte_parts
        kernels = {k: {"ms": times[k], "gbs": parts[k] / (times[k] / 1e3) / 1e9} for k in times}
        top = max(kernels, key=lambda k: kernels[k]["ms"])
        g = kernels[top]["gbs"]
        line["config"]["shards"] = step.P
        line["roofline"] = {
            "kernel": {"partials": "dsplit_partials_tc_kernel", "finish": "dsplit_finish_tc_kernel"}[top],
            "bound": "hbm", "achieved": g, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": g / peaks["hbm_gbs"], "frac_of_nominal_8000": g / NOMINAL_HBM_GBS,
            "peak_source": peaks["source"], "traffic": None, "per_kernel": kernels}
    else:
        line["roofline"] = block_roofline(step, ms, stream, peaks)

    if not args.no_e2e:
        ems, h2d, d2h = run_e2e(step, max(4, min(args.steps, 20)), 3, stream)
        ems = max_over_ranks(ems, world)
        line["e2e"] = {"value": tokens / (ems / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "ms_per_step": ems,
                       "note": "uploads, passes and downloads of consecutive steps overlap on three streams"}
        torch.cuda.empty_cache()
    base_data = None
    if rank == 0 and not args.no_cpu_baseline:
        # The oracle's rows are taken from the inputs already on the device.
        base_data = step
    base = None
    if base_data is not None:
        base, _ = cpu_baseline(args.workload, step=base_data)
    del step, base_data
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    if not args.no_extras and args.op == "read":
        line["extras"] = {}
        for name in EXTRA_WORKLOADS:
            if name != args.workload:
                line["extras"][name] = measure_extra(name, dev, args.steps, args.warmup, world, stream, peaks)
    if base is not None:
        line["cpu_baseline"] = base
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = inputs.WORKLOADS[args.workload]
    # The inputs are drawn on the GPU when there is one (the same bits as the
    # bench's own arm); only the oracle's fp64 CPU run is timed.
    device = "cuda" if torch.cuda.is_available() else "cpu"
    base, (run, rows) = cpu_baseline(args.workload, target_s=4.0, device=device)
    if device == "cuda":
        torch.cuda.empty_cache()
    for _ in range(args.warmup):
        run(rows[:8])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run(rows)
    dt = (time.perf_counter() - t0) / args.steps
    value = len(rows) / dt
    base["value"] = value
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "kind": wl.kind, "T": wl.T, "d": wl.d,
                   "sample_rows_per_step": len(rows)},
        "cpu_baseline": base,
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(
        n for n, w in inputs.WORKLOADS.items() if w.kind != "full_read"))
    p.add_argument("--op", choices=["read", "prenorm", "prenorm_both", "bwd", "dynq", "dsplit"], default="read",
                   help="Full pass: plain reads, reads emitting the sublayer pre-norm instead of "
                        "their result, or both, the pass backward (dV, dW, dGamma), or reads with "
                        "input-dependent queries (projection + read). Block pass: dsplit, the stage-1 "
                        "reads with the features split over 4 shards; bwd, the pass backward")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-extras", "--no-block", dest="no_extras", action="store_true",
                   help="skip the other bench workloads measured after the headline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-sustained", action="store_true")
    args = p.parse_args()
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    if args.op != "read":
        # The variants are measured on the device alone.
        args.no_e2e = args.no_extras = args.no_cpu_baseline = True
    if args.impl == "reference":
        reference(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
