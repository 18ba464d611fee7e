"""Seeded synthetic inputs for the AttnRes aggregation (no method arithmetic).

This module is shared by the CUDA path's tests and benchmark and by the fp64
oracle's tests. It only draws random numbers and casts them to the storage
dtype; it computes nothing of the aggregation itself.

The pages' workloads are language-model pretraining runs (FineWeb-Edu, context
2048, 400M to 1.6B models). Neither data nor trained weights are available, so
Gaussian tensors of the pages' shapes stand in for the stored sublayer outputs:

* Full AttnRes history: v_i ~ N(0, 1) * sqrt(i + 1) (i = 0 is the embedding),
  so later outputs are larger, the growth the key RMSNorm exists to neutralise
  (LLMRes blog, "Kimi AttnRes").
* Block AttnRes: embedding and sublayer outputs ~ N(0, 1).
* Pseudo-queries w_l ~ N(0, sigma^2) per read (sigma 0.02 or 0.05); key
  RMSNorm gain gamma = 1; eps = 1e-6.

Draw order for one seed (one torch.Generator): the history / embedding first,
then the sublayer outputs in order, then the rows of W. fp32 draws are cast to
bf16 with round-to-nearest-even (torch's cast).
"""
from __future__ import annotations

import dataclasses
import math

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One of the five standard workloads (shapes from the pages' models)."""

    name: str
    kind: str            # "full_read", "full_pass" or "block_pass"
    T: int
    d: int
    dtype: str           # storage dtype: "f32" or "bf16"
    w_std: float
    n_src: int = 0       # full_read: sources of the one read
    R: int = 0           # full_pass: number of reads (history length)
    N: int = 0           # block_pass: blocks
    S: int = 0           # block_pass: sublayers per block
    eps: float = 1e-6
    seed: int = 0
    depth_scaled: bool = True

    @property
    def tokens(self) -> int:
        return self.T


WORKLOADS = {
    # One read over the embedding + 7 sublayer outputs, fp32, T=256, d=256.
    "full_read_8x256x256_f32": Workload(
        "full_read_8x256x256_f32", "full_read", T=256, d=256, dtype="f32",
        w_std=0.02, n_src=8),
    # 400M model at 32 layers x d=896: 64 sublayers, T = 4 x 2048 tokens.
    "full_pass_64x8192x896_bf16": Workload(
        "full_pass_64x8192x896_bf16", "full_pass", T=8192, d=896, dtype="bf16",
        w_std=0.02, R=64),
    # Block AttnRes, 64 sublayers in 8 blocks of 8, d=1024, T=16384.
    "block_pass_8x8x16384x1024_bf16": Workload(
        "block_pass_8x8x16384x1024_bf16", "block_pass", T=16384, d=1024,
        dtype="bf16", w_std=0.02, N=8, S=8, depth_scaled=False),
    # The same blocks at 2048 tokens (about 1.2 GB on the device with the
    # backward's buffers): a case small enough for profiler captures whose
    # per-launch data still exceeds the 129 MB L2.
    "block_pass_8x8x2048x1024_bf16": Workload(
        "block_pass_8x8x2048x1024_bf16", "block_pass", T=2048, d=1024,
        dtype="bf16", w_std=0.02, N=8, S=8, depth_scaled=False),
    # Deep-narrow 70 layers x d=640: 140 sublayers + the LM-head read.
    "full_pass_141x32768x640_bf16": Workload(
        "full_pass_141x32768x640_bf16", "full_pass", T=32768, d=640,
        dtype="bf16", w_std=0.05, R=141),
    # The long-context blocks at 8192 tokens (about 4 GB on the device): a case
    # small enough for profiler captures of every launch of a pass, whose
    # per-launch data still exceeds the 129 MB L2.
    "block_pass_8x6x8192x2048_bf16": Workload(
        "block_pass_8x6x8192x2048_bf16", "block_pass", T=8192, d=2048,
        dtype="bf16", w_std=0.02, N=8, S=6, depth_scaled=False),
    # Long-context prefill, 128K tokens, d=2048, 48 sublayers in 8 blocks of 6.
    "block_pass_8x6x131072x2048_bf16": Workload(
        "block_pass_8x6x131072x2048_bf16", "block_pass", T=131072, d=2048,
        dtype="bf16", w_std=0.02, N=8, S=6, depth_scaled=False),
}


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def history(n: int, T: int, d: int, dtype: str, g: torch.Generator, device,
            depth_scaled: bool = True) -> torch.Tensor:
    """[n, T, d] stored history; slice i ~ N(0,1) * sqrt(i+1) if depth_scaled."""
    out = torch.empty((n, T, d), dtype=DTYPES[dtype], device=device)
    for i in range(n):
        x = torch.randn((T, d), generator=g, device=device, dtype=torch.float32)
        if depth_scaled:
            x.mul_(math.sqrt(i + 1))
        out[i].copy_(x)
    return out


def queries(R: int, d: int, std: float, g: torch.Generator, device) -> torch.Tensor:
    """[R, d] fp32 pseudo-queries ~ N(0, std^2)."""
    return torch.randn((R, d), generator=g, device=device, dtype=torch.float32).mul_(std)


def full_inputs(wl: Workload, device="cpu", seed=None):
    """History V, queries W, gains Gamma for a full_read / full_pass workload."""
    g = generator(wl.seed if seed is None else seed, device)
    n = wl.n_src if wl.kind == "full_read" else wl.R
    R = 1 if wl.kind == "full_read" else wl.R
    V = history(n, wl.T, wl.d, wl.dtype, g, device, wl.depth_scaled)
    W = queries(R, wl.d, wl.w_std, g, device)
    Gamma = torch.ones((R, wl.d), dtype=torch.float32, device=device)
    return V, W, Gamma


def block_inputs(wl: Workload, device="cpu", seed=None):
    """Embedding [T, d], sublayer outputs F [N*S, T, d], W, Gamma [N*S, d]."""
    g = generator(wl.seed if seed is None else seed, device)
    emb = history(1, wl.T, wl.d, wl.dtype, g, device, False)[0]
    F = history(wl.N * wl.S, wl.T, wl.d, wl.dtype, g, device, wl.depth_scaled)
    W = queries(wl.N * wl.S, wl.d, wl.w_std, g, device)
    Gamma = torch.ones((wl.N * wl.S, wl.d), dtype=torch.float32, device=device)
    return emb, F, W, Gamma


def randn(shape, dtype: str, g: torch.Generator, device, scale: float = 1.0) -> torch.Tensor:
    """Plain N(0, scale^2) draw cast to a storage dtype (for small test cases)."""
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(DTYPES[dtype])


def sample_rows(T: int, n: int) -> torch.Tensor:
    """Deterministic stride-sampled token rows (first and last row included)."""
    n = max(1, min(n, T))
    if n == 1:
        return torch.zeros(1, dtype=torch.int64)
    idx = torch.linspace(0, T - 1, n, dtype=torch.float64).round().to(torch.int64)
    return torch.unique(idx)
