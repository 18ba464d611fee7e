"""The next rows at full size, in the launch configuration bench.py times (GPU).

Each variant step of bench.py runs once on its workload; sampled token rows
are checked against the oracle (every output of a read depends only on its
own token's rows, so the sample is exact). Sums over all tokens (dw, dgamma)
are covered by the small cases of the row's own test file.
"""
import numpy as np
import pytest
import torch

import bench
import oracle
from depth_wise_attention_attnres_gb300 import inputs
from tests._gpu import TOL, dev, rel_err

pytestmark = pytest.mark.gpu

FULL = "full_pass_64x8192x896_bf16"
BLOCK = "block_pass_8x8x16384x1024_bf16"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _run(step):
    step()
    torch.cuda.synchronize()
    assert step.ar.attnres_device_status() == 0


def test_prenorm_pass_full_size_sampled():
    """64 reads emitting the result and its sublayer pre-norm (`--op prenorm_both`)."""
    step = bench.make_step(FULL, dev(), "prenorm_both")
    _run(step)
    wl = step.wl
    rows = inputs.sample_rows(wl.T, 48).to(dev())
    zs = oracle.full_pass(step.V[:, rows, :].cpu(), wl.R, step.W.cpu().double(), step.G.cpu().double(), wl.eps)
    worst_z = worst_n = 0.0
    for r in range(wl.R):
        ref = oracle.prenorm(zs[r], step.Gpre[r].cpu().double().numpy(), wl.eps)
        worst_n = max(worst_n, rel_err(step.normed[r][rows], ref))
        worst_z = max(worst_z, rel_err(step.out[r][rows], zs[r]))
    assert worst_n <= TOL["bf16"] and worst_z <= TOL["bf16"], (worst_n, worst_z)


def test_dynamic_query_pass_full_size_sampled():
    """64 reads, each with its query projected from its newest source (`--op dynq`)."""
    step = bench.make_step(FULL, dev(), "dynq")
    _run(step)
    wl = step.wl
    rows = inputs.sample_rows(wl.T, 32).to(dev())
    Vs = step.V[:, rows, :].cpu()
    worst = 0.0
    for r in range(wl.R):
        q = oracle.query_projection(Vs[r], step.Wq[r].cpu())
        ref, _ = oracle.read_dynamic_query([Vs[i] for i in range(r + 1)], q, step.G[r].cpu().double().numpy(),
                                           wl.eps)
        worst = max(worst, rel_err(step.out[r][rows], ref))
    assert worst <= TOL["bf16"], worst


def test_pass_backward_full_size_sampled():
    """The 64-read pass backward (`--op bwd`): dV on sampled token rows."""
    step = bench.make_step(FULL, dev(), "bwd")
    _run(step)
    wl = step.wl
    rows = inputs.sample_rows(wl.T, 24).to(dev())
    Vs = step.V[:, rows, :].cpu()
    ref = np.zeros((wl.R, len(rows), wl.d))
    for r in range(wl.R):
        rV, _, _ = oracle.full_read_bwd(Vs, r + 1, step.W[r].cpu().double(), step.G[r].cpu().double(), wl.eps,
                                        step.dZ[r][rows].cpu())
        ref[: r + 1] += rV
    assert rel_err(step.dV[:, rows, :], ref) <= TOL["f32"]


def test_dsplit_stage1_full_size_sampled():
    """The Block workload's stage-1 reads over 4 feature shards (`--op dsplit`):
    after the step the buffers hold the last block's reads (8 sources)."""
    step = bench.make_step(BLOCK, dev(), "dsplit")
    _run(step)
    wl = step.wl
    n = wl.N
    rows = inputs.sample_rows(wl.T, 64).to(dev())
    src = torch.cat([step.Src[p][:, rows, :] for p in range(step.P)], dim=2).cpu()
    k0 = (n - 1) * wl.S
    W = torch.cat(step.Wp, dim=1)[k0:k0 + wl.S].cpu().double()
    G = torch.cat(step.Gp, dim=1)[k0:k0 + wl.S].cpu().double()
    refO, refL = oracle.block_stage1(src, n, W, G, wl.eps)
    for j in range(wl.S):
        got = torch.cat([step.outs[p][j][rows] for p in range(step.P)], dim=1)
        assert rel_err(got, refO[j]) <= TOL["bf16"], f"O[{j}]"
    assert float(np.max(np.abs(step.lse[:, rows].cpu().double().numpy() - refL))) <= 1e-4


def test_block_pass_backward_full_size_sampled():
    """The Block pass backward (`--op bwd` on the Block workload): dEmb and dF on
    sampled token rows (the forward's frozen summaries as the sources)."""
    step = bench.make_step(BLOCK, dev(), "bwd")
    _run(step)
    wl = step.wl
    rows = inputs.sample_rows(wl.T, 24).to(dev())
    rE, rF, _, _ = oracle.block_pass_bwd(step.Src[:, rows, :].cpu(), step.F[:, rows, :].cpu(), wl.N, wl.S,
                                         step.W.cpu().double().numpy(), step.G.cpu().double().numpy(), wl.eps,
                                         step.dOut[:, rows, :].cpu())
    assert rel_err(step.dEmb[rows], rE) <= TOL["f32"]
    assert rel_err(step.dF[:, rows, :], rF) <= TOL["f32"]
