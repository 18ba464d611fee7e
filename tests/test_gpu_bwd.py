"""Backward of a read (dV, dw, dgamma): CUDA vs the pinned oracle (GPU).

The gradients are stored in fp32 and computed in fp32 from sources and dz
that the oracle widens exactly, so the fp32 bar (1e-5, max-norm relative)
holds for bf16 sources too.
"""
import numpy as np
import pytest
import torch

import oracle
from depth_wise_attention_attnres_gb300 import binding as ar
from depth_wise_attention_attnres_gb300 import inputs
from tests._gpu import TOL, dev, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _case(seed, n, T, d, dt, dzt):
    g = inputs.generator(seed, dev())
    V = inputs.history(n, T, d, dt, g, dev(), depth_scaled=True)
    w = inputs.queries(1, d, 0.05, g, dev())[0].contiguous()
    gam = (1 + 0.3 * inputs.queries(1, d, 1.0, g, dev())[0]).contiguous()
    dz = inputs.randn((T, d), dzt, g, dev())
    return V, w, gam, dz


@pytest.mark.parametrize("dt,dzt", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")])
@pytest.mark.parametrize("n,T,d", [(5, 70, 896), (8, 33, 640), (3, 33, 100), (1, 16, 256),
                                   (64, 9, 1024), (300, 5, 128), (16, 41, 2048), (7, 19, 256)])
def test_full_bwd_vs_oracle(dt, dzt, n, T, d):
    V, w, gam, dz = _case(30, n, T, d, dt, dzt)
    dV = torch.zeros(n, T, d, device=dev())
    dw = torch.zeros(d, device=dev())
    dg = torch.zeros(d, device=dev())
    ar.attnres_full_bwd(V, n, w, gam, 1e-6, dz, dV, dw, dg)
    torch.cuda.synchronize()
    rV, rw, rg = oracle.full_read_bwd(V.cpu(), n, w.cpu().double(), gam.cpu().double(), 1e-6, dz.cpu())
    assert rel_err(dV, rV) <= TOL["f32"]
    assert rel_err(dw, rw) <= TOL["f32"]
    assert rel_err(dg, rg) <= TOL["f32"]
    assert ar.attnres_device_status() == 0


def test_full_bwd_accumulates_and_skips_null_gains():
    n, T, d = 6, 40, 512
    V, w, gam, dz = _case(31, n, T, d, "bf16", "bf16")
    base = inputs.randn((n, T, d), "f32", inputs.generator(32, dev()), dev())
    dV = base.clone()
    dw = torch.full((d,), 0.5, device=dev())
    ar.attnres_full_bwd(V, n, w, gam, 1e-6, dz, dV, dw, None)
    ar.attnres_full_bwd(V, n, w, gam, 1e-6, dz, dV, dw, None)
    torch.cuda.synchronize()
    rV, rw, _ = oracle.full_read_bwd(V.cpu(), n, w.cpu().double(), gam.cpu().double(), 1e-6, dz.cpu())
    assert rel_err(dV, base.cpu().double().numpy() + 2 * rV) <= TOL["f32"]
    assert rel_err(dw, 0.5 + 2 * rw) <= TOL["f32"]


def test_full_pass_backward_composes_read_by_read():
    """A pass's backward: read r's gradient is added to dV[0 .. r] for every r
    (what a model does in reverse layer order); compare with the sum of the
    oracle's per-read gradients."""
    R, T, d = 6, 24, 256
    g = inputs.generator(33, dev())
    V = inputs.history(R, T, d, "bf16", g, dev(), depth_scaled=True)
    W = inputs.queries(R, d, 0.05, g, dev())
    G = torch.ones(R, d, device=dev())
    dZ = inputs.randn((R, T, d), "f32", g, dev())
    dV = torch.zeros(R, T, d, device=dev())
    dW = torch.zeros(R, d, device=dev())
    for r in reversed(range(R)):
        ar.attnres_full_bwd(V, r + 1, W[r], G[r], 1e-6, dZ[r], dV, dW[r], None)
    torch.cuda.synchronize()
    ref = np.zeros((R, T, d))
    Vc = V.cpu()
    for r in range(R):
        rV, rw, _ = oracle.full_read_bwd(Vc, r + 1, W[r].cpu().double(), G[r].cpu().double(), 1e-6,
                                         dZ[r].cpu())
        ref[: r + 1] += rV
        assert rel_err(dW[r], rw) <= TOL["f32"], f"dw of read {r}"
    assert rel_err(dV, ref) <= TOL["f32"]
