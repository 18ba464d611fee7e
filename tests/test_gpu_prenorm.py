"""Sublayer pre-norm fused into the aggregation epilogues: CUDA vs oracle (GPU).

The oracle side is the read (or merge) by definition followed by the pinned
pre-norm, gamma_pre * z / sqrt(mean(z^2) + eps_pre) (DepthBench reading notes
section 2.3: f_l = F_l(RMSNorm_pre,l(z_l))).
"""
import numpy as np
import pytest
import torch

import oracle
from depth_wise_attention_attnres_gb300 import binding as ar
from depth_wise_attention_attnres_gb300 import inputs
from tests._gpu import TOL, dev, dtype_of, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _gain(d, g):
    return 1 + 0.5 * inputs.queries(1, d, 1.0, g, dev())[0].contiguous()


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("n,T,d", [(5, 70, 896), (8, 33, 640), (3, 33, 100), (1, 16, 256), (4, 9, 1024)])
@pytest.mark.parametrize("with_z", [True, False])
def test_full_fwd_prenorm(dt, n, T, d, with_z):
    g = inputs.generator(20, dev())
    V = inputs.history(n, T, d, dt, g, dev(), depth_scaled=True)
    w = inputs.queries(1, d, 0.05, g, dev())[0].contiguous()
    gam = _gain(d, g)
    gpre = _gain(d, g)
    out = torch.empty(T, d, device=dev(), dtype=dtype_of(dt)) if with_z else None
    normed = torch.empty(T, d, device=dev(), dtype=dtype_of(dt))
    ar.attnres_full_fwd_prenorm(V, n, w, gam, 1e-6, gpre, 1e-5, out, normed)
    torch.cuda.synchronize()
    z, _ = oracle.full_read(V.cpu(), n, w.cpu().double(), gam.cpu().double(), 1e-6)
    ref = oracle.prenorm(z, gpre.cpu().double().numpy(), 1e-5)
    assert rel_err(normed, ref) <= TOL[dt]
    if with_z:
        assert rel_err(out, z) <= TOL[dt]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_full_pass_prenorm(dt):
    R, T, d = 6, 40, 256
    g = inputs.generator(21, dev())
    V = inputs.history(R, T, d, dt, g, dev(), depth_scaled=True)
    W = inputs.queries(R, d, 0.05, g, dev())
    G = torch.ones(R, d, device=dev())
    Gpre = 1 + 0.5 * inputs.queries(R, d, 1.0, g, dev())
    normed = torch.empty(R, T, d, device=dev(), dtype=dtype_of(dt))
    out = torch.empty(R, T, d, device=dev(), dtype=dtype_of(dt))
    ar.attnres_full_pass_prenorm(V, W, G, 1e-6, Gpre, 1e-6, out, normed)
    torch.cuda.synchronize()
    zs = oracle.full_pass(V.cpu(), R, W.cpu().double(), G.cpu().double(), 1e-6)
    for r in range(R):
        ref = oracle.prenorm(zs[r], Gpre[r].cpu().double().numpy(), 1e-6)
        assert rel_err(normed[r], ref) <= TOL[dt], f"read {r}"
        assert rel_err(out[r], zs[r]) <= TOL[dt], f"read {r} z"
    # Without z: the same normalised rows.
    normed2 = torch.empty_like(normed)
    ar.attnres_full_pass_prenorm(V, W, G, 1e-6, Gpre, 1e-6, None, normed2)
    torch.cuda.synchronize()
    assert torch.equal(normed2, normed)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("T,d", [(100, 1024), (33, 2048), (64, 896), (10, 100), (41, 1096)])
@pytest.mark.parametrize("mode", ["extend", "start", "as_is"])
@pytest.mark.parametrize("with_z", [True, False])
def test_merge_prenorm(dt, T, d, mode, with_z):
    n = 3
    g = inputs.generator(22, dev())
    Src = inputs.history(n, T, d, dt, g, dev())
    w = inputs.queries(1, d, 0.05, g, dev())
    gam = 1 + 0.3 * inputs.queries(1, d, 1.0, g, dev())
    gpre = _gain(d, g)
    P0 = inputs.randn((T, d), "f32", g, dev(), scale=2.0)
    f = inputs.randn((T, d), dt, g, dev())
    refO, refL = oracle.block_stage1(Src.cpu(), n, w.cpu().double(), gam.cpu().double(), 1e-6)
    O = torch.from_numpy(refO[0]).to(dev(), dtype=dtype_of(dt))
    lse = torch.from_numpy(refL[0]).to(dev(), dtype=torch.float32)
    P = P0.clone()
    f_prev = None if mode == "as_is" else f
    empty = mode == "start"
    out = torch.empty(T, d, device=dev(), dtype=dtype_of(dt)) if with_z else None
    normed = torch.empty(T, d, device=dev(), dtype=dtype_of(dt))
    ar.attnres_block_merge_prenorm(O, lse, P, f_prev, empty, w[0].contiguous(), gam[0].contiguous(),
                                   1e-6, gpre, 1e-5, out, normed)
    torch.cuda.synchronize()
    # The merge by definition over {Src, P_new}; the stage-1 result enters as
    # stored (rounded), as on the GPU, so compare with the definition's read.
    z, p_new = oracle.block_merge(Src.cpu(), n, P0.cpu(), None if f_prev is None else f.cpu(), empty,
                                  w[0].cpu().double(), gam[0].cpu().double(), 1e-6)
    ref = oracle.prenorm(z, gpre.cpu().double().numpy(), 1e-5)
    assert rel_err(normed, ref) <= TOL[dt]
    if with_z:
        assert rel_err(out, z) <= TOL[dt]
    if f_prev is not None:
        assert rel_err(P, p_new) <= TOL["f32"]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("T,d", [(50, 1024), (7, 3), (33, 2048)])
def test_rmsnorm(dt, T, d):
    g = inputs.generator(23, dev())
    x = inputs.randn((T, d), dt, g, dev(), scale=3.0)
    gam = _gain(d, g)
    out = torch.empty_like(x)
    ar.attnres_rmsnorm(x, gam, 1e-5, out)
    torch.cuda.synchronize()
    ref = oracle.prenorm(x.cpu(), gam.cpu().double().numpy(), 1e-5)
    assert rel_err(out, ref) <= TOL[dt]
    # in place
    y = x.clone()
    ar.attnres_rmsnorm(y, gam, 1e-5, y)
    torch.cuda.synchronize()
    assert torch.equal(y, out)
