"""Full AttnRes read and pass: CUDA path vs the fp64 oracle (GPU)."""
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


def _read_case(n, T, d, dt, w_std=0.05, seed=0, offset=0, out_dt=None, eps=1e-6, gamma_rand=True):
    g = inputs.generator(seed, dev())
    base = inputs.history(n, T * d + offset, 1, dt, g, dev()).view(n, -1) if offset else None
    if offset:
        V = base[:, offset:].reshape(n, T, d)   # sources with a misaligned start
    else:
        V = inputs.history(n, T, d, dt, g, dev())
    w = inputs.queries(1, d, w_std, g, dev())[0]
    gamma = (1 + 0.3 * inputs.queries(1, d, 1.0, g, dev())[0]) if gamma_rand else torch.ones(d, device=dev())
    out = torch.empty(T, d, device=dev(), dtype=dtype_of(out_dt or dt))
    ar.attnres_full_fwd(V, n, w, gamma, eps, out)
    torch.cuda.synchronize()
    ref, _ = oracle.full_read(V.cpu(), n, w.cpu().double(), gamma.cpu().double(), eps)
    return out, ref


def test_standard_single_read_f32():
    """One read over the embedding + 7 outputs, T=256, d=256, fp32."""
    wl = inputs.WORKLOADS["full_read_8x256x256_f32"]
    V, W, G = inputs.full_inputs(wl, dev())
    out = torch.empty(wl.T, wl.d, device=dev())
    ar.attnres_full_fwd(V, wl.n_src, W[0], G[0], wl.eps, out)
    torch.cuda.synchronize()
    ref, _ = oracle.full_read(V.cpu(), wl.n_src, W[0].cpu().double(), G[0].cpu().double(), wl.eps)
    assert rel_err(out, ref) <= TOL["f32"]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("n,T,d", [(1, 37, 128), (2, 8, 256), (5, 100, 384), (9, 1000, 896),
                                   (17, 257, 640), (3, 64, 1024), (4, 33, 2048),
                                   # many sources, one token
                                   (64, 9, 1024), (300, 5, 128), (6, 1, 896)])
def test_fast_read_vs_oracle(dt, n, T, d):
    out, ref = _read_case(n, T, d, dt)
    assert rel_err(out, ref) <= TOL[dt]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("n,T,d,offset", [(3, 5, 3, 0), (4, 9, 100, 0), (2, 3, 1, 0),
                                          (6, 50, 256, 1), (7, 11, 130, 3)])
def test_general_read_vs_oracle(dt, n, T, d, offset):
    path = ar.attnres_kernel_path(0, 1 << 20, 1 << 21, n, 0, T, d, 1 if dt == "bf16" else 0)
    if offset == 0 and d % 128 == 0:
        assert path == 1
    out, ref = _read_case(n, T, d, dt, offset=offset)
    assert rel_err(out, ref) <= TOL[dt]


def test_bf16_sources_fp32_output():
    """bf16 storage, fp32 output: only the fp32 arithmetic separates it from fp64."""
    out, ref = _read_case(8, 300, 512, "bf16", out_dt="f32")
    assert rel_err(out, ref) <= 1e-5


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_single_source_is_exact(dt):
    """n_src = 1 returns the source bit for bit."""
    g = inputs.generator(3, dev())
    V = inputs.history(1, 77, 384, dt, g, dev())
    w = inputs.queries(1, 384, 1.0, g, dev())[0]
    out = torch.empty(77, 384, device=dev(), dtype=dtype_of(dt))
    ar.attnres_full_fwd(V, 1, w, torch.ones(384, device=dev()), 1e-6, out)
    assert torch.equal(out, V[0])


def test_zero_query_is_mean():
    g = inputs.generator(4, dev())
    V = inputs.history(6, 50, 256, "f32", g, dev())
    out = torch.empty(50, 256, device=dev())
    ar.attnres_full_fwd(V, 6, torch.zeros(256, device=dev()), torch.ones(256, device=dev()), 1e-6, out)
    ref = V.double().mean(0).cpu().numpy()
    assert rel_err(out, ref) <= 1e-6


def test_permutation_invariance():
    g = inputs.generator(5, dev())
    V = inputs.history(7, 64, 512, "f32", g, dev())
    w = inputs.queries(1, 512, 0.1, g, dev())[0]
    gam = torch.ones(512, device=dev())
    a = torch.empty(64, 512, device=dev())
    b = torch.empty_like(a)
    ar.attnres_full_fwd(V, 7, w, gam, 1e-6, a)
    ar.attnres_full_fwd(V[torch.tensor([3, 0, 6, 1, 5, 2, 4])].contiguous(), 7, w, gam, 1e-6, b)
    assert rel_err(b, a.double().cpu().numpy()) <= 1e-5


def test_full_pass_small_vs_oracle():
    g = inputs.generator(6, dev())
    R, T, d = 12, 150, 256
    V = inputs.history(R, T, d, "bf16", g, dev())
    W = inputs.queries(R, d, 0.05, g, dev())
    G = torch.ones(R, d, device=dev())
    out = torch.empty(R, T, d, device=dev(), dtype=torch.bfloat16)
    ar.attnres_full_pass(V, W, G, 1e-6, out)
    torch.cuda.synchronize()
    ref = oracle.full_pass(V.cpu(), R, W.cpu().double(), G.cpu().double(), 1e-6)
    for r in range(R):
        assert rel_err(out[r], ref[r]) <= TOL["bf16"], f"read {r}"


def _sampled_pass_check(name, nrows):
    wl = inputs.WORKLOADS[name]
    V, W, G = inputs.full_inputs(wl, dev())
    out = torch.empty(wl.R, wl.T, wl.d, device=dev(), dtype=torch.bfloat16)
    ar.attnres_full_pass(V, W, G, wl.eps, out)
    torch.cuda.synchronize()
    assert ar.attnres_device_status() == 0
    rows = inputs.sample_rows(wl.T, nrows).to(dev())
    Vs = V[:, rows, :].cpu()
    got = out[:, rows, :].cpu()
    ref = oracle.full_pass(Vs, wl.R, W.cpu().double(), G.cpu().double(), wl.eps)
    worst = max(rel_err(got[r], ref[r]) for r in range(wl.R))
    assert worst <= TOL["bf16"], worst


def test_standard_pass_400m_full_size_sampled():
    """64 reads over the 8192 x 896 history, checked on sampled token rows."""
    _sampled_pass_check("full_pass_64x8192x896_bf16", 96)


def test_standard_pass_deep_narrow_full_size_sampled():
    """141 reads over the 32768 x 640 history (5.9 GB), checked on sampled rows."""
    _sampled_pass_check("full_pass_141x32768x640_bf16", 48)
