"""Input-dependent query: projection and per-token-query read, CUDA vs oracle (GPU).

The pages' ablation (LLMRes blog, on the paper's ablation): the query is
projected from the current hidden state by a per-layer d x d matrix; the
read then scores each token with its own query.
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


def _wq(d, g):
    return (inputs.randn((d, d), "f32", g, dev()) / d ** 0.5).to(torch.bfloat16).contiguous()


# Single CTAs take 128-wide tiles, or the widest of 256, 224, 192, 160
# dividing d; products with d a multiple of 256 that give every CTA pair a
# 256 x 256 tile run on CTA pairs. The ragged pair cases end in a 256-row tile
# whose second CTA has some rows (8392) or none (8292, 4103) inside the product.
@pytest.mark.parametrize("T,d", [(300, 128), (1000, 896), (129, 256), (50, 100), (7, 1024), (200, 640), (77, 384),
                                 (130, 2048), (4096, 2048), (16384, 896), (32768, 384), (16383, 640), (8192, 896),
                                 (16384, 1024), (8192, 2048), (8292, 1024), (8392, 1024), (4103, 2048), (8200, 1280)])
def test_query_projection(T, d):
    g = inputs.generator(40, dev())
    H = inputs.randn((T, d), "bf16", g, dev())
    Wq = _wq(d, g)
    Q = torch.full((T, d), float("nan"), device=dev())
    ar.attnres_query_projection(H, Wq, Q)
    torch.cuda.synchronize()
    ref = oracle.query_projection(H.cpu(), Wq.cpu())
    assert rel_err(Q, ref) <= TOL["f32"]


@pytest.mark.parametrize("T,d,path", [(16384, 1024, 2), (8192, 2048, 2), (8292, 1024, 2), (8392, 1024, 2),
                                      (4103, 2048, 2), (8192, 896, 1), (1000, 896, 1), (300, 128, 1), (130, 2048, 1),
                                      (50, 100, 0)])
def test_query_projection_kernel_choice(T, d, path):
    """Which of the projection's kernels the shapes above reach (so that both
    tensor-core kernels are covered)."""
    H = torch.empty(T, d, device=dev(), dtype=torch.bfloat16)
    Q = torch.empty(T, d, device=dev())
    assert ar.attnres_kernel_path(4, H.data_ptr(), Q.data_ptr(), 0, 0, T, d, ar.BF16) == path


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("n,T,d", [(5, 70, 896), (8, 33, 640), (3, 33, 100), (1, 16, 256), (12, 9, 1024)])
def test_full_fwd_dynq(dt, n, T, d):
    g = inputs.generator(41, dev())
    V = inputs.history(n, T, d, dt, g, dev(), depth_scaled=True)
    Q = inputs.randn((T, d), "f32", g, dev(), scale=0.05)
    gam = (1 + 0.3 * inputs.queries(1, d, 1.0, g, dev())[0]).contiguous()
    out = torch.empty(T, d, device=dev(), dtype=dtype_of(dt))
    ar.attnres_full_fwd_dynq(V, n, Q, gam, 1e-6, out)
    torch.cuda.synchronize()
    Vc = V.cpu()
    ref, _ = oracle.read_dynamic_query([Vc[i] for i in range(n)], Q.cpu().double().numpy(),
                                       gam.cpu().double().numpy(), 1e-6)
    assert rel_err(out, ref) <= TOL[dt]


def test_projected_query_read():
    """Read r's query projected from its newest source, then the read."""
    n, T, d = 6, 200, 896
    g = inputs.generator(42, dev())
    V = inputs.history(n, T, d, "bf16", g, dev(), depth_scaled=True)
    Wq = _wq(d, g)
    gam = torch.ones(d, device=dev())
    Q = torch.empty(T, d, device=dev())
    out = torch.empty(T, d, device=dev(), dtype=torch.bfloat16)
    ar.attnres_query_projection(V[n - 1], Wq, Q)
    ar.attnres_full_fwd_dynq(V, n, Q, gam, 1e-6, out)
    torch.cuda.synchronize()
    Vc = V.cpu()
    q = oracle.query_projection(Vc[n - 1], Wq.cpu())
    ref, _ = oracle.read_dynamic_query([Vc[i] for i in range(n)], q, np.ones(d), 1e-6)
    assert rel_err(out, ref) <= TOL["bf16"]
