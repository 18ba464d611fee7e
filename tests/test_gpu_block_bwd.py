"""Block pass backward: CUDA vs oracle (GPU).

The forward Block pass runs on the GPU first; its frozen summaries (Src) are
what the backward reads, and the oracle takes the same stored values, so the
comparison sees only the backward's own arithmetic: fp32 gradients from
exactly widened inputs, bar 1e-5 for both storage dtypes.
"""
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


def _forward(N, S, T, d, dt, seed):
    g = inputs.generator(seed, dev())
    emb = inputs.randn((T, d), dt, g, dev())
    F = inputs.randn((N * S, T, d), dt, g, dev())
    W = inputs.queries(N * S, d, 0.3, g, dev())
    G = 1 + 0.2 * inputs.queries(N * S, d, 1.0, g, dev())
    Src = torch.empty(N, T, d, device=dev(), dtype=dtype_of(dt))
    Src[0].copy_(emb)
    O = torch.empty(max(S - 1, 1), T, d, device=dev(), dtype=dtype_of(dt))
    lse = torch.empty(S, T, device=dev())
    P = torch.empty(T, d, device=dev())
    out = torch.empty(N * S, T, d, device=dev(), dtype=dtype_of(dt))
    ar.attnres_block_pass(F, N, S, W, G, 1e-6, Src, O, lse, P, out)
    dOut = inputs.randn((N * S, T, d), dt, g, dev())
    return Src, F, W, G, dOut


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("N,S,T,d", [(3, 4, 33, 256), (2, 3, 17, 100), (4, 1, 9, 128), (1, 5, 20, 384),
                                     (2, 2, 40, 1024), (1, 1, 1, 64), (2, 2, 1, 37), (9, 2, 5, 128),
                                     # batched: 8 blocks of 8 with fewer tokens than CTAs; one token
                                     (8, 8, 19, 256), (3, 3, 1, 128)])
def test_block_bwd_vs_oracle(dt, N, S, T, d):
    Src, F, W, G, dOut = _forward(N, S, T, d, dt, 70)
    dEmb = torch.zeros(T, d, device=dev())
    dF = torch.zeros(N * S, T, d, device=dev())
    dW = torch.zeros(N * S, d, device=dev())
    dG = torch.zeros(N * S, d, device=dev())
    ar.attnres_block_bwd(Src, F, N, S, W, G, 1e-6, dOut, dEmb, dF, dW, dG)
    torch.cuda.synchronize()
    assert ar.attnres_device_status() == 0
    rE, rF, rW, rG = oracle.block_pass_bwd(Src.cpu(), F.cpu(), N, S, W.cpu().double().numpy(),
                                           G.cpu().double().numpy(), 1e-6, dOut.cpu())
    assert rel_err(dEmb, rE) <= TOL["f32"], "dEmb"
    assert rel_err(dF, rF) <= TOL["f32"], "dF"
    assert rel_err(dW, rW) <= TOL["f32"], "dW"
    assert rel_err(dG, rG) <= TOL["f32"], "dGamma"


def test_block_bwd_accumulates():
    """Outputs are added to (a model sums the gradient over its uses); dW and
    dGamma may be omitted."""
    N, S, T, d = 2, 3, 24, 256
    Src, F, W, G, dOut = _forward(N, S, T, d, "bf16", 71)
    dEmb = torch.full((T, d), 0.5, device=dev())
    dF = torch.full((N * S, T, d), -0.25, device=dev())
    ar.attnres_block_bwd(Src, F, N, S, W, G, 1e-6, dOut, dEmb, dF)
    torch.cuda.synchronize()
    rE, rF, _, _ = oracle.block_pass_bwd(Src.cpu(), F.cpu(), N, S, W.cpu().double().numpy(),
                                         G.cpu().double().numpy(), 1e-6, dOut.cpu())
    assert rel_err(dEmb, rE + 0.5) <= TOL["f32"]
    assert rel_err(dF, rF - 0.25) <= TOL["f32"]


def test_block_bwd_fp32_gradient_input_with_bf16_storage():
    """dL/dout may be fp32 while the pass stores bf16."""
    N, S, T, d = 2, 3, 21, 256
    Src, F, W, G, _ = _forward(N, S, T, d, "bf16", 72)
    dOut = inputs.randn((N * S, T, d), "f32", inputs.generator(73, dev()), dev())
    dEmb = torch.zeros(T, d, device=dev())
    dF = torch.zeros(N * S, T, d, device=dev())
    ar.attnres_block_bwd(Src, F, N, S, W, G, 1e-6, dOut, dEmb, dF)
    torch.cuda.synchronize()
    rE, rF, _, _ = oracle.block_pass_bwd(Src.cpu(), F.cpu(), N, S, W.cpu().double().numpy(),
                                         G.cpu().double().numpy(), 1e-6, dOut.cpu().double().numpy())
    assert rel_err(dEmb, rE) <= TOL["f32"]
    assert rel_err(dF, rF) <= TOL["f32"]
