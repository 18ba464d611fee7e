"""Stage 1 with the features split into shards: CUDA vs oracle (GPU).

The shards of one GPU add their parts of the score sums into one buffer (the
exchange step a tensor-parallel layout does with an all-reduce); each shard
then finishes its features of the outputs. Joined, they must equal stage 1 by
definition (the oracle's per-query reads over the full width).
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


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("n,S,T,d,P", [(8, 8, 70, 1024, 4), (3, 6, 33, 2048, 4), (5, 3, 41, 512, 2),
                                       (1, 1, 16, 256, 2), (12, 16, 9, 384, 3),
                                       (4, 5, 37, 360, 3), (20, 4, 23, 512, 2), (8, 8, 1, 512, 2),
                                       (16, 2, 5, 256, 2), (2, 16, 3, 128, 1)])
def test_dsplit_stage1(dt, n, S, T, d, P):
    g = inputs.generator(50, dev())
    Src = inputs.history(n, T, d, dt, g, dev(), depth_scaled=True)
    W = inputs.queries(S, d, 0.05, g, dev())
    G = 1 + 0.3 * inputs.queries(S, d, 1.0, g, dev())
    ds = d // P
    part = torch.empty(T, n, S + 1, device=dev())
    shards = [Src[:, :, s * ds:(s + 1) * ds].contiguous() for s in range(P)]
    for s in range(P):
        ar.attnres_stage1_dsplit_partials(shards[s], n, W[:, s * ds:(s + 1) * ds].contiguous(),
                                          G[:, s * ds:(s + 1) * ds].contiguous(), part, s > 0)
    outs = [[torch.empty(T, ds, device=dev(), dtype=dtype_of(dt)) for _ in range(S)] for _ in range(P)]
    lse = torch.empty(S, T, device=dev())
    for s in range(P):
        ar.attnres_stage1_dsplit_finish(shards[s], n, d, part, 1e-6, outs[s], lse if s == 0 else None)
    torch.cuda.synchronize()
    refO, refL = oracle.block_stage1(Src.cpu(), n, W.cpu().double(), G.cpu().double(), 1e-6)
    for j in range(S):
        got = torch.cat([outs[s][j] for s in range(P)], dim=1)
        assert rel_err(got, refO[j]) <= TOL[dt], f"O[{j}]"
    assert float(np.max(np.abs(lse.cpu().double().numpy() - refL))) <= 1e-4
    # The summed partials are the full-width sums.
    V = Src.cpu().double().numpy()
    u = (W.cpu().double() * G.cpu().double()).numpy()
    ss = np.sum(V * V, axis=-1)
    assert rel_err(part[:, :, 0], ss.T) <= 1e-5
    assert rel_err(part[:, :, 1:], np.einsum("itk,jk->tij", V, u)) <= 1e-5
