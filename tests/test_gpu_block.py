"""Block AttnRes stage 1, merge, accumulate and pass: CUDA vs oracle (GPU)."""
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
@pytest.mark.parametrize("n,S,T,d", [(1, 8, 100, 1024), (4, 8, 77, 1024), (8, 8, 130, 1024),
                                     (9, 3, 41, 512), (3, 6, 50, 2048), (8, 6, 19, 2048),
                                     (2, 1, 64, 256), (5, 5, 33, 896),
                                     # bf16 tensor-core outputs: two source blocks, ragged
                                     # tails, one 64-feature chunk, odd query counts
                                     (12, 8, 37, 1024), (6, 8, 45, 640), (7, 8, 23, 64),
                                     (16, 3, 29, 192)])
def test_stage1_vs_oracle(dt, n, S, T, d):
    g = inputs.generator(10, dev())
    Src = inputs.history(n, T, d, dt, g, dev(), depth_scaled=True)
    W = inputs.queries(S, d, 0.05, g, dev())
    G = 1 + 0.3 * inputs.queries(S, d, 1.0, g, dev())
    O = [torch.empty(T, d, device=dev(), dtype=dtype_of(dt)) for _ in range(S)]
    lse = torch.empty(S, T, device=dev())
    ar.attnres_block_stage1(Src, n, W, G, 1e-6, O, lse)
    torch.cuda.synchronize()
    refO, refL = oracle.block_stage1(Src.cpu(), n, W.cpu().double(), G.cpu().double(), 1e-6)
    for j in range(S):
        assert rel_err(O[j], refO[j]) <= TOL[dt], f"O[{j}]"
    # lse is a log-mass: compare absolutely (scores are O(1)).
    assert float(np.max(np.abs(lse.cpu().double().numpy() - refL))) <= 1e-4


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("n,S,T,d", [(4, 12, 40, 256), (3, 4, 21, 100), (2, 2, 5, 3)])
def test_stage1_general_kernel(dt, n, S, T, d):
    g = inputs.generator(11, dev())
    Src = inputs.history(n, T, d, dt, g, dev())
    W = inputs.queries(S, d, 0.05, g, dev())
    G = torch.ones(S, d, device=dev())
    O = [torch.empty(T, d, device=dev(), dtype=dtype_of(dt)) for _ in range(S)]
    lse = torch.empty(S, T, device=dev())
    ar.attnres_block_stage1(Src, n, W, G, 1e-6, O, lse)
    torch.cuda.synchronize()
    refO, refL = oracle.block_stage1(Src.cpu(), n, W.cpu().double(), G.cpu().double(), 1e-6)
    for j in range(S):
        assert rel_err(O[j], refO[j]) <= TOL[dt]
    assert float(np.max(np.abs(lse.cpu().double().numpy() - refL))) <= 1e-4


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("T,d", [(100, 1024), (33, 2048), (64, 896), (10, 100), (7, 3), (41, 1096)])
@pytest.mark.parametrize("mode", ["extend", "start", "as_is"])
def test_merge_vs_oracle(dt, T, d, mode):
    """Stage-1 result from the oracle, merged on the GPU with the running sum."""
    g = inputs.generator(12, dev())
    n = 3
    Src = inputs.history(n, T, d, dt, g, dev())
    w = inputs.queries(1, d, 0.05, g, dev())
    gam = 1 + 0.3 * inputs.queries(1, d, 1.0, g, dev())
    P0 = inputs.randn((T, d), "f32", g, dev(), scale=2.0)
    f = inputs.randn((T, d), dt, g, dev())
    refO, refL = oracle.block_stage1(Src.cpu(), n, w.cpu().double(), gam.cpu().double(), 1e-6)
    O = torch.tensor(refO[0], dtype=dtype_of(dt), device=dev())      # stage-1 values, rounded
    lse = torch.tensor(refL[0], dtype=torch.float32, device=dev())
    P = P0.clone()
    out = torch.empty(T, d, device=dev(), dtype=dtype_of(dt))
    f_prev = None if mode == "as_is" else f
    empty = mode == "start"
    ar.attnres_block_merge(O, lse, P, f_prev, empty, w[0], gam[0], 1e-6, out)
    torch.cuda.synchronize()
    # Reference: the read over {Src, P_new}, with the stage-1 output as stored.
    ref_out, ref_P = oracle.block_merge(Src.cpu(), n, P0.cpu(), None if f_prev is None else f.cpu(),
                                        empty, w[0].cpu().double(), gam[0].cpu().double(), 1e-6)
    assert rel_err(P, ref_P) <= 1e-6
    tol = TOL[dt] if dt == "bf16" else 2e-5  # O was rounded to fp32 before the merge
    assert rel_err(out, ref_out) <= tol


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("T,d", [(100, 1024), (9, 3), (64, 2048)])
def test_accumulate_and_freeze(dt, T, d):
    g = inputs.generator(13, dev())
    P0 = inputs.randn((T, d), "f32", g, dev())
    f = inputs.randn((T, d), dt, g, dev())
    P = P0.clone()
    ar.attnres_block_summary_accumulate(P, f, False)
    assert torch.equal(P, P0 + f.float())
    P = P0.clone()
    ar.attnres_block_summary_accumulate(P, f, True)
    assert torch.equal(P, f.float())
    summ = torch.empty(T, d, device=dev(), dtype=dtype_of(dt))
    P = P0.clone()
    ar.attnres_block_summary_accumulate(P, f, False, summ)
    assert torch.equal(P, P0)                              # freeze leaves P alone
    assert torch.equal(summ, (P0 + f.float()).to(dtype_of(dt)))   # RNE rounding of the fp32 sum


def _block_case(N, S, T, d, dt, seed=14, w_std=0.05):
    g = inputs.generator(seed, dev())
    emb = inputs.randn((T, d), dt, g, dev())
    F = inputs.randn((N * S, T, d), dt, g, dev())
    W = inputs.queries(N * S, d, w_std, g, dev())
    G = torch.ones(N * S, d, device=dev())
    return emb, F, W, G


def _run_block(emb, F, W, G, N, S, eps=1e-6):
    T, d = emb.shape
    dt = emb.dtype
    Src = torch.empty(N, T, d, device=dev(), dtype=dt)
    Src[0].copy_(emb)
    O = torch.empty(max(S - 1, 1), T, d, device=dev(), dtype=dt)
    lse = torch.empty(S, T, device=dev())
    P = torch.empty(T, d, device=dev())
    out = torch.empty(N * S, T, d, device=dev(), dtype=dt)
    ar.attnres_block_pass(F, N, S, W, G, eps, Src, O, lse, P, out)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("N,S,T,d", [(4, 4, 70, 1024), (3, 6, 40, 2048), (2, 3, 30, 640),
                                     (1, 5, 17, 256), (5, 1, 23, 512), (3, 2, 9, 100)])
def test_block_pass_vs_oracle(dt, N, S, T, d):
    emb, F, W, G = _block_case(N, S, T, d, dt)
    out = _run_block(emb, F, W, G, N, S)
    ref = oracle.block_pass(emb.cpu(), F.cpu(), N, S, W.cpu().double(), G.cpu().double(), 1e-6)
    for k in range(N * S):
        assert rel_err(out[k], ref[k]) <= TOL[dt], f"sublayer {k}"


def test_block_s1_equals_full_on_gpu():
    """Block AttnRes with one sublayer per block is Full AttnRes."""
    N, T, d = 6, 50, 512
    emb, F, W, G = _block_case(N, 1, T, d, "f32", w_std=0.2)
    blk = _run_block(emb, F, W, G, N, 1)
    hist = torch.cat([emb[None], F[:-1]]).contiguous()
    full = torch.empty(N, T, d, device=dev())
    ar.attnres_full_pass(hist, W, G, 1e-6, full)
    torch.cuda.synchronize()
    assert rel_err(blk, full.double().cpu().numpy()) <= 1e-5


def _sampled_block_check(name, nrows):
    wl = inputs.WORKLOADS[name]
    emb, F, W, G = inputs.block_inputs(wl, dev())
    out = _run_block(emb, F, W, G, wl.N, wl.S, wl.eps)
    assert ar.attnres_device_status() == 0
    rows = inputs.sample_rows(wl.T, nrows).to(dev())
    ref = oracle.block_pass(emb[rows].cpu(), F[:, rows, :].cpu(), wl.N, wl.S, W.cpu().double(),
                            G.cpu().double(), wl.eps)
    got = out[:, rows, :].cpu()
    worst = max(rel_err(got[k], ref[k]) for k in range(wl.N * wl.S))
    assert worst <= TOL["bf16"], worst


def test_standard_block_pass_full_size_sampled():
    """8 blocks of 8 sublayers at 16384 x 1024, checked on sampled token rows."""
    _sampled_block_check("block_pass_8x8x16384x1024_bf16", 96)


def test_standard_block_prefill_128k_full_size_sampled():
    """8 blocks of 6 sublayers at 131072 x 2048 (about 60 GB resident)."""
    _sampled_block_check("block_pass_8x6x131072x2048_bf16", 48)
