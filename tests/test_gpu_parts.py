"""Merges and freezes with the running sum given in parts (GPU).

A block's running sum P_j = f_0 + ... + f_{j-1} (LLMRes blog "Block Attention
Residuals"; DepthBench reading notes section 2.5) can be kept in an fp32
buffer step by step, or formed again from a kept P_m plus the outputs since.
Both add the same fp32 values in the same order, so the running sums (and
the frozen summaries rounded from them) must agree bit for bit. The merged
outputs may differ in their last bit: the tiled merge sizes its tiles by the
bytes a row brings in, and the rows of a tile split the score's two sums
over fewer or more warps, which changes the order of fp32 additions in those
sums (not in the running sum). They are held to 1e-6 relative (fp32) and one
bf16 ulp (bf16). These tests hold attnres_block_merge_parts and
attnres_block_summary_parts to the one-step calls (attnres_block_merge,
attnres_block_summary_accumulate) on the fast and the general kernels, and
hold the Block pass, which mixes the two by its running-sum plan, to the pass
written out with the one-step calls. One case also meets the fp64 oracle.
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


# Reduction-order differences in the score, relative to the largest output.
ORDER_TOL = {"f32": 1e-6, "bf16": 2.0 ** -8}


def _one_step_sums(F, j):
    """P_1 .. P_j by the one-step calls: P_1 = f_0, P_i = P_{i-1} + f_{i-1}."""
    T, d = F.shape[1:]
    sums = []
    P = torch.empty(T, d, device=dev())
    for i in range(j):
        ar.attnres_block_summary_accumulate(P, F[i], i == 0)
        sums.append(P.clone())
    return sums


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("T,d", [(300, 1024), (77, 2048), (45, 640), (13, 100), (9, 3)])
def test_merge_parts_equals_one_step_merges(dt, T, d):
    g = inputs.generator(80, dev())
    J = 6
    F = inputs.randn((J, T, d), dt, g, dev())
    O = inputs.randn((T, d), dt, g, dev())
    lse = torch.randn(T, device=dev())
    w = inputs.queries(1, d, 0.05, g, dev())[0]
    gam = 1 + 0.3 * inputs.queries(1, d, 1.0, g, dev())[0]
    sums = _one_step_sums(F, J)
    for j in range(1, J + 1):
        ref = torch.empty(T, d, device=dev(), dtype=dtype_of(dt))
        ar.attnres_block_merge(O, lse, sums[j - 1].clone(), None, False, w, gam, 1e-6, ref)
        for m in range(0, j + 1):
            base = sums[m - 1] if m > 0 else None
            if base is None and m == j:
                continue          # no base and no part: no source
            out = torch.full((T, d), float("nan"), device=dev(), dtype=dtype_of(dt))
            P_out = torch.full((T, d), float("nan"), device=dev())
            ar.attnres_block_merge_parts(O, lse, base, F[m:], j - m, P_out, w, gam, 1e-6, out)
            torch.cuda.synchronize()
            assert torch.equal(P_out, sums[j - 1]), (j, m)
            assert rel_err(out, ref.double().cpu().numpy()) <= ORDER_TOL[dt], (j, m)
        # In place: P_out is the base buffer itself.
        if j >= 2:
            P = sums[0].clone()
            out = torch.empty(T, d, device=dev(), dtype=dtype_of(dt))
            ar.attnres_block_merge_parts(O, lse, P, F[1:], j - 1, P, w, gam, 1e-6, out)
            torch.cuda.synchronize()
            assert torch.equal(P, sums[j - 1])
            assert rel_err(out, ref.double().cpu().numpy()) <= ORDER_TOL[dt]


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("T,d", [(300, 1024), (64, 2048), (9, 3)])
def test_summary_parts_equals_one_step_freeze(dt, T, d):
    g = inputs.generator(81, dev())
    S = 6
    F = inputs.randn((S, T, d), dt, g, dev())
    sums = _one_step_sums(F, S)
    ref = torch.empty(T, d, device=dev(), dtype=dtype_of(dt))
    ar.attnres_block_summary_accumulate(sums[S - 2].clone(), F[S - 1], False, ref)
    for m in range(0, S):
        base = sums[m - 1] if m > 0 else None
        got = torch.empty(T, d, device=dev(), dtype=dtype_of(dt))
        ar.attnres_block_summary_parts(base, F[m:], S - m, summary_out=got)
        P_out = torch.empty(T, d, device=dev())
        ar.attnres_block_summary_parts(base, F[m:], S - m, P_out=P_out)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), m
        assert torch.equal(P_out, sums[S - 1]), m


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("T,d", [(300, 1024), (77, 2048), (45, 640), (13, 100), (9, 3)])
def test_merge_parts_with_summary(dt, T, d):
    """The block's last merge freezing its summary: summary_out must hold the
    freeze's bits (attnres_block_summary_parts over one part more), P_out the
    running sum's, and out the merge (to the reduction-order tolerance: the
    extra part changes the tile shape)."""
    g = inputs.generator(84, dev())
    J = 6
    F = inputs.randn((J, T, d), dt, g, dev())
    O = inputs.randn((T, d), dt, g, dev())
    lse = torch.randn(T, device=dev())
    w = inputs.queries(1, d, 0.05, g, dev())[0]
    gam = 1 + 0.3 * inputs.queries(1, d, 1.0, g, dev())[0]
    sums = _one_step_sums(F, J)
    for j in range(1, J):
        for m in range(0, j + 1):
            base = sums[m - 1] if m > 0 else None
            if base is None and m == j:
                continue
            ref_out = torch.empty(T, d, device=dev(), dtype=dtype_of(dt))
            ar.attnres_block_merge_parts(O, lse, base, F[m:], j - m, None, w, gam, 1e-6, ref_out)
            ref_sum = torch.empty(T, d, device=dev(), dtype=dtype_of(dt))
            ar.attnres_block_summary_parts(base, F[m:], j + 1 - m, summary_out=ref_sum)
            out = torch.full((T, d), float("nan"), device=dev(), dtype=dtype_of(dt))
            summ = torch.full((T, d), float("nan"), device=dev(), dtype=dtype_of(dt))
            P_out = torch.full((T, d), float("nan"), device=dev())
            ar.attnres_block_merge_parts(O, lse, base, F[m:], j - m, P_out, w, gam, 1e-6, out, summary_out=summ)
            torch.cuda.synchronize()
            assert torch.equal(summ, ref_sum), (j, m)
            assert torch.equal(P_out, sums[j - 1]), (j, m)
            assert rel_err(out, ref_out.double().cpu().numpy()) <= ORDER_TOL[dt], (j, m)


def _pass_by_one_step_calls(F, emb, N, S, W, G):
    """The Block pass written out with the one-step merge and freeze calls
    (the running sum kept in P at every step)."""
    T, d = emb.shape
    Src = torch.empty(N, T, d, device=dev(), dtype=emb.dtype)
    Src[0].copy_(emb)
    O = torch.empty(max(S - 1, 1), T, d, device=dev(), dtype=emb.dtype)
    lse = torch.empty(S, T, device=dev())
    P = torch.empty(T, d, device=dev())
    out = torch.empty(N * S, T, d, device=dev(), dtype=emb.dtype)
    for n in range(N):
        k0 = n * S
        ar.attnres_block_stage1(Src, n + 1, W[k0:k0 + S], G[k0:k0 + S], 1e-6,
                                [out[k0]] + [O[j - 1] for j in range(1, S)], lse)
        for j in range(1, S):
            ar.attnres_block_merge(O[j - 1], lse[j], P, F[k0 + j - 1], j == 1, W[k0 + j], G[k0 + j], 1e-6,
                                   out[k0 + j])
        if n + 1 < N:
            ar.attnres_block_summary_accumulate(P, F[k0 + S - 1], S == 1, Src[n + 1])
    return out, Src


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("N,S,T,d", [(3, 6, 200, 2048), (3, 8, 130, 1024), (4, 3, 77, 640), (2, 16, 33, 256),
                                     (3, 5, 21, 100)])
def test_block_pass_plan_changes_no_running_sum(dt, N, S, T, d):
    g = inputs.generator(82, dev())
    emb = inputs.randn((T, d), dt, g, dev())
    F = inputs.randn((N * S, T, d), dt, g, dev())
    W = inputs.queries(N * S, d, 0.05, g, dev())
    G = 1 + 0.2 * inputs.queries(N * S, d, 1.0, g, dev())
    plan = ar.attnres_block_running_sum_plan(S, ar.BF16 if dt == "bf16" else ar.F32)
    ref_out, ref_src = _pass_by_one_step_calls(F, emb, N, S, W, G)
    Src = torch.empty(N, T, d, device=dev(), dtype=emb.dtype)
    Src[0].copy_(emb)
    O = torch.empty(max(S - 1, 1), T, d, device=dev(), dtype=emb.dtype)
    lse = torch.empty(S, T, device=dev())
    P = torch.empty(T, d, device=dev())
    out = torch.empty(N * S, T, d, device=dev(), dtype=emb.dtype)
    ar.attnres_block_pass(F, N, S, W, G, 1e-6, Src, O, lse, P, out)
    torch.cuda.synchronize()
    assert torch.equal(Src, ref_src), plan          # the frozen summaries: bit for bit
    for k in range(N * S):
        assert rel_err(out[k], ref_out[k].double().cpu().numpy()) <= ORDER_TOL[dt], (plan, k)


def test_merge_parts_meets_the_oracle():
    T, d, n = 150, 1024, 3
    g = inputs.generator(83, dev())
    Src = inputs.history(n, T, d, "f32", g, dev(), depth_scaled=False)
    F = inputs.randn((4, T, d), "f32", g, dev())
    w = inputs.queries(1, d, 0.05, g, dev())
    gam = torch.ones(1, d, device=dev())
    Oj = torch.empty(T, d, device=dev())
    lse = torch.empty(1, T, device=dev())
    ar.attnres_block_stage1(Src, n, w, gam, 1e-6, [Oj], lse)
    out = torch.empty(T, d, device=dev())
    ar.attnres_block_merge_parts(Oj, lse[0], None, F, 4, None, w[0], gam[0], 1e-6, out)
    torch.cuda.synchronize()
    P_exact = oracle.widen(F.cpu()).sum(0)
    ref, _ = oracle.read([Src[i].cpu() for i in range(n)] + [P_exact], w[0].cpu().double(),
                         gam[0].cpu().double(), 1e-6)
    assert rel_err(out, ref) <= TOL["f32"]
