"""Failure paths on the GPU, driven by the library's test hooks (no fault).

* A simulated launch failure (attnres_test_fail_launch) inside a Full pass and
  a Block pass: the call returns ATTNRES_ERR_CUDA at the failed launch, the
  reads before it are correct, nothing after it was written, and the next
  call runs normally.
* A producer that withholds one stage (attnres_test_withhold_stage) in each
  pipelined kernel (the Full-read bulk kernel, the tensor-core stage 1, the
  tiled merge): the consumers' bounded wait runs out, the kernel drains the
  copies it issued and returns, attnres_device_status reports
  ATTNRES_ERR_TIMEOUT once, and a following call on the same context is
  correct. Every wait is bounded (about 2 s), so nothing here can hang.
"""
import pytest
import torch

from depth_wise_attention_attnres_gb300 import binding as ar
from depth_wise_attention_attnres_gb300 import inputs
from tests._gpu import TOL, dev, rel_err

pytestmark = pytest.mark.gpu
CUDA_ERR, TIMEOUT = 3, 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    ar.attnres_test_fail_launch(-1)
    ar.attnres_test_withhold_stage(ar.WITHHOLD_NONE)


@pytest.fixture(autouse=True)
def _hooks_off():
    assert ar.attnres_device_status() == 0
    yield
    ar.attnres_test_fail_launch(-1)
    ar.attnres_test_withhold_stage(ar.WITHHOLD_NONE)


def test_injected_failure_stops_a_full_pass(oracle_mod):
    R, T, d = 6, 300, 256
    g = inputs.generator(60, dev())
    V = inputs.history(R, T, d, "bf16", g, dev())
    W = inputs.queries(R, d, 0.05, g, dev())
    G = torch.ones(R, d, device=dev())
    out = torch.full((R, T, d), float("nan"), device=dev(), dtype=torch.bfloat16)
    ar.attnres_test_fail_launch(3)            # reads 0, 1, 2 launch; read 3 fails
    with pytest.raises(ar.AttnResError) as ei:
        ar.attnres_full_pass(V, W, G, 1e-6, out)
    assert ei.value.status == CUDA_ERR
    assert ar.attnres_test_fail_launch(-1) == -1   # the failure fired
    assert ar.attnres_device_status() == 0         # nothing ran that failed on the device
    Vc, Wc, Gc = V.cpu(), W.cpu().double(), G.cpu().double()
    for r in range(3):
        ref, _ = oracle_mod.full_read(Vc, r + 1, Wc[r], Gc[r], 1e-6)
        assert rel_err(out[r], ref) <= TOL["bf16"]
    assert torch.isnan(out[3:].float()).all()      # nothing after the failed launch
    ar.attnres_full_pass(V, W, G, 1e-6, out)       # the context is fine
    torch.cuda.synchronize()
    for r in range(R):
        ref, _ = oracle_mod.full_read(Vc, r + 1, Wc[r], Gc[r], 1e-6)
        assert rel_err(out[r], ref) <= TOL["bf16"]


def test_injected_failure_stops_a_block_pass(oracle_mod):
    N, S, T, d = 3, 3, 200, 512
    g = inputs.generator(61, dev())
    emb = inputs.randn((T, d), "bf16", g, dev())
    F = inputs.randn((N * S, T, d), "bf16", g, dev())
    W = inputs.queries(N * S, d, 0.05, g, dev())
    G = torch.ones(N * S, d, device=dev())
    Src = torch.empty(N, T, d, device=dev(), dtype=torch.bfloat16)
    Src[0].copy_(emb)
    O = torch.empty(S - 1, T, d, device=dev(), dtype=torch.bfloat16)
    lse = torch.empty(S, T, device=dev())
    P = torch.empty(T, d, device=dev())
    out = torch.full((N * S, T, d), float("nan"), device=dev(), dtype=torch.bfloat16)
    # Block 0 makes 4 launches (stage 1, 2 merges, freeze); block 1's stage 1 fails.
    ar.attnres_test_fail_launch(4)
    with pytest.raises(ar.AttnResError) as ei:
        ar.attnres_block_pass(F, N, S, W, G, 1e-6, Src, O, lse, P, out)
    assert ei.value.status == CUDA_ERR
    assert ar.attnres_device_status() == 0
    ref = oracle_mod.block_pass(emb.cpu(), F.cpu(), N, S, W.cpu().double(), G.cpu().double(), 1e-6)
    assert rel_err(out[:S], ref[:S]) <= TOL["bf16"]
    assert torch.isnan(out[S:].float()).all()
    ar.attnres_block_pass(F, N, S, W, G, 1e-6, Src, O, lse, P, out)
    torch.cuda.synchronize()
    assert rel_err(out, ref) <= TOL["bf16"]


def _full_case(oracle_mod):
    # 4 sources, d = 256: every CTA of the bulk kernel has more than 8 copies.
    n, T, d = 4, 16384, 256
    g = inputs.generator(62, dev())
    V = inputs.history(n, T, d, "bf16", g, dev())
    w = inputs.queries(1, d, 0.05, g, dev())[0]
    gamma = torch.ones(d, device=dev())
    out = torch.empty(T, d, device=dev(), dtype=torch.bfloat16)

    def run():
        ar.attnres_full_fwd(V, n, w, gamma, 1e-6, out)

    def check():
        rows = inputs.sample_rows(T, 64).to(dev())
        ref, _ = oracle_mod.full_read(V[:, rows].cpu(), n, w.cpu().double(), gamma.cpu().double(), 1e-6)
        return rel_err(out[rows], ref)
    return run, check, [out]


def _stage1_case(oracle_mod):
    n, S, T, d = 4, 4, 16384, 1024
    g = inputs.generator(63, dev())
    Src = inputs.history(n, T, d, "bf16", g, dev(), depth_scaled=False)
    W = inputs.queries(S, d, 0.05, g, dev())
    G = torch.ones(S, d, device=dev())
    O = [torch.empty(T, d, device=dev(), dtype=torch.bfloat16) for _ in range(S)]
    lse = torch.empty(S, T, device=dev())
    assert ar.attnres_kernel_path(1, Src.data_ptr(), O[0].data_ptr(), n, S, T, d, ar.BF16) == 1

    def run():
        ar.attnres_block_stage1(Src, n, W, G, 1e-6, O, lse)

    def check():
        rows = inputs.sample_rows(T, 64).to(dev())
        refO, _ = oracle_mod.block_stage1(Src[:, rows].cpu(), n, W.cpu().double(), G.cpu().double(), 1e-6)
        return max(rel_err(O[j][rows], refO[j]) for j in range(S))
    return run, check, O + [lse]


def _merge_case(oracle_mod):
    # Stage 1 of one query over 2 sources, then its merge with a running sum.
    n, T, d = 2, 16384, 1024
    g = inputs.generator(64, dev())
    Src = inputs.history(n, T, d, "bf16", g, dev(), depth_scaled=False)
    w = inputs.queries(1, d, 0.05, g, dev())
    gamma = torch.ones(1, d, device=dev())
    Oj = torch.empty(T, d, device=dev(), dtype=torch.bfloat16)
    lse = torch.empty(1, T, device=dev())
    ar.attnres_block_stage1(Src, n, w, gamma, 1e-6, [Oj], lse)
    P0 = inputs.randn((T, d), "f32", g, dev())
    P = P0.clone()
    f = inputs.randn((T, d), "bf16", g, dev())
    out = torch.empty(T, d, device=dev(), dtype=torch.bfloat16)

    def run():
        P.copy_(P0)
        ar.attnres_block_merge(Oj, lse[0], P, f, False, w[0], gamma[0], 1e-6, out)

    def check():
        rows = inputs.sample_rows(T, 64).to(dev())
        ref, _ = oracle_mod.block_merge(Src[:, rows].cpu(), n, P0[rows].cpu(), f[rows].cpu(), False,
                                        w[0].cpu().double(), gamma[0].cpu().double(), 1e-6)
        return rel_err(out[rows], ref)
    return run, check, [out, P]


@pytest.mark.parametrize("kernel,make,index", [
    (ar.WITHHOLD_FULL, _full_case, 5),
    (ar.WITHHOLD_STAGE1_TC, _stage1_case, 3),
    (ar.WITHHOLD_MERGE, _merge_case, 4),
])
def test_withheld_stage_times_out_and_recovers(oracle_mod, kernel, make, index):
    run, check, outputs = make(oracle_mod)
    run()
    torch.cuda.synchronize()
    assert check() <= TOL["bf16"]
    good = [t.clone() for t in outputs]
    ar.attnres_test_withhold_stage(kernel, index)
    run()
    assert ar.attnres_device_status() == TIMEOUT   # the bounded wait ran out
    assert ar.attnres_device_status() == 0         # reported once
    ar.attnres_test_withhold_stage(ar.WITHHOLD_NONE)
    for t in outputs:
        t.fill_(float("nan"))
    run()
    assert ar.attnres_device_status() == 0
    # The same context computes the same bits as before the timeout.
    assert all(torch.equal(t, u) for t, u in zip(outputs, good))
