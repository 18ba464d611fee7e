"""The no-allocation Block pass entry point matches the regular one (GPU).

attnres_block_pass_noalloc exists for callers that cannot allocate device
memory (a process that budgets all device memory up front, or a thread that
must not make calls that can synchronise the device, as cudaMalloc can). It
keeps its workspace in one array the library defines, shared by all calls.
This test calls it through the C ABI twice in a row, with different inputs and
shapes, and compares each result with attnres_block_pass run on workspace
allocated here; the second call also shows that what the first call left in
the shared array does not leak into the next result. The file is named so
that pytest collects it last.
"""
import ctypes

import pytest
import torch

from depth_wise_attention_attnres_gb300 import binding as ar
from depth_wise_attention_attnres_gb300 import inputs
from tests._gpu import TOL, dev, dtype_of, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return ar.lib()


def _inputs(N, S, T, d, dt, seed):
    g = inputs.generator(seed, dev())
    emb = inputs.randn((T, d), dt, g, dev())
    F = inputs.randn((N * S, T, d), dt, g, dev())
    W = inputs.queries(N * S, d, 0.05, g, dev())
    G = 1 + 0.2 * inputs.queries(N * S, d, 1.0, g, dev())
    return emb, F, W, G


def _regular(emb, F, W, G, N, S):
    T, d = emb.shape
    Src = torch.empty(N, T, d, device=dev(), dtype=emb.dtype)
    Src[0].copy_(emb)
    O = torch.empty(max(S - 1, 1), T, d, device=dev(), dtype=emb.dtype)
    lse = torch.empty(S, T, device=dev())
    P = torch.empty(T, d, device=dev())
    out = torch.empty(N * S, T, d, device=dev(), dtype=emb.dtype)
    ar.attnres_block_pass(F, N, S, W, G, 1e-6, Src, O, lse, P, out)
    return out, Src


def _noalloc_c_abi(lib, emb, F, W, G, N, S):
    T, d = emb.shape
    Src = torch.empty(N, T, d, device=dev(), dtype=emb.dtype)
    Src[0].copy_(emb)
    out = torch.empty(N * S, T, d, device=dev(), dtype=emb.dtype)
    code = 1 if emb.dtype == torch.bfloat16 else 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.attnres_block_pass_noalloc(
        ctypes.c_void_p(F.data_ptr()), T * d, N, S, T, d, code, ctypes.c_void_p(W.data_ptr()),
        ctypes.c_void_p(G.data_ptr()), ctypes.c_float(1e-6), ctypes.c_void_p(Src.data_ptr()), T * d,
        0, ctypes.c_void_p(out.data_ptr()), T * d, stream)
    assert st == 0, ar.status_string(st)
    return out, Src


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_noalloc_matches_regular_pass_two_calls(lib, dt):
    cases = [(3, 4, 700, 1024, 41), (4, 3, 257, 640, 42)]
    for N, S, T, d, seed in cases:
        emb, F, W, G = _inputs(N, S, T, d, dt, seed)
        ref_out, ref_src = _regular(emb, F, W, G, N, S)
        got_out, got_src = _noalloc_c_abi(lib, emb, F, W, G, N, S)
        torch.cuda.synchronize()
        assert ar.attnres_device_status() == 0
        assert rel_err(got_out, ref_out.double().cpu().numpy()) <= TOL[dt]
        assert rel_err(got_src[1:], ref_src[1:].double().cpu().numpy()) <= TOL[dt]


def test_noalloc_rejects_workspace_beyond_limit(lib):
    # bf16, d = 1024, S = 8 needs about 18 KiB per token: 8192 tokens exceed 64 MiB.
    N, S, T, d = 2, 8, 8192, 1024
    P = 1 << 20
    st = lib.attnres_block_pass_noalloc(P, T * d, N, S, T, d, 1, P, P, ctypes.c_float(1e-6),
                                        P, T * d, 0, P, T * d, None)
    assert st == 2  # ATTNRES_ERR_UNSUPPORTED, nothing launched
