"""The no-allocation Block pass entry point matches the regular one (GPU).

attnres_block_pass_noalloc exists for callers that cannot allocate device
memory (a process that budgets all device memory up front, or a thread that
must not make calls that can synchronise the device, as cudaMalloc can). It
keeps its workspace in one array the library defines, shared by all calls.

Both entry points run the same kernels in the same order on 256-byte-aligned
workspace, so their results must agree bit for bit: these tests compare with
torch.equal, on two calls in a row with different inputs and shapes (the
second call also shows that what the first left in the shared array does not
leak into the next result), and cover one query per block (S = 1: no stage-1
workspace and no running sum), a frozen last summary, the largest accepted
size, the Python wrapper, and that a repeated call allocates no device memory.
One case is also held against the fp64 oracle. The file is named so that
pytest collects it last.
"""
import ctypes

import pytest
import torch

from depth_wise_attention_attnres_gb300 import binding as ar
from depth_wise_attention_attnres_gb300 import inputs
from tests._gpu import TOL, dev, rel_err

pytestmark = pytest.mark.gpu
LIMIT = 64 * 1024 * 1024  # ATTNRES_NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return ar.lib()


def _workspace_bytes(S, T, d, es):
    r = lambda x: (x + 255) // 256 * 256  # noqa: E731
    return (r((S - 1) * T * d * es) + r(4 * T * d) if S > 1 else 0) + r(4 * S * T)


def _inputs(N, S, T, d, dt, seed):
    g = inputs.generator(seed, dev())
    emb = inputs.randn((T, d), dt, g, dev())
    F = inputs.randn((N * S, T, d), dt, g, dev())
    W = inputs.queries(N * S, d, 0.05, g, dev())
    G = 1 + 0.2 * inputs.queries(N * S, d, 1.0, g, dev())
    return emb, F, W, G


def _buffers(emb, N, S, freeze_last):
    T, d = emb.shape
    Src = torch.empty(N + (1 if freeze_last else 0), T, d, device=dev(), dtype=emb.dtype)
    Src[0].copy_(emb)
    out = torch.full((N * S, T, d), float("nan"), device=dev(), dtype=emb.dtype)
    return Src, out


def _regular(emb, F, W, G, N, S, freeze_last=False):
    T, d = emb.shape
    Src, out = _buffers(emb, N, S, freeze_last)
    O = torch.empty(max(S - 1, 1), T, d, device=dev(), dtype=emb.dtype)
    lse = torch.empty(S, T, device=dev())
    P = torch.empty(T, d, device=dev())
    ar.attnres_block_pass(F, N, S, W, G, 1e-6, Src, O, lse, P, out, freeze_last=freeze_last)
    return out, Src


def _noalloc_c_abi(lib, emb, F, W, G, N, S, freeze_last=False):
    T, d = emb.shape
    Src, out = _buffers(emb, N, S, freeze_last)
    code = 1 if emb.dtype == torch.bfloat16 else 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.attnres_block_pass_noalloc(
        ctypes.c_void_p(F.data_ptr()), T * d, N, S, T, d, code, ctypes.c_void_p(W.data_ptr()),
        ctypes.c_void_p(G.data_ptr()), ctypes.c_float(1e-6), ctypes.c_void_p(Src.data_ptr()), T * d,
        int(freeze_last), ctypes.c_void_p(out.data_ptr()), T * d, stream)
    assert st == 0, ar.status_string(st)
    return out, Src


def _same(a, b):
    return torch.equal(a, b)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_noalloc_matches_regular_pass_two_calls(lib, dt):
    cases = [(3, 4, 700, 1024, 41), (4, 3, 257, 640, 42)]
    for N, S, T, d, seed in cases:
        emb, F, W, G = _inputs(N, S, T, d, dt, seed)
        ref_out, ref_src = _regular(emb, F, W, G, N, S)
        got_out, got_src = _noalloc_c_abi(lib, emb, F, W, G, N, S)
        torch.cuda.synchronize()
        assert ar.attnres_device_status() == 0
        assert _same(got_out, ref_out)
        assert _same(got_src, ref_src)


def test_noalloc_one_query_per_block_and_frozen_last(lib):
    # S = 1: no stage-1 workspace beyond lse and no running sum (O, P null).
    emb, F, W, G = _inputs(5, 1, 333, 512, "bf16", 43)
    ref_out, ref_src = _regular(emb, F, W, G, 5, 1, freeze_last=True)
    got_out, got_src = _noalloc_c_abi(lib, emb, F, W, G, 5, 1, freeze_last=True)
    torch.cuda.synchronize()
    assert _same(got_out, ref_out) and _same(got_src, ref_src)
    # freeze_last with several queries: the last block's summary is written too.
    emb, F, W, G = _inputs(2, 3, 129, 256, "f32", 44)
    ref_out, ref_src = _regular(emb, F, W, G, 2, 3, freeze_last=True)
    got_out, got_src = _noalloc_c_abi(lib, emb, F, W, G, 2, 3, freeze_last=True)
    torch.cuda.synchronize()
    assert _same(got_out, ref_out) and _same(got_src, ref_src)


def test_noalloc_matches_the_oracle(lib, oracle_mod):
    N, S, T, d = 3, 3, 96, 384
    emb, F, W, G = _inputs(N, S, T, d, "f32", 45)
    got_out, _ = _noalloc_c_abi(lib, emb, F, W, G, N, S)
    torch.cuda.synchronize()
    ref = oracle_mod.block_pass(emb.cpu(), F.cpu(), N, S, W.cpu().double(), G.cpu().double(), 1e-6)
    assert rel_err(got_out, ref) <= TOL["f32"]


def test_noalloc_at_the_size_limit_and_python_wrapper(lib):
    # bf16, d = 1024, S = 8: T = 3634 is the largest workspace that fits.
    N, S, d = 2, 8, 1024
    assert _workspace_bytes(S, 3634, d, 2) <= LIMIT < _workspace_bytes(S, 3635, d, 2)
    emb, F, W, G = _inputs(N, S, 3634, d, "bf16", 46)
    ref_out, ref_src = _regular(emb, F, W, G, N, S)
    Src, out = _buffers(emb, N, S, False)
    ar.attnres_block_pass_noalloc(F, N, S, W, G, 1e-6, Src, out)  # the Python wrapper
    torch.cuda.synchronize()
    assert _same(out, ref_out) and _same(Src, ref_src)
    # One token more is refused before anything runs.
    emb1, F1, W1, G1 = _inputs(N, S, 3635, d, "bf16", 47)
    Src1, out1 = _buffers(emb1, N, S, False)
    with pytest.raises(ar.AttnResError) as ei:
        ar.attnres_block_pass_noalloc(F1, N, S, W1, G1, 1e-6, Src1, out1)
    assert ei.value.status == 2  # ATTNRES_ERR_UNSUPPORTED
    assert torch.isnan(out1.float()).all()


def test_noalloc_repeated_call_allocates_nothing(lib):
    emb, F, W, G = _inputs(3, 4, 512, 1024, "bf16", 48)
    Src, out = _buffers(emb, 3, 4, False)
    ar.attnres_block_pass_noalloc(F, 3, 4, W, G, 1e-6, Src, out)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    ar.attnres_block_pass_noalloc(F, 3, 4, W, G, 1e-6, Src, out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_rejects_workspace_beyond_limit(lib):
    # bf16, d = 1024, S = 8 needs about 18 KiB per token: 8192 tokens exceed 64 MiB.
    N, S, T, d = 2, 8, 8192, 1024
    P = 1 << 20
    st = lib.attnres_block_pass_noalloc(P, T * d, N, S, T, d, 1, P, P, ctypes.c_float(1e-6),
                                        P, T * d, 0, P, T * d, None)
    assert st == 2  # ATTNRES_ERR_UNSUPPORTED, nothing launched
