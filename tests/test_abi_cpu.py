"""The C ABI library builds, loads and exports every declared symbol (no GPU).

Only host-side logic runs here: argument validation returns its status codes
before any CUDA call, and kernel selection is a pure function of the
arguments.
"""
import ctypes

import pytest

from depth_wise_attention_attnres_gb300 import binding, build

INVALID, UNSUPPORTED = 1, 2


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def test_every_declared_symbol_is_exported(lib):
    names = binding.header_functions()
    assert len(names) >= 10
    handle = ctypes.CDLL(build.LIB)
    missing = [n for n in names if not hasattr(handle, n)]
    assert not missing, f"not exported: {missing}"
    assert set(names) == set(binding._SIGNATURES)


def test_version_and_status_strings(lib):
    assert binding.attnres_abi_version() == 1
    for code in range(5):
        assert binding.status_string(code)
    assert binding.status_string(99) == "unknown status"


P = 1 << 20  # aligned stand-in pointers: validation never dereferences them


@pytest.mark.parametrize("args,expect", [
    # (V, stride, n_src, T, d, dtype, w, gamma, eps, out, out_dtype)
    ((P, 64, 0, 4, 16, 1, P, P, 1e-6, 8 * P, 1), INVALID),          # n_src = 0
    ((P, 64, 2, 4, 16, 1, P, P, -1.0, 8 * P, 1), INVALID),          # eps < 0
    ((P, 64, 2, 4, 16, 7, P, P, 1e-6, 8 * P, 1), INVALID),          # bad dtype
    ((P, 63, 2, 4, 16, 1, P, P, 1e-6, 8 * P, 1), INVALID),          # stride < T*d
    ((P, 64, 2, 4, 16, 1, P, P, 1e-6, P + 64, 1), INVALID),         # out overlaps V
    ((None, 64, 2, 4, 16, 1, P, P, 1e-6, 8 * P, 1), INVALID),       # null V
    ((None, 0, 3, 0, 16, 1, None, None, 1e-6, None, 1), 0),         # T = 0: nothing to do
])
def test_full_fwd_validation(lib, args, expect):
    assert lib.attnres_full_fwd(*args, None) == expect


def test_other_entry_validation(lib):
    ptrs = (ctypes.c_void_p * 2)(P * 8, P * 16)
    # stage 1: S out of range, overlapping outputs
    assert lib.attnres_block_stage1(P, 64, 2, 4, 16, 1, P, P, 0, 1e-6, ptrs, None, None) == INVALID
    assert lib.attnres_block_stage1(P, 64, 2, 4, 16, 1, P, P, 17, 1e-6, ptrs, None, None) == INVALID
    same = (ctypes.c_void_p * 2)(P * 8, P * 8)
    assert lib.attnres_block_stage1(P, 64, 2, 4, 16, 1, P, P, 2, 1e-6, same, None, None) == INVALID
    # merge: empty running sum needs f_prev; out must not alias P
    assert lib.attnres_block_merge(P, 2 * P, 3 * P, None, 1, P, P, 1e-6, 4, 16, 1, 5 * P, None) == INVALID
    assert lib.attnres_block_merge(P, 2 * P, 3 * P, None, 0, P, P, 1e-6, 4, 16, 1, 3 * P, None) == INVALID
    # accumulate: summary aliasing f
    assert lib.attnres_block_summary_accumulate(P, 2 * P, 0, 2 * P, 4, 16, 1, None) == INVALID
    # passes
    assert lib.attnres_full_pass(P, 64, 0, 4, 16, 1, P, P, 1e-6, 8 * P, 64, 1, None) == INVALID
    assert lib.attnres_block_pass(P, 64, 0, 2, 4, 16, 1, P, P, 1e-6, 2 * P, 64, 0, 3 * P, 4 * P,
                                  5 * P, 6 * P, 64, None) == INVALID


def test_prenorm_entry_validation(lib):
    # (V, stride, n, T, d, dtype, w, gamma, eps, gamma_pre, eps_pre, out, out_normed, dtype)
    ok = (P, 64, 2, 4, 16, 1, P, P, 1e-6, P, 1e-6, 8 * P, 9 * P, 1)
    bad = [
        ok[:9] + (None,) + ok[10:],                      # no gamma_pre
        ok[:12] + (None,) + ok[13:],                     # no out_normed
        ok[:10] + (-1.0,) + ok[11:],                     # eps_pre < 0
        ok[:12] + (P + 64,) + ok[13:],                   # out_normed overlaps V
        ok[:12] + (8 * P + 16,) + ok[13:],               # out_normed overlaps out
    ]
    for args in bad:
        assert lib.attnres_full_fwd_prenorm(*args, None) == INVALID, args
    none_out = ok[:11] + (None,) + ok[12:]
    assert lib.attnres_full_fwd_prenorm(*(none_out[:3] + (0,) + none_out[4:]), None) == 0  # T = 0
    # pass: normed outputs overlapping the history
    assert lib.attnres_full_pass_prenorm(P, 64, 2, 4, 16, 1, P, P, 1e-6, P, 1e-6, None, P + 64, 64, 1,
                                         None) == INVALID
    # merge: no out_normed, out_normed aliasing P
    assert lib.attnres_block_merge_prenorm(P, 2 * P, 3 * P, 4 * P, 0, P, P, 1e-6, P, 1e-6, 4, 16, 1,
                                           5 * P, None, None) == INVALID
    assert lib.attnres_block_merge_prenorm(P, 2 * P, 3 * P, 4 * P, 0, P, P, 1e-6, P, 1e-6, 4, 16, 1,
                                           5 * P, 3 * P, None) == INVALID
    # rmsnorm: partial overlap (in place is fine, validated only)
    assert lib.attnres_rmsnorm(P, 4, 16, 1, P, 1e-6, P + 32, None) == INVALID
    assert lib.attnres_rmsnorm(P, 0, 16, 1, P, 1e-6, P, None) == 0


def test_full_bwd_validation(lib):
    # (V, stride, n, T, d, dtype, w, gamma, eps, dz, dz_dtype, dV, dv_stride, dw, dgamma)
    ok = (P, 64, 2, 4, 16, 1, P, P, 1e-6, 2 * P, 1, 8 * P, 64, 16 * P, 17 * P)
    bad = [
        ok[:2] + (0,) + ok[3:],                          # n_src = 0
        ok[:11] + (None,) + ok[12:],                     # no dV
        ok[:11] + (P + 64,) + ok[12:],                   # dV overlaps V
        ok[:11] + (2 * P,) + ok[12:],                    # dV overlaps dz
        ok[:13] + (8 * P + 64,) + ok[14:],               # dw overlaps dV
        ok[:14] + (16 * P + 32,),                        # dgamma overlaps dw
        ok[:10] + (9,) + ok[11:],                        # bad dz dtype
        ok[:12] + (63,) + ok[13:],                       # dv_stride < T*d
    ]
    for args in bad:
        assert lib.attnres_full_bwd(*args, None) == INVALID, args
    assert lib.attnres_full_bwd(*(ok[:3] + (0,) + ok[4:]), None) == 0  # T = 0


def test_block_bwd_validation(lib):
    need = (2 * 3 + 2 + 1) * 64
    assert lib.attnres_block_bwd_scratch_floats(2, 2, 4, 16) == need
    assert lib.attnres_block_bwd_scratch_floats(0, 2, 4, 16) == -1
    # (Src, src_stride, F, f_stride, N, S, T, d, dtype, W, Gamma, eps, dOut, dout_stride, dout_dtype,
    #  dEmb, dF, df_stride, dW, dGamma, scratch, scratch_floats)
    ok = (P, 64, 2 * P, 64, 2, 2, 4, 16, 1, 3 * P, 4 * P, 1e-6, 5 * P, 64, 1, 6 * P, 7 * P, 64, 8 * P, 9 * P,
          10 * P, need)
    bad = [
        ok[:4] + (0,) + ok[5:],                          # N = 0
        ok[:21] + (need - 1,),                           # scratch too short
        ok[:16] + (2 * P + 8,) + ok[17:],                # dF overlaps F
        ok[:20] + (6 * P + 16,) + ok[21:],               # scratch overlaps dEmb
        ok[:14] + (9,) + ok[15:],                        # bad dOut dtype
        ok[:17] + (63,) + ok[18:],                       # df_stride < T*d
        ok[:15] + (None,) + ok[16:],                     # no dEmb
    ]
    for args in bad:
        assert lib.attnres_block_bwd(*args, None) == INVALID, args
    assert lib.attnres_block_bwd(*(ok[:6] + (0,) + ok[7:]), None) == 0  # T = 0


def test_dynamic_query_validation(lib):
    # projection: fp32 H unsupported, Q overlapping H, null Wq, T = 0
    assert lib.attnres_query_projection(P, 4, 16, 0, 2 * P, 3 * P, None) == UNSUPPORTED
    assert lib.attnres_query_projection(P, 4, 16, 1, 2 * P, P + 32, None) == INVALID
    assert lib.attnres_query_projection(P, 4, 16, 1, None, 3 * P, None) == INVALID
    assert lib.attnres_query_projection(P, 0, 16, 1, 2 * P, 3 * P, None) == 0
    # read with per-token queries: no Q, Q overlapping out
    assert lib.attnres_full_fwd_dynq(P, 64, 2, 4, 16, 1, None, P, 1e-6, 8 * P, 1, None) == INVALID
    assert lib.attnres_full_fwd_dynq(P, 64, 2, 4, 16, 1, 8 * P + 16, P, 1e-6, 8 * P, 1, None) == INVALID


def test_dsplit_validation(lib):
    ptrs = (ctypes.c_void_p * 2)(P * 8, P * 16)
    same = (ctypes.c_void_p * 2)(P * 8, P * 8)
    # partials: S out of range, partials overlapping Src, shard wider than 512
    assert lib.attnres_stage1_dsplit_partials(P, 64, 2, 4, 16, 1, P, P, 0, 2 * P, 0, None) == INVALID
    assert lib.attnres_stage1_dsplit_partials(P, 64, 2, 4, 16, 1, P, P, 2, P + 32, 0, None) == INVALID
    assert lib.attnres_stage1_dsplit_partials(P, 4096, 2, 4, 1024, 1, P, P, 2, 8 * P, 0, None) == UNSUPPORTED
    # finish: d_total below the shard, overlapping outputs
    assert lib.attnres_stage1_dsplit_finish(P, 64, 2, 4, 16, 8, 1, 2 * P, 2, 1e-6, ptrs, None, None) == INVALID
    assert lib.attnres_stage1_dsplit_finish(P, 64, 2, 4, 16, 64, 1, 2 * P, 2, 1e-6, same, None, None) == INVALID


def test_kernel_selection(lib):
    A = 1 << 20
    # Full read: d multiple of 128 and 16-byte alignment -> fast kernel.
    assert binding.attnres_kernel_path(0, A, 2 * A, 8, 0, 8192, 896, 1) == 1
    assert binding.attnres_kernel_path(0, A, 2 * A, 141, 0, 32768, 640, 1) == 1
    assert binding.attnres_kernel_path(0, A, 2 * A, 8, 0, 256, 256, 0) == 1
    assert binding.attnres_kernel_path(0, A + 2, 2 * A, 8, 0, 256, 256, 1) == 0   # misaligned
    assert binding.attnres_kernel_path(0, A, 2 * A, 8, 0, 256, 100, 1) == 0       # d % 128
    # Stage 1 at the block shapes of the standard workloads.
    for n in range(1, 10):
        assert binding.attnres_kernel_path(1, A, 2 * A, n, 8, 16384, 1024, 1) == 1
        assert binding.attnres_kernel_path(1, A, 2 * A, n, 6, 131072, 2048, 1) == 1
    assert binding.attnres_kernel_path(1, A, 2 * A, 4, 9, 16384, 1024, 1) == 0    # S > 8
    # Merge and accumulate.
    assert binding.attnres_kernel_path(2, A, 2 * A, 0, 0, 16384, 1024, 1) == 1
    assert binding.attnres_kernel_path(2, A, 2 * A, 0, 0, 131072, 2048, 1) == 1
    assert binding.attnres_kernel_path(3, A, 2 * A, 0, 0, 16384, 1024, 1) == 1
    assert binding.attnres_kernel_path(2, A, 2 * A, 0, 0, 10, 3, 1) == 0
    assert binding.attnres_kernel_path(9, A, 2 * A, 0, 0, 10, 3, 1) == -1


def test_injected_launch_failure_reports_cuda_error(lib):
    """The launch-failure test hook: an armed failure makes the next launch
    return ATTNRES_ERR_CUDA without being made (before any CUDA call, so this
    runs without a GPU), and disarms itself once it fired."""
    CUDA_ERR = 3
    ptrs = (ctypes.c_void_p * 2)(P * 8, P * 16)
    calls = [
        lambda: lib.attnres_full_fwd(P, 64, 2, 4, 16, 1, P, P, 1e-6, 8 * P, 1, None),
        lambda: lib.attnres_full_pass(P, 64, 3, 4, 16, 1, P, P, 1e-6, 8 * P, 64, 1, None),
        lambda: lib.attnres_block_merge(P, 2 * P, 3 * P, 4 * P, 0, P, P, 1e-6, 4, 16, 1, 5 * P, None),
        lambda: lib.attnres_block_summary_accumulate(P, 2 * P, 0, 3 * P, 4, 16, 1, None),
        lambda: lib.attnres_rmsnorm(P, 4, 16, 1, P, 1e-6, 2 * P, None),
        lambda: lib.attnres_block_pass(P, 64, 2, 2, 4, 16, 1, 9 * P, 9 * P, 1e-6, 2 * P, 64, 0, 3 * P, 4 * P,
                                       5 * P, 6 * P, 64, None),
    ]
    assert binding.attnres_test_fail_launch(-1) == -1      # off by default
    for call in calls:
        assert binding.attnres_test_fail_launch(0) == -1
        assert call() == CUDA_ERR
        assert binding.attnres_test_fail_launch(-1) == -1  # it fired and disarmed
    # Argument errors are found before any launch: they leave it armed.
    binding.attnres_test_fail_launch(0)
    assert lib.attnres_full_fwd(P, 64, 0, 4, 16, 1, P, P, 1e-6, 8 * P, 1, None) == INVALID
    assert lib.attnres_block_stage1(P, 64, 2, 4, 16, 1, P, P, 0, 1e-6, ptrs, None, None) == INVALID
    assert binding.attnres_test_fail_launch(-1) == 0
    # Counting down: two more launches allowed, then the failure.
    binding.attnres_test_fail_launch(2)
    assert binding.attnres_test_fail_launch(-1) == 2


def test_withhold_hook_validation(lib):
    assert lib.attnres_test_withhold_stage(9, 0) == INVALID
    assert lib.attnres_test_withhold_stage(1, -1) == INVALID
    assert lib.attnres_test_withhold_stage(-1, 0) == INVALID
    assert lib.attnres_test_withhold_stage(2, 3) == 0
    assert lib.attnres_test_withhold_stage(0, -1) == 0      # off again


def test_noalloc_validation_order(lib):
    """attnres_block_pass_noalloc checks its arguments before its workspace
    limit, so a call that is both malformed and too large reports the
    malformed argument; a well-formed oversized call is refused as
    unsupported. Neither reaches the GPU."""
    N, S, T, d = 2, 8, 8192, 1024          # needs about 144 MiB of workspace: too large
    E = T * d
    f = ctypes.c_float(1e-6)
    assert lib.attnres_block_pass_noalloc(P, E, N, S, T, d, 1, P, P, f, 2 * P, E, 0, 3 * P, E, None) == UNSUPPORTED
    assert lib.attnres_block_pass_noalloc(None, E, N, S, T, d, 1, P, P, f, 2 * P, E, 0, 3 * P, E, None) == INVALID
    assert lib.attnres_block_pass_noalloc(P, E - 1, N, S, T, d, 1, P, P, f, 2 * P, E, 0, 3 * P, E, None) == INVALID
    assert lib.attnres_block_pass_noalloc(P, E, N, S, T, d, 1, P, P, ctypes.c_float(-1.0), 2 * P, E, 0, 3 * P, E,
                                          None) == INVALID
    assert lib.attnres_block_pass_noalloc(P, E, N, 0, T, d, 1, P, P, f, 2 * P, E, 0, 3 * P, E, None) == INVALID
    assert lib.attnres_block_pass_noalloc(P, E, N, S, 0, d, 1, P, P, f, 2 * P, E, 0, 3 * P, E, None) == 0


def _plan_bytes(S, es, kept):
    """Bytes per element the running sums of one block move under a plan
    (kept: the positions j < S whose sum is stored): position j (1..S, S the
    freeze) reads the outputs since the last kept position m (es each) and,
    if m > 0, the kept fp32 sum (4); a kept sum is written once (4)."""
    total, m = 0, 0
    for j in range(1, S + 1):
        total += es * (j - m) + (4 if m > 0 else 0)
        if j < S and j in kept:
            total += 4
            m = j
    return total


@pytest.mark.parametrize("dtype,es", [(1, 2), (0, 4)])
def test_running_sum_plan_is_the_cheapest(lib, dtype, es):
    import itertools
    for S in range(1, 17):
        plan = binding.attnres_block_running_sum_plan(S, dtype)
        assert len(plan) == S + 1 and plan[0] == 0 and plan[S] == 0
        kept = {j for j in range(1, S) if plan[j]}
        got = _plan_bytes(S, es, kept)
        best = min(_plan_bytes(S, es, set(c)) for r in range(S) for c in itertools.combinations(range(1, S), r))
        assert got == best, (S, kept, got, best)
        fewest = min(len(c) for r in range(S) for c in itertools.combinations(range(1, S), r)
                     if _plan_bytes(S, es, set(c)) == best)
        assert len(kept) == fewest
    # The long-context workload's blocks (bf16, S = 6) keep P_4 alone:
    # 38 bytes per element instead of 52 for a sum stored at every step.
    assert binding.attnres_block_running_sum_plan(6, 1) == [0, 0, 0, 0, 1, 0, 0]
    assert _plan_bytes(6, 2, {4}) == 38 and _plan_bytes(6, 2, {1, 2, 3, 4, 5}) == 52
    assert lib.attnres_block_running_sum_plan(0, 1, None) == INVALID


def test_merge_parts_validation(lib):
    # (O, lse, P_base, F_parts, part_stride, n_parts, P_out, w, gamma, eps, T, d, dtype, out, summary_out)
    f = ctypes.c_float(1e-6)
    E = 64
    assert lib.attnres_block_merge_parts(P, 2 * P, None, None, E, 0, None, P, P, f, 4, 16, 1, 5 * P, None,
                                         None) == INVALID
    assert lib.attnres_block_merge_parts(P, 2 * P, None, 3 * P, E - 1, 2, None, P, P, f, 4, 16, 1, 5 * P,
                                         None, None) == INVALID                   # parts overlap each other
    assert lib.attnres_block_merge_parts(P, 2 * P, None, 3 * P, E, 17, None, P, P, f, 4, 16, 1, 5 * P,
                                         None, None) == INVALID                   # too many parts
    assert lib.attnres_block_merge_parts(P, 2 * P, 4 * P, 3 * P, E, 2, 4 * P + 64, P, P, f, 4, 16, 1, 5 * P,
                                         None, None) == INVALID                   # P_out partly over P_base
    assert lib.attnres_block_merge_parts(P, 2 * P, None, 3 * P, E, 2, 3 * P, P, P, f, 4, 16, 1, 5 * P,
                                         None, None) == INVALID                   # P_out over the parts
    # The summary: one part more (16 at most), written over nothing else.
    assert lib.attnres_block_merge_parts(P, 2 * P, None, 3 * P, E, 16, None, P, P, f, 4, 16, 1, 5 * P,
                                         6 * P, None) == INVALID                  # 17 parts
    assert lib.attnres_block_merge_parts(P, 2 * P, None, 3 * P, E, 2, None, P, P, f, 4, 16, 1, 5 * P,
                                         5 * P, None) == INVALID                  # summary over out
    assert lib.attnres_block_merge_parts(P, 2 * P, None, 3 * P, E, 2, None, P, P, f, 4, 16, 1, 5 * P,
                                         3 * P + 2 * E * 2, None) == INVALID      # summary over the extra part
    assert lib.attnres_block_merge_parts(P, 2 * P, None, None, E, 0, None, P, P, f, 4, 16, 1, 5 * P,
                                         6 * P, None) == INVALID                  # no parts, no base
    binding.attnres_test_fail_launch(0)                                         # valid: reaches the launch
    assert lib.attnres_block_merge_parts(P, 2 * P, 4 * P, 3 * P, E, 2, 4 * P, P, P, f, 4, 16, 1, 5 * P,
                                         None, None) == 3
    binding.attnres_test_fail_launch(0)
    assert lib.attnres_block_merge_parts(P, 2 * P, 4 * P, 3 * P, E, 2, 4 * P, P, P, f, 4, 16, 1, 5 * P,
                                         6 * P, None) == 3
    binding.attnres_test_fail_launch(0)
    assert lib.attnres_block_summary_parts(None, 3 * P, E, 3, None, 5 * P, 4, 16, 1, None) == 3
    binding.attnres_test_fail_launch(-1)
    assert lib.attnres_block_summary_parts(None, 3 * P, E, 0, None, 5 * P, 4, 16, 1, None) == INVALID
    assert lib.attnres_block_summary_parts(None, 3 * P, E, 2, None, None, 4, 16, 1, None) == INVALID
