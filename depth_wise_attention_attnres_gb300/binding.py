"""Thin Python binding over libattnres.so (argument marshalling only).

Every function has the name of the C entry point it calls and does nothing
but turn torch CUDA tensors into pointers, sizes and dtype codes, pass the
current stream, and raise ``AttnResError`` on a non-zero status. All
arithmetic happens in the library's CUDA kernels; there is no other path. If
the library has not been built the first call raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from . import build as _build

F32, BF16 = 0, 1
_STATUS = {0: "ATTNRES_OK", 1: "ATTNRES_ERR_INVALID_ARG", 2: "ATTNRES_ERR_UNSUPPORTED",
           3: "ATTNRES_ERR_CUDA", 4: "ATTNRES_ERR_TIMEOUT"}

_lib = None
_lock = threading.Lock()

_VP, _I32, _I64, _F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
_SIGNATURES = {
    "attnres_full_fwd": [_VP, _I64, _I32, _I64, _I32, _I32, _VP, _VP, _F, _VP, _I32, _VP],
    "attnres_full_pass": [_VP, _I64, _I32, _I64, _I32, _I32, _VP, _VP, _F, _VP, _I64, _I32, _VP],
    "attnres_full_fwd_prenorm": [_VP, _I64, _I32, _I64, _I32, _I32, _VP, _VP, _F, _VP, _F, _VP, _VP,
                                 _I32, _VP],
    "attnres_full_pass_prenorm": [_VP, _I64, _I32, _I64, _I32, _I32, _VP, _VP, _F, _VP, _F, _VP,
                                  _VP, _I64, _I32, _VP],
    "attnres_rmsnorm": [_VP, _I64, _I32, _I32, _VP, _F, _VP, _VP],
    "attnres_stage1_dsplit_partials": [_VP, _I64, _I32, _I64, _I32, _I32, _VP, _VP, _I32, _VP, _I32, _VP],
    "attnres_stage1_dsplit_finish": [_VP, _I64, _I32, _I64, _I32, _I32, _I32, _VP, _I32, _F,
                                     ctypes.POINTER(_VP), _VP, _VP],
    "attnres_query_projection": [_VP, _I64, _I32, _I32, _VP, _VP, _VP],
    "attnres_full_fwd_dynq": [_VP, _I64, _I32, _I64, _I32, _I32, _VP, _VP, _F, _VP, _I32, _VP],
    "attnres_full_bwd": [_VP, _I64, _I32, _I64, _I32, _I32, _VP, _VP, _F, _VP, _I32, _VP, _I64, _VP, _VP,
                         _VP],
    "attnres_block_bwd": [_VP, _I64, _VP, _I64, _I32, _I32, _I64, _I32, _I32, _VP, _VP, _F, _VP, _I64, _I32,
                          _VP, _VP, _I64, _VP, _VP, _VP, _I64, _VP],
    "attnres_block_bwd_scratch_floats": [_I32, _I32, _I64, _I32],
    "attnres_block_stage1": [_VP, _I64, _I32, _I64, _I32, _I32, _VP, _VP, _I32, _F,
                             ctypes.POINTER(_VP), _VP, _VP],
    "attnres_block_merge": [_VP, _VP, _VP, _VP, _I32, _VP, _VP, _F, _I64, _I32, _I32, _VP, _VP],
    "attnres_block_merge_prenorm": [_VP, _VP, _VP, _VP, _I32, _VP, _VP, _F, _VP, _F, _I64, _I32, _I32,
                                    _VP, _VP, _VP],
    "attnres_block_summary_accumulate": [_VP, _VP, _I32, _VP, _I64, _I32, _I32, _VP],
    "attnres_block_merge_parts": [_VP, _VP, _VP, _VP, _I64, _I32, _VP, _VP, _VP, _F, _I64, _I32, _I32, _VP,
                                  _VP, _VP],
    "attnres_block_summary_parts": [_VP, _VP, _I64, _I32, _VP, _VP, _I64, _I32, _I32, _VP],
    "attnres_block_running_sum_plan": [_I32, _I32, ctypes.POINTER(_I32)],
    "attnres_block_pass": [_VP, _I64, _I32, _I32, _I64, _I32, _I32, _VP, _VP, _F, _VP, _I64,
                           _I32, _VP, _VP, _VP, _VP, _I64, _VP],
    "attnres_block_pass_noalloc": [_VP, _I64, _I32, _I32, _I64, _I32, _I32, _VP, _VP, _F, _VP,
                                   _I64, _I32, _VP, _I64, _VP],
    "attnres_device_status": [_VP],
    "attnres_selftest_wait_timeout": [_VP],
    "attnres_test_fail_launch": [_I64],
    "attnres_test_withhold_stage": [_I32, _I64],
    "attnres_status_string": [_I32],
    "attnres_kernel_path": [_I32, _VP, _VP, _I32, _I32, _I64, _I32, _I32],
    "attnres_abi_version": [],
}


class AttnResError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {_STATUS.get(status, status)}: "
                         f"{status_string(status)}")


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libattnres.so not found at {path}: build it first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            handle = ctypes.CDLL(path)
            for name, args in _SIGNATURES.items():
                fn = getattr(handle, name)
                fn.argtypes = args
                fn.restype = (ctypes.c_char_p if name == "attnres_status_string" else
                              ctypes.c_int64 if name in ("attnres_block_bwd_scratch_floats",
                                                         "attnres_test_fail_launch") else ctypes.c_int)
            _lib = handle
    return _lib


def header_functions(path: str | None = None) -> list[str]:
    """Names of the functions declared in include/attnres.h."""
    path = path or os.path.join(_build.INCLUDE, "attnres.h")
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attnres_[a-z0-9_]+)\s*\(", text)))


# ------------------------------------------------------------ marshalling ----

def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"storage dtype must be float32 or bfloat16, got {t.dtype}")


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("tensors passed to libattnres must be on a CUDA device")
    return t.data_ptr()


def _rows(t: torch.Tensor) -> tuple[int, int]:
    """(T, d) of a [T, d] tensor with contiguous rows."""
    if t.dim() != 2 or t.stride(1) != 1 or t.stride(0) != t.shape[1]:
        raise ValueError("expected a contiguous [T, d] tensor")
    return t.shape[0], t.shape[1]


def _slices(t: torch.Tensor) -> tuple[int, int, int, int]:
    """(n, T, d, stride) of [n, T, d] consecutive [T, d] slices."""
    if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
        raise ValueError("expected [n, T, d] with contiguous [T, d] slices")
    return t.shape[0], t.shape[1], t.shape[2], t.stride(0)


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(name: str, status: int) -> None:
    if status != 0:
        raise AttnResError(name, status)


# ---------------------------------------------------------------- entries ----

def attnres_full_fwd(V: torch.Tensor, n_src: int, w: torch.Tensor, gamma: torch.Tensor,
                     eps: float, out: torch.Tensor, stream=None) -> torch.Tensor:
    """One Full AttnRes read over V[0 .. n_src) (V is [n, T, d]) into out [T, d]."""
    _, T, d, stride = _slices(V)
    if _rows(out) != (T, d):
        raise ValueError("out must be [T, d]")
    _check("attnres_full_fwd", lib().attnres_full_fwd(
        _ptr(V), stride, n_src, T, d, _dtype(V), _ptr(w), _ptr(gamma), eps, _ptr(out),
        _dtype(out), _stream(stream)))
    return out


def attnres_full_pass(V: torch.Tensor, W: torch.Tensor, Gamma: torch.Tensor, eps: float,
                      out: torch.Tensor, R: int | None = None, stream=None) -> torch.Tensor:
    """R reads over history V [R, T, d]; read r uses V[0 .. r] and writes out[r]."""
    n, T, d, stride = _slices(V)
    R = n if R is None else R
    on, oT, od, ostride = _slices(out)
    if (oT, od) != (T, d) or on < R:
        raise ValueError("out must be [R, T, d]")
    _check("attnres_full_pass", lib().attnres_full_pass(
        _ptr(V), stride, R, T, d, _dtype(V), _ptr(W), _ptr(Gamma), eps, _ptr(out), ostride,
        _dtype(out), _stream(stream)))
    return out


def attnres_full_fwd_prenorm(V: torch.Tensor, n_src: int, w: torch.Tensor, gamma: torch.Tensor,
                             eps: float, gamma_pre: torch.Tensor, eps_pre: float,
                             out: torch.Tensor | None, out_normed: torch.Tensor,
                             stream=None) -> torch.Tensor:
    """A Full read that also writes the sublayer pre-norm of its result into
    out_normed [T, d]; out (z itself) may be None."""
    _, T, d, stride = _slices(V)
    if _rows(out_normed) != (T, d) or (out is not None and _rows(out) != (T, d)):
        raise ValueError("out and out_normed must be [T, d]")
    if out is not None and out.dtype != out_normed.dtype:
        raise ValueError("out and out_normed must have one dtype")
    _check("attnres_full_fwd_prenorm", lib().attnres_full_fwd_prenorm(
        _ptr(V), stride, n_src, T, d, _dtype(V), _ptr(w), _ptr(gamma), eps, _ptr(gamma_pre),
        eps_pre, _ptr(out), _ptr(out_normed), _dtype(out_normed), _stream(stream)))
    return out_normed


def attnres_full_pass_prenorm(V: torch.Tensor, W: torch.Tensor, Gamma: torch.Tensor, eps: float,
                              Gamma_pre: torch.Tensor, eps_pre: float, out: torch.Tensor | None,
                              out_normed: torch.Tensor, R: int | None = None,
                              stream=None) -> torch.Tensor:
    """R reads over history V [R, T, d], read r also writing the pre-norm of its
    result (with Gamma_pre[r]) into out_normed[r]; out may be None."""
    n, T, d, stride = _slices(V)
    R = n if R is None else R
    on, oT, od, ostride = _slices(out_normed)
    if (oT, od) != (T, d) or on < R:
        raise ValueError("out_normed must be [R, T, d]")
    if out is not None:
        if _slices(out)[1:] != (T, d, ostride) or out.shape[0] < R or out.dtype != out_normed.dtype:
            raise ValueError("out must match out_normed")
    _check("attnres_full_pass_prenorm", lib().attnres_full_pass_prenorm(
        _ptr(V), stride, R, T, d, _dtype(V), _ptr(W), _ptr(Gamma), eps, _ptr(Gamma_pre), eps_pre,
        _ptr(out), _ptr(out_normed), ostride, _dtype(out_normed), _stream(stream)))
    return out_normed


def attnres_full_bwd(V: torch.Tensor, n_src: int, w: torch.Tensor, gamma: torch.Tensor, eps: float,
                     dz: torch.Tensor, dV: torch.Tensor, dw: torch.Tensor | None = None,
                     dgamma: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Backward of the read over V[0 .. n_src): ADD dL/dV (fp32 [n, T, d]) into dV
    and dL/dw, dL/dgamma (fp32 [d]) into dw, dgamma, given dz = dL/dz [T, d]."""
    _, T, d, stride = _slices(V)
    dn, dT, dd, dstride = _slices(dV)
    if (dT, dd) != (T, d) or dn < n_src or dV.dtype != torch.float32:
        raise ValueError("dV must be fp32 [n_src, T, d]")
    if _rows(dz) != (T, d):
        raise ValueError("dz must be [T, d]")
    for t in (dw, dgamma):
        if t is not None and (t.dtype != torch.float32 or t.numel() != d):
            raise ValueError("dw and dgamma must be fp32 [d]")
    _check("attnres_full_bwd", lib().attnres_full_bwd(
        _ptr(V), stride, n_src, T, d, _dtype(V), _ptr(w), _ptr(gamma), eps, _ptr(dz), _dtype(dz),
        _ptr(dV), dstride, _ptr(dw), _ptr(dgamma), _stream(stream)))
    return dV


def attnres_block_bwd_scratch_floats(N: int, S: int, T: int, d: int) -> int:
    """fp32 scratch elements attnres_block_bwd needs."""
    return int(lib().attnres_block_bwd_scratch_floats(N, S, T, d))


def attnres_block_bwd(Src: torch.Tensor, F: torch.Tensor, N: int, S: int, W: torch.Tensor, Gamma: torch.Tensor,
                      eps: float, dOut: torch.Tensor, dEmb: torch.Tensor, dF: torch.Tensor,
                      dW: torch.Tensor | None = None, dGamma: torch.Tensor | None = None,
                      scratch: torch.Tensor | None = None, stream=None) -> None:
    """Backward of a Block pass: ADD dL/d(embedding) into dEmb (fp32 [T, d]), dL/dF
    into dF (fp32 [N*S, T, d]) and dL/dW, dL/dGamma into dW, dGamma (fp32 [N*S, d]),
    given dOut = dL/dout [N*S, T, d]. Src holds the embedding and the frozen block
    summaries the forward left (Src[0 .. N-1]). scratch: fp32, at least
    attnres_block_bwd_scratch_floats(N, S, T, d) elements (allocated here if None)."""
    _, T, d, fstride = _slices(F)
    _, _, _, sstride = _slices(Src)
    _, _, _, zstride = _slices(dOut)
    dn, dT, dd, dfstride = _slices(dF)
    if (dT, dd) != (T, d) or dn < N * S or dF.dtype != torch.float32:
        raise ValueError("dF must be fp32 [N*S, T, d]")
    if _rows(dEmb) != (T, d) or dEmb.dtype != torch.float32:
        raise ValueError("dEmb must be fp32 [T, d]")
    for t in (dW, dGamma):
        if t is not None and (t.dtype != torch.float32 or t.numel() != N * S * d or not t.is_contiguous()):
            raise ValueError("dW and dGamma must be contiguous fp32 [N*S, d]")
    need = attnres_block_bwd_scratch_floats(N, S, T, d)
    if scratch is None:
        scratch = torch.empty(need, device=F.device, dtype=torch.float32)
    if scratch.dtype != torch.float32 or scratch.numel() < need:
        raise ValueError(f"scratch must be fp32 with at least {need} elements")
    _check("attnres_block_bwd", lib().attnres_block_bwd(
        _ptr(Src), sstride, _ptr(F), fstride, N, S, T, d, _dtype(F), _ptr(W), _ptr(Gamma), eps, _ptr(dOut),
        zstride, _dtype(dOut), _ptr(dEmb), _ptr(dF), dfstride, _ptr(dW), _ptr(dGamma), _ptr(scratch),
        scratch.numel(), _stream(stream)))


def attnres_query_projection(H: torch.Tensor, Wq: torch.Tensor, Q: torch.Tensor, stream=None) -> torch.Tensor:
    """Q = H Wq^T (H bf16 [T, d], Wq bf16 [d, d], Q fp32 [T, d]): the input-dependent query."""
    T, d = _rows(H)
    if tuple(Wq.shape) != (d, d) or Wq.dtype != torch.bfloat16 or not Wq.is_contiguous():
        raise ValueError("Wq must be contiguous bf16 [d, d]")
    if _rows(Q) != (T, d) or Q.dtype != torch.float32:
        raise ValueError("Q must be fp32 [T, d]")
    _check("attnres_query_projection", lib().attnres_query_projection(
        _ptr(H), T, d, _dtype(H), _ptr(Wq), _ptr(Q), _stream(stream)))
    return Q


def attnres_full_fwd_dynq(V: torch.Tensor, n_src: int, Q: torch.Tensor, gamma: torch.Tensor, eps: float,
                          out: torch.Tensor, stream=None) -> torch.Tensor:
    """The Full read over V[0 .. n_src) with token t scored by its own query Q[t] (fp32 [T, d])."""
    _, T, d, stride = _slices(V)
    if _rows(out) != (T, d) or _rows(Q) != (T, d) or Q.dtype != torch.float32:
        raise ValueError("out must be [T, d] and Q fp32 [T, d]")
    _check("attnres_full_fwd_dynq", lib().attnres_full_fwd_dynq(
        _ptr(V), stride, n_src, T, d, _dtype(V), _ptr(Q), _ptr(gamma), eps, _ptr(out), _dtype(out),
        _stream(stream)))
    return out


def attnres_stage1_dsplit_partials(Src: torch.Tensor, n_src: int, W: torch.Tensor, Gamma: torch.Tensor,
                                   partials: torch.Tensor, accumulate: bool, stream=None) -> torch.Tensor:
    """One feature shard's part of the stage-1 score sums: Src [n, T, d_shard], W and
    Gamma fp32 [S, d_shard] (the shard's slices); partials fp32 [T, n_src, S + 1]."""
    _, T, ds, stride = _slices(Src)
    S = W.shape[0]
    if tuple(partials.shape) != (T, n_src, S + 1) or partials.dtype != torch.float32:
        raise ValueError("partials must be fp32 [T, n_src, S + 1]")
    _check("attnres_stage1_dsplit_partials", lib().attnres_stage1_dsplit_partials(
        _ptr(Src), stride, n_src, T, ds, _dtype(Src), _ptr(W), _ptr(Gamma), S, _ptr(partials),
        int(bool(accumulate)), _stream(stream)))
    return partials


def attnres_stage1_dsplit_finish(Src: torch.Tensor, n_src: int, d_total: int, partials: torch.Tensor,
                                 eps: float, O: list, lse: torch.Tensor | None, stream=None) -> None:
    """A shard's features of the S normalised reads from the summed partials."""
    _, T, ds, stride = _slices(Src)
    S = len(O)
    ptrs = (ctypes.c_void_p * max(S, 1))(*[_ptr(o) for o in O])
    _check("attnres_stage1_dsplit_finish", lib().attnres_stage1_dsplit_finish(
        _ptr(Src), stride, n_src, T, ds, d_total, _dtype(Src), _ptr(partials), S, eps, ptrs,
        _ptr(lse), _stream(stream)))


def attnres_rmsnorm(x: torch.Tensor, gamma: torch.Tensor, eps: float, out: torch.Tensor,
                    stream=None) -> torch.Tensor:
    """out = gamma * x / sqrt(mean(x^2) + eps) per row of x [T, d] (out may be x)."""
    T, d = _rows(x)
    if _rows(out) != (T, d) or out.dtype != x.dtype:
        raise ValueError("out must be like x")
    _check("attnres_rmsnorm", lib().attnres_rmsnorm(
        _ptr(x), T, d, _dtype(x), _ptr(gamma), eps, _ptr(out), _stream(stream)))
    return out


def attnres_block_stage1(Src: torch.Tensor, n_src: int, W: torch.Tensor, Gamma: torch.Tensor,
                         eps: float, O: list, lse: torch.Tensor | None, stream=None) -> None:
    """Stage 1: the S = len(O) queries of W [S, d] over Src[0 .. n_src)."""
    _, T, d, stride = _slices(Src)
    S = len(O)
    ptrs = (ctypes.c_void_p * max(S, 1))(*[_ptr(o) for o in O])
    _check("attnres_block_stage1", lib().attnres_block_stage1(
        _ptr(Src), stride, n_src, T, d, _dtype(Src), _ptr(W), _ptr(Gamma), S, eps, ptrs,
        _ptr(lse), _stream(stream)))


def attnres_block_merge(O_j: torch.Tensor, lse_j: torch.Tensor, P: torch.Tensor, f_prev,
                        p_is_empty: bool, w: torch.Tensor, gamma: torch.Tensor, eps: float,
                        out: torch.Tensor, stream=None) -> torch.Tensor:
    """Stage 2 for one sublayer (running sum P updated in place when f_prev is given)."""
    T, d = _rows(O_j)
    _check("attnres_block_merge", lib().attnres_block_merge(
        _ptr(O_j), _ptr(lse_j), _ptr(P), _ptr(f_prev), int(bool(p_is_empty)), _ptr(w),
        _ptr(gamma), eps, T, d, _dtype(O_j), _ptr(out), _stream(stream)))
    return out


def attnres_block_merge_prenorm(O_j: torch.Tensor, lse_j: torch.Tensor, P: torch.Tensor, f_prev,
                                p_is_empty: bool, w: torch.Tensor, gamma: torch.Tensor, eps: float,
                                gamma_pre: torch.Tensor, eps_pre: float, out, out_normed: torch.Tensor,
                                stream=None) -> torch.Tensor:
    """Stage 2 that also writes the sublayer pre-norm of the merged row into
    out_normed; out (the merged row itself) may be None."""
    T, d = _rows(O_j)
    _check("attnres_block_merge_prenorm", lib().attnres_block_merge_prenorm(
        _ptr(O_j), _ptr(lse_j), _ptr(P), _ptr(f_prev), int(bool(p_is_empty)), _ptr(w),
        _ptr(gamma), eps, _ptr(gamma_pre), eps_pre, T, d, _dtype(O_j), _ptr(out), _ptr(out_normed),
        _stream(stream)))
    return out_normed


def attnres_block_summary_accumulate(P, f: torch.Tensor, p_is_empty: bool, summary_out=None,
                                     stream=None) -> None:
    """P += f, or (freeze) summary_out = round(P + f)."""
    T, d = _rows(f)
    _check("attnres_block_summary_accumulate", lib().attnres_block_summary_accumulate(
        _ptr(P), _ptr(f), int(bool(p_is_empty)), _ptr(summary_out), T, d, _dtype(f),
        _stream(stream)))


def _parts(F_parts: torch.Tensor, n_parts: int) -> tuple[int, int, int, int]:
    """(T, d, part stride, dtype code) of the first n_parts slices of F_parts."""
    if F_parts.dim() == 2:
        if n_parts > 1:
            raise ValueError("several parts need an [n, T, d] tensor")
        T, d = _rows(F_parts)
        return T, d, T * d, _dtype(F_parts)
    n, T, d, stride = _slices(F_parts)
    if n < n_parts:
        raise ValueError(f"F_parts holds {n} slices, {n_parts} requested")
    return T, d, stride, _dtype(F_parts)


def attnres_block_merge_parts(O_j: torch.Tensor, lse_j: torch.Tensor, P_base, F_parts: torch.Tensor,
                              n_parts: int, P_out, w: torch.Tensor, gamma: torch.Tensor, eps: float,
                              out: torch.Tensor, summary_out=None, stream=None) -> torch.Tensor:
    """Merge with the running sum P_base + F_parts[0] + ... + F_parts[n_parts-1]
    (P_base may be None), storing it to P_out when given; with summary_out,
    also the block summary: that sum plus F_parts[n_parts], rounded."""
    T, d, pstride, code = _parts(F_parts, n_parts + (1 if summary_out is not None else 0))
    _check("attnres_block_merge_parts", lib().attnres_block_merge_parts(
        _ptr(O_j), _ptr(lse_j), _ptr(P_base), _ptr(F_parts), pstride, n_parts, _ptr(P_out), _ptr(w),
        _ptr(gamma), eps, T, d, code, _ptr(out), _ptr(summary_out), _stream(stream)))
    return out


def attnres_block_summary_parts(P_base, F_parts: torch.Tensor, n_parts: int, P_out=None, summary_out=None,
                                stream=None) -> None:
    """summary_out <- round(P_base + parts), or P_out <- that sum in fp32."""
    T, d, pstride, code = _parts(F_parts, n_parts)
    _check("attnres_block_summary_parts", lib().attnres_block_summary_parts(
        _ptr(P_base), _ptr(F_parts), pstride, n_parts, _ptr(P_out), _ptr(summary_out), T, d, code,
        _stream(stream)))


def attnres_block_running_sum_plan(S: int, dtype: int = BF16) -> list[int]:
    """stored[j] (0 <= j <= S): whether the Block pass keeps running sum P_j."""
    arr = (ctypes.c_int32 * (S + 1))()
    _check("attnres_block_running_sum_plan", lib().attnres_block_running_sum_plan(S, dtype, arr))
    return list(arr)


def attnres_block_pass(F: torch.Tensor, N: int, S: int, W: torch.Tensor, Gamma: torch.Tensor,
                       eps: float, Src: torch.Tensor, O_scratch, lse_scratch: torch.Tensor,
                       P_scratch, out: torch.Tensor, freeze_last: bool = False,
                       stream=None) -> torch.Tensor:
    """N blocks of S sublayers by the two-stage computation (Src[0] = embedding)."""
    _, T, d, fstride = _slices(F)
    _, _, _, sstride = _slices(Src)
    _, _, _, ostride = _slices(out)
    _check("attnres_block_pass", lib().attnres_block_pass(
        _ptr(F), fstride, N, S, T, d, _dtype(F), _ptr(W), _ptr(Gamma), eps, _ptr(Src), sstride,
        int(bool(freeze_last)), _ptr(O_scratch), _ptr(lse_scratch), _ptr(P_scratch), _ptr(out),
        ostride, _stream(stream)))
    return out


def attnres_block_pass_noalloc(F: torch.Tensor, N: int, S: int, W: torch.Tensor,
                               Gamma: torch.Tensor, eps: float, Src: torch.Tensor, out: torch.Tensor,
                               freeze_last: bool = False, stream=None) -> torch.Tensor:
    """The Block pass with the library's own fixed workspace (no allocation)."""
    _, T, d, fstride = _slices(F)
    _, _, _, sstride = _slices(Src)
    _, _, _, ostride = _slices(out)
    _check("attnres_block_pass_noalloc", lib().attnres_block_pass_noalloc(
        _ptr(F), fstride, N, S, T, d, _dtype(F), _ptr(W), _ptr(Gamma), eps, _ptr(Src), sstride,
        int(bool(freeze_last)), _ptr(out), ostride, _stream(stream)))
    return out


def attnres_device_status(stream=None) -> int:
    return int(lib().attnres_device_status(_stream(stream)))


def attnres_selftest_wait_timeout(stream=None) -> None:
    """Run the bounded-wait self-test kernel (its wait runs out after ~2 s)."""
    _check("attnres_selftest_wait_timeout", lib().attnres_selftest_wait_timeout(_stream(stream)))


def attnres_test_fail_launch(after: int) -> int:
    """Test hook: the launch after `after` more successful ones fails with
    ATTNRES_ERR_CUDA without being made (after < 0 disarms). Returns the
    previous setting (-1 once an armed failure has fired)."""
    return int(lib().attnres_test_fail_launch(int(after)))


# Kernels whose copy producer attnres_test_withhold_stage can starve.
WITHHOLD_NONE, WITHHOLD_FULL, WITHHOLD_STAGE1_TC, WITHHOLD_MERGE = 0, 1, 2, 3


def attnres_test_withhold_stage(kernel: int, index: int = 0) -> None:
    """Test hook: the producer of `kernel` leaves its copy number `index` (per
    CTA) unissued, so the consumers' bounded wait runs out (kernel 0: off)."""
    _check("attnres_test_withhold_stage", lib().attnres_test_withhold_stage(int(kernel), int(index)))


def status_string(status: int) -> str:
    return lib().attnres_status_string(int(status)).decode()


attnres_status_string = status_string


def attnres_kernel_path(op: int, src_ptr: int, out_ptr: int, n_or_s: int, s: int, T: int, d: int,
                        dtype: int) -> int:
    return int(lib().attnres_kernel_path(op, src_ptr, out_ptr, n_or_s, s, T, d, dtype))


def attnres_abi_version() -> int:
    return int(lib().attnres_abi_version())
