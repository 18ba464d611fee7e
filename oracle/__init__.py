"""fp64 CPU oracle for the AttnRes depth-wise aggregation.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package. The CUDA
library and its Python binding never import it, and it imports nothing from
them: the two share no code. The one thing both sides use is the seeded input
generator module, which holds none of the method's arithmetic.

The arithmetic of one read lives in ``attnres_oracle.c`` (plain fp64 loops).
This module adds the sequencing the pages describe on top of it:

* ``full_read`` / ``full_pass``: Full AttnRes. Read r of a pass aggregates the
  embedding and the r sublayer outputs before it (DepthBench reading notes,
  section 2.3 "Full AttnRes", Appendix A; LLMRes blog, "Kimi AttnRes":
  h_l = sum_{i=0}^{l-1} alpha_{i->l} v_i).
* ``block_pass``: Block AttnRes by its plain definition (DepthBench reading
  notes section 2.5; LLMRes blog "Block Attention Residuals"; datacamp
  explainer "block attention residuals"): sublayer k in block n (0-based) with
  in-block index j reads {embedding, b_1 .. b_n, P_k if j >= 1}, where b_m is
  the plain sum of block m's member outputs and P_k the sum of the outputs of
  the earlier sublayers of the current block. An empty running sum (j = 0) is
  not a source. Sums are exact fp64 additions of the stored outputs.
* ``read_bwd`` / ``full_read_bwd``: the gradients of one read with respect to
  its sources, its query w and its key-norm gain gamma, given the gradient of
  the result, by the chain rule through the read's definition (the
  backward the pages point to when they note that stored sublayer outputs
  are reused for it; DepthBench reading notes section 2.3 for the read).
* ``block_pass_bwd``: the gradients of a whole Block pass by the chain rule
  through its definition: each read's ``read_bwd`` over its source set, the
  gradient of a block summary b_m (a plain sum) passed unchanged to every
  member output of block m, and that of the running sum P_k to every earlier
  output of the current block.
* ``query_projection`` / ``read_dynamic_query``: the input-dependent query
  the pages report as an ablation (LLMRes blog, on the paper's ablation: a
  query projected from the current hidden state by a per-layer d x d matrix
  instead of the fixed learned pseudo-query): q(t) = W_q h(t) per token, and
  the read scored with that per-token query.
* ``prenorm``: the consuming sublayer's pre-norm of an aggregated row,
  RMSNorm_pre(z) (DepthBench reading notes section 2.3: f_l =
  F_l(RMSNorm_pre,l(z_l))), which the library can emit next to z.
* ``block_stage1`` / ``block_merge`` / ``block_accumulate``: the per-operation
  references for the two-stage computation (datacamp explainer, "two-stage
  computation"), each written as the plain read over the source set the
  operation stands for, not as the two-stage algorithm.

parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, hand-worked golden cases and an independent
pure-Python brute force, ``oracle/bruteforce.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attnres_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

F32, BF16, F64 = 0, 1, 2

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``attnres_oracle.c`` into ``oracle/_build/liboracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", "-Wall",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Open an oracle shared library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    lib.attnres_oracle_read.restype = ctypes.c_int
    lib.attnres_oracle_read.argtypes = [
        ctypes.c_int, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_int),
        ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_double, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
        ctypes.c_void_p]
    lib.attnres_oracle_threads.restype = ctypes.c_int
    lib.attnres_oracle_threads.argtypes = []
    lib.attnres_oracle_set_threads.restype = None
    lib.attnres_oracle_set_threads.argtypes = [ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def threads() -> int:
    """OpenMP threads one oracle call uses."""
    return int(_load().attnres_oracle_threads())


def set_threads(n: int) -> None:
    """Threads later oracle calls use (results do not depend on it)."""
    _load().attnres_oracle_set_threads(int(n))


# ---------------------------------------------------------------- storage ----

def as_stored(x):
    """Return (contiguous numpy array, dtype tag) for a stored tensor.

    Accepts numpy float32/float64 arrays, numpy uint16 arrays holding bf16 bit
    patterns (tag must then be given by wrapping in ``Bf16Bits``), and CPU torch
    tensors of dtype float32, float64 or bfloat16.
    """
    if isinstance(x, Bf16Bits):
        return np.ascontiguousarray(x.bits, dtype=np.uint16), BF16
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach()
            if x.device.type != "cpu":
                raise ValueError("the oracle takes host tensors only")
            if x.dtype == torch.bfloat16:
                return np.ascontiguousarray(x.contiguous().view(torch.int16).numpy().view(np.uint16)), BF16
            if x.dtype == torch.float32:
                return np.ascontiguousarray(x.numpy()), F32
            if x.dtype == torch.float64:
                return np.ascontiguousarray(x.numpy()), F64
            raise TypeError(f"unsupported tensor dtype {x.dtype}")
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    x = np.asarray(x)
    if x.dtype == np.float32:
        return np.ascontiguousarray(x), F32
    if x.dtype == np.float64:
        return np.ascontiguousarray(x), F64
    raise TypeError(f"unsupported array dtype {x.dtype}")


class Bf16Bits:
    """A numpy uint16 array marked as holding bf16 bit patterns."""

    def __init__(self, bits):
        self.bits = np.asarray(bits, dtype=np.uint16)
        self.shape = self.bits.shape


def widen(x) -> np.ndarray:
    """Exact fp64 copy of a stored tensor (bf16 widened bit-exactly)."""
    arr, tag = as_stored(x)
    if tag == BF16:
        return (arr.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return arr.astype(np.float64)


# ------------------------------------------------------------------ reads ----

def read(sources, w, gamma, eps, rows=None):
    """One AttnRes read over ``sources`` (each a stored [T, d] tensor).

    Returns ``(out, lse)``: fp64 [n_rows, d] and fp64 [n_rows]. ``rows`` picks
    token rows (default: all T).
    """
    if len(sources) < 1:
        raise ValueError("a read needs at least one source")
    arrs = [as_stored(s) for s in sources]
    T, d = arrs[0][0].shape
    for a, _ in arrs:
        if a.shape != (T, d):
            raise ValueError("all sources of a read must be [T, d]")
    w64 = np.ascontiguousarray(np.asarray(w, dtype=np.float64).reshape(d))
    g64 = np.ascontiguousarray(np.asarray(gamma, dtype=np.float64).reshape(d))
    rows64 = np.arange(T, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n_rows = rows64.shape[0]
    out = np.empty((n_rows, d), dtype=np.float64)
    lse = np.empty((n_rows,), dtype=np.float64)
    n = len(arrs)
    bases = (ctypes.c_void_p * n)(*[a.ctypes.data for a, _ in arrs])
    tags = (ctypes.c_int * n)(*[t for _, t in arrs])
    rc = _load().attnres_oracle_read(
        n, bases, tags, T, d, w64.ctypes.data, g64.ctypes.data, float(eps),
        rows64.ctypes.data if n_rows else None, n_rows,
        out.ctypes.data if n_rows else None, lse.ctypes.data if n_rows else None)
    if rc != 0:
        raise ValueError(f"attnres_oracle_read failed with code {rc}")
    return out, lse


def query_projection(H, Wq):
    """Per-token query q(t) = Wq h(t): fp64 [T, d_out] from H [T, d_in] and Wq
    [d_out, d_in] (stored or fp64)."""
    h = np.asarray(H, np.float64) if isinstance(H, np.ndarray) else widen(H)
    w = np.asarray(Wq, np.float64) if isinstance(Wq, np.ndarray) else widen(Wq)
    return h @ w.T


def read_dynamic_query(sources, Q, gamma, eps):
    """A read whose query differs per token: e_i(t) = Q(t) . (gamma * v_i(t)) *
    r_i(t), a(t) = softmax_i(e(t)), z(t) = sum_i a_i(t) v_i(t). Q is [T, d].
    Returns (z fp64 [T, d], lse fp64 [T])."""
    V = np.stack([widen(s) if not isinstance(s, np.ndarray) else np.asarray(s, np.float64)
                  for s in sources])                      # [n, T, d]
    q = np.asarray(Q, np.float64) if isinstance(Q, np.ndarray) else widen(Q)
    g = np.asarray(gamma, np.float64).reshape(-1)
    r = 1.0 / np.sqrt(np.mean(V * V, axis=-1) + eps)      # [n, T]
    e = r * np.einsum("ntk,tk->nt", V, q * g)
    m = e.max(axis=0)
    p = np.exp(e - m)
    z = p.sum(axis=0)
    out = np.einsum("nt,ntk->tk", p / z, V)
    return out, m + np.log(z)


def read_bwd(sources, w, gamma, eps, dz):
    """Gradients of one read: (dV fp64 [n, T, d], dw fp64 [d], dgamma fp64 [d]).

    dz is dL/dz for the read's result z ([T, d], stored or fp64). The read is
    e_i = w . (gamma * v_i) * r_i with r_i = 1 / sqrt(mean_k v_ik^2 + eps),
    a = softmax_i(e), z = sum_i a_i v_i. With u = w * gamma, per token:
      dL/da_i = dz . v_i;  dL/de_i = a_i (dL/da_i - sum_j a_j dL/da_j)
      dL/dv_i = a_i dz + dL/de_i (r_i u - e_i r_i^2 v_i / d)
      dL/du = sum_i dL/de_i r_i v_i  (summed over tokens);
      dL/dw = dL/du * gamma, dL/dgamma = dL/du * w.
    """
    V = np.stack([widen(s) if not isinstance(s, np.ndarray) else np.asarray(s, np.float64)
                  for s in sources])                      # [n, T, d]
    g = np.asarray(dz, dtype=np.float64) if isinstance(dz, np.ndarray) else widen(dz)
    d = V.shape[-1]
    w64 = np.asarray(w, dtype=np.float64).reshape(d)
    g64 = np.asarray(gamma, dtype=np.float64).reshape(d)
    u = w64 * g64
    r = 1.0 / np.sqrt(np.mean(V * V, axis=-1) + eps)      # [n, T]
    e = r * np.einsum("ntk,k->nt", V, u)
    a = np.exp(e - e.max(axis=0, keepdims=True))
    a /= a.sum(axis=0, keepdims=True)
    da = np.einsum("ntk,tk->nt", V, g)
    de = a * (da - np.sum(a * da, axis=0, keepdims=True))
    dV = a[..., None] * g[None] + de[..., None] * (r[..., None] * u - (e * r * r / d)[..., None] * V)
    du = np.einsum("nt,ntk->k", de * r, V)
    return dV, du * g64, du * w64


def full_read_bwd(V, n_src, w, gamma, eps, dz):
    """Gradients of the Full read over V[0 .. n_src) (see ``read_bwd``)."""
    return read_bwd(_slices(V, n_src), w, gamma, eps, dz)


def block_pass_bwd(Src, F, N, S, W, Gamma, eps, dOut):
    """Gradients of a Block AttnRes pass with loss sum_k <dOut[k], out_k>.

    Src: the embedding (Src[0]) and the frozen block summaries b_1 .. b_{N-1}
    as the forward stored them; the reads take them as given. F: [N*S, T, d]
    sublayer outputs; the running sums P_k are exact fp64 sums of them. W,
    Gamma: [N*S, d]. dOut: [N*S, T, d]. Returns fp64 (dEmb [T, d], dF [N*S, T,
    d], dW [N*S, d], dGamma [N*S, d]). A summary b_m is the plain sum of block
    (m-1)'s outputs, so its gradient reaches each of them unchanged; the
    gradient of P_k reaches each output of the current block before k.
    """
    s64 = [widen(Src[i]) if not isinstance(Src, np.ndarray) else np.asarray(Src[i], np.float64)
           for i in range(N)]
    f64 = widen(F) if not isinstance(F, np.ndarray) else np.asarray(F, np.float64)
    g = widen(dOut) if not isinstance(dOut, np.ndarray) else np.asarray(dOut, np.float64)
    W64 = np.asarray(W, np.float64)
    G64 = np.asarray(Gamma, np.float64)
    dEmb = np.zeros_like(s64[0])
    dF = np.zeros_like(f64)
    dW = np.zeros((N * S, W64.shape[-1]))
    dG = np.zeros_like(dW)
    for k in range(N * S):
        n, j = divmod(k, S)
        srcs = [s64[m] for m in range(n + 1)]
        if j >= 1:
            srcs.append(np.sum(f64[n * S:k], axis=0))
        dV, dW[k], dG[k] = read_bwd(srcs, W64[k], G64[k], eps, g[k])
        dEmb += dV[0]
        for m in range(1, n + 1):
            dF[(m - 1) * S:m * S] += dV[m]
        if j >= 1:
            dF[n * S:k] += dV[n + 1]
    return dEmb, dF, dW, dG


def _slices(V, n):
    if isinstance(V, Bf16Bits):
        return [Bf16Bits(V.bits[i]) for i in range(n)]
    return [V[i] for i in range(n)]


def full_read(V, n_src, w, gamma, eps, rows=None):
    """Full AttnRes read over the first ``n_src`` entries of history V[n, T, d]."""
    return read(_slices(V, n_src), w, gamma, eps, rows)


def full_pass(V, R, W, Gamma, eps, rows=None):
    """Full AttnRes pass: read r (0 <= r < R) aggregates V[0 .. r].

    Returns fp64 [R, n_rows, d]. Sublayer r's own output is V[r + 1], so read r
    sees the embedding and every earlier sublayer output, as in the pages'
    h_l = sum_{i<l} alpha_{i->l} v_i.
    """
    outs = []
    for r in range(R):
        o, _ = full_read(V, r + 1, W[r], Gamma[r], eps, rows)
        outs.append(o)
    return np.stack(outs)


def block_sources(k, S, emb64, F64):
    """Source list of sublayer k of a Block AttnRes pass (all fp64, [rows, d]).

    k is the 0-based global sublayer index, S the sublayers per block;
    F64[q] is sublayer q's output. Returns [embedding, b_1 .. b_n] plus the
    running sum of the current block when it is non-empty.
    """
    n, j = divmod(k, S)
    srcs = [emb64]
    for m in range(1, n + 1):
        srcs.append(np.sum(F64[(m - 1) * S: m * S], axis=0))
    if j >= 1:
        srcs.append(np.sum(F64[n * S: k], axis=0))
    return srcs


def block_pass(emb, F, N, S, W, Gamma, eps, rows=None):
    """Block AttnRes pass over N blocks of S sublayers, by definition.

    emb: stored [T, d]; F: stored [N*S, T, d] sublayer outputs (F[q] is the
    output of sublayer q and only feeds reads of later sublayers).
    Returns fp64 [N*S, n_rows, d].
    """
    e64 = widen(emb)
    f64 = widen(F)
    T = e64.shape[0]
    sel = np.arange(T, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    e64 = np.ascontiguousarray(e64[sel])
    f64 = np.ascontiguousarray(f64[:, sel])
    outs = []
    for k in range(N * S):
        srcs = [np.ascontiguousarray(s) for s in block_sources(k, S, e64, f64)]
        o, _ = read(srcs, W[k], Gamma[k], eps)
        outs.append(o)
    return np.stack(outs)


def block_stage1(Src, n_src, W, Gamma, eps, rows=None):
    """Stage-1 reference: for each of the S queries, the read over Src[0 .. n_src).

    Returns (O fp64 [S, n_rows, d], lse fp64 [S, n_rows]), O normalised.
    """
    outs, lses = [], []
    for j in range(len(W)):
        o, l = full_read(Src, n_src, W[j], Gamma[j], eps, rows)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def prenorm(z, gamma, eps):
    """RMSNorm_pre of each row of z: gamma * z / sqrt(mean_k z_k^2 + eps).

    DepthBench reading notes section 2.3: the sublayer reads
    F_l(RMSNorm_pre,l(z_l)); RMSNorm is read as for the keys (learned gain,
    mean of squares over d, eps inside the root). z is fp64 (an oracle
    result) or a stored tensor (widened exactly); gamma is [d].
    """
    z64 = np.asarray(z, dtype=np.float64) if isinstance(z, np.ndarray) else widen(z)
    g = np.asarray(gamma, dtype=np.float64).reshape(-1)
    ms = np.mean(z64 * z64, axis=-1, keepdims=True)
    return g * z64 / np.sqrt(ms + eps)


def block_accumulate(P, f, first):
    """Running sum update P + f (or f alone when the running sum is empty)."""
    f64 = widen(f)
    return f64 if first else widen(P) + f64


def block_merge(Src, n_src, P, f_prev, p_is_empty, w, gamma, eps, rows=None):
    """Stage-2 reference: the read over {Src[0 .. n_src), P_new}.

    P_new = P + f_prev (f_prev may be None: P_new = P; p_is_empty: P_new =
    f_prev). Returns (out fp64 [n_rows, d], P_new fp64 [T, d]).
    """
    if f_prev is None:
        if p_is_empty:
            raise ValueError("an empty running sum with no f_prev has no source")
        p_new = widen(P)
    else:
        p_new = block_accumulate(P, f_prev, p_is_empty)
    srcs = _slices(Src, n_src) + [np.ascontiguousarray(p_new)]
    out, _ = read(srcs, w, gamma, eps, rows)
    return out, p_new
