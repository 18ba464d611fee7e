"""Planted mistakes in the oracle must each be caught by a pin (CPU only).

Every mutant is a copy of the oracle with one plausible error: a dropped or
misplaced term, a wrong sign or index, a wrong source set for Block AttnRes.
The pins in tests/_pins.py are run against the mutant; at least one must fail.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
from tests import _pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attnres_oracle.c")

C_MUTANTS = {
    "eps_outside_root": ("1.0 / sqrt(sq / (double)d + eps)", "1.0 / (sqrt(sq / (double)d) + eps)"),
    "sum_not_mean": ("sqrt(sq / (double)d + eps)", "sqrt(sq + eps)"),
    "no_key_rmsnorm": ("double inv_rms = 1.0 / sqrt(sq / (double)d + eps);", "double inv_rms = 1.0; (void)sq;"),
    "no_gain": ("w[k] * (gamma[k] * v[i][k] * inv_rms)", "w[k] * (v[i][k] * inv_rms)"),
    "negated_score": ("e[i] = dot;", "e[i] = -dot;"),
    "sqrt_d_scale": ("e[i] = dot;", "e[i] = dot / sqrt((double)d);"),
    "gain_on_values": ("out[k] += a * v[i][k];", "out[k] += a * gamma[k] * v[i][k];"),
    "reversed_query": ("w[k] * (gamma[k]", "w[d - 1 - k] * (gamma[k]"),
    "unnormalised_weights": ("double a = exp(e[i] - m) / z;", "double a = exp(e[i] - m);"),
    "lse_without_max": ("*lse = m + log(z);", "*lse = log(z);"),
    "bf16_shift": ("<< 16;", "<< 15;"),
    "first_source_dropped": ("for (int i = 0; i < n; ++i) {\n    double a", "for (int i = 1; i < n; ++i) {\n    double a"),
}


def _run_pins(orc):
    failures = []
    for pin in _pins.ALL_PINS:
        try:
            pin(orc)
        except Exception as exc:  # any failure counts as caught
            failures.append((pin.__name__, repr(exc)[:120]))
    return failures


@pytest.mark.parametrize("name", sorted(C_MUTANTS))
def test_c_mutant_is_caught(name, tmp_path, monkeypatch):
    old, new = C_MUTANTS[name]
    text = open(SRC).read()
    assert old in text, f"mutation site for {name} not found"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib_path = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", "-o",
                    str(lib_path), str(src), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_lib", oracle.load_library(str(lib_path)))
    assert _run_pins(oracle), f"mutant {name} passed every pin"


def _block_mutant(kind):
    def sources(k, S, emb64, F64):
        n, j = divmod(k, S)
        zero = np.zeros_like(emb64)
        srcs = [emb64]
        for m in range(1, n + 1):
            b = np.sum(F64[(m - 1) * S: m * S], axis=0)
            if kind == "summary_is_mean":
                b = b / S
            if kind == "embedding_in_first_block" and m == 1:
                b = b + emb64
            srcs.append(b)
        if kind == "one_block_short" and n >= 1:
            srcs.pop()
        if kind == "running_sum_as_zero_when_empty" and j == 0:
            srcs.append(zero)
        if j >= 1 and kind != "no_running_sum":
            hi = k + 1 if kind == "running_sum_includes_self" else k
            srcs.append(np.sum(F64[n * S: hi], axis=0))
        return srcs
    return sources


@pytest.mark.parametrize("kind", ["summary_is_mean", "embedding_in_first_block",
                                  "one_block_short", "running_sum_as_zero_when_empty",
                                  "no_running_sum", "running_sum_includes_self"])
def test_block_mutant_is_caught(kind, monkeypatch, oracle_mod):
    monkeypatch.setattr(oracle, "block_sources", _block_mutant(kind))
    assert _run_pins(oracle), f"block mutant {kind} passed every pin"


def _prenorm_mutant(kind):
    def prenorm(z, gamma, eps):
        z64 = np.asarray(z, dtype=np.float64) if isinstance(z, np.ndarray) else oracle.widen(z)
        g = np.asarray(gamma, dtype=np.float64).reshape(-1)
        ms = np.mean(z64 * z64, axis=-1, keepdims=True)
        if kind == "sum_not_mean":
            return g * z64 / np.sqrt(ms * z64.shape[-1] + eps)
        if kind == "eps_outside_root":
            return g * z64 / (np.sqrt(ms) + eps)
        if kind == "no_gain":
            return z64 / np.sqrt(ms + eps)
        if kind == "gain_squared":
            return g * g * z64 / np.sqrt(ms + eps)
        if kind == "no_root":
            return g * z64 / (ms + eps)
        if kind == "mean_over_rows":
            return g * z64 / np.sqrt(np.mean(z64 * z64, axis=0, keepdims=True) + eps)
        raise ValueError(kind)
    return prenorm


@pytest.mark.parametrize("kind", ["sum_not_mean", "eps_outside_root", "no_gain", "gain_squared",
                                  "no_root", "mean_over_rows"])
def test_prenorm_mutant_is_caught(kind, monkeypatch, oracle_mod):
    monkeypatch.setattr(oracle, "prenorm", _prenorm_mutant(kind))
    assert _run_pins(oracle), f"pre-norm mutant {kind} passed every pin"


def _bwd_mutant(kind):
    real = oracle.read_bwd

    def read_bwd(sources, w, gamma, eps, dz):
        V = np.stack([np.asarray(s, np.float64) if isinstance(s, np.ndarray) else oracle.widen(s)
                      for s in sources])
        g = np.asarray(dz, np.float64) if isinstance(dz, np.ndarray) else oracle.widen(dz)
        d = V.shape[-1]
        w64 = np.asarray(w, np.float64).reshape(d)
        g64 = np.asarray(gamma, np.float64).reshape(d)
        u = w64 * g64
        r = 1.0 / np.sqrt(np.mean(V * V, axis=-1) + eps)
        e = r * np.einsum("ntk,k->nt", V, u)
        a = np.exp(e - e.max(axis=0, keepdims=True))
        a /= a.sum(axis=0, keepdims=True)
        da = np.einsum("ntk,tk->nt", V, g)
        de = a * (da - np.sum(a * da, axis=0, keepdims=True))
        if kind == "score_grad_sign":
            de = -de
        rms_term = (e * r * r / d)[..., None] * V
        if kind == "no_rms_derivative":
            rms_term = 0.0 * V
        if kind == "rms_derivative_r_cubed":
            rms_term = (e * r * r * r / d)[..., None] * V
        value_term = a[..., None] * g[None]
        if kind == "no_value_path":
            value_term = 0.0 * V
        dV = value_term + de[..., None] * (r[..., None] * u - rms_term)
        du = np.einsum("nt,ntk->k", de * r, V)
        if kind == "du_from_weights":
            du = np.einsum("nt,ntk->k", a * r, V)
        if kind == "dw_without_gain":
            return dV, du, du * w64
        if kind == "gains_swapped":
            return dV, du * w64, du * g64
        raise ValueError(kind)
    del real
    return read_bwd


@pytest.mark.parametrize("kind", ["score_grad_sign", "no_rms_derivative", "rms_derivative_r_cubed",
                                  "no_value_path", "du_from_weights", "dw_without_gain", "gains_swapped"])
def test_bwd_mutant_is_caught(kind, monkeypatch, oracle_mod):
    monkeypatch.setattr(oracle, "read_bwd", _bwd_mutant(kind))
    assert _run_pins(oracle), f"backward mutant {kind} passed every pin"


def _block_bwd_mutant(kind):
    def block_pass_bwd(Src, F, N, S, W, Gamma, eps, dOut):
        s64 = [np.asarray(Src[i], np.float64) for i in range(N)]
        f64 = np.asarray(F, np.float64)
        g = np.asarray(dOut, np.float64)
        dEmb = np.zeros_like(s64[0])
        dF = np.zeros_like(f64)
        dW = np.zeros((N * S, np.asarray(W).shape[-1]))
        dG = np.zeros_like(dW)
        for k in range(N * S):
            n, j = divmod(k, S)
            srcs = [s64[m] for m in range(n + 1)]
            if j >= 1:
                srcs.append(np.sum(f64[n * S:k], axis=0))
            dV, dW[k], dG[k] = oracle.read_bwd(srcs, np.asarray(W[k], np.float64), np.asarray(Gamma[k], np.float64),
                                               eps, g[k])
            if kind != "embedding_grad_dropped":
                dEmb += dV[0]
            for m in range(1, n + 1):
                if kind == "summary_to_first_member":
                    dF[(m - 1) * S] += dV[m]
                elif kind == "summary_to_next_block":
                    dF[m * S:(m + 1) * S] += dV[m]
                else:
                    dF[(m - 1) * S:m * S] += dV[m]
            if j >= 1 and kind != "running_sum_grad_dropped":
                hi = k + 1 if kind == "running_sum_includes_current" else k
                dF[n * S:hi] += dV[n + 1]
        return dEmb, dF, dW, dG
    return block_pass_bwd


@pytest.mark.parametrize("kind", ["embedding_grad_dropped", "summary_to_first_member", "summary_to_next_block",
                                  "running_sum_grad_dropped", "running_sum_includes_current"])
def test_block_bwd_mutant_is_caught(kind, monkeypatch, oracle_mod):
    monkeypatch.setattr(oracle, "block_pass_bwd", _block_bwd_mutant(kind))
    assert _run_pins(oracle), f"Block backward mutant {kind} passed every pin"


def _dynq_mutant(kind):
    def read_dynamic_query(sources, Q, gamma, eps):
        V = np.stack([np.asarray(s, np.float64) if isinstance(s, np.ndarray) else oracle.widen(s)
                      for s in sources])
        q = np.asarray(Q, np.float64)
        g = np.asarray(gamma, np.float64).reshape(-1)
        r = 1.0 / np.sqrt(np.mean(V * V, axis=-1) + eps)
        if kind == "query_of_token_0":
            q = np.repeat(q[:1], q.shape[0], axis=0)
        if kind == "no_gain":
            g = np.ones_like(g)
        if kind == "query_transposed_tokens":
            q = q[::-1]
        e = r * np.einsum("ntk,tk->nt", V, q * g)
        m = e.max(axis=0)
        p = np.exp(e - m)
        z = p.sum(axis=0)
        return np.einsum("nt,ntk->tk", p / z, V), m + np.log(z)
    return read_dynamic_query


def _proj_mutant(kind):
    def query_projection(H, Wq):
        h = np.asarray(H, np.float64)
        w = np.asarray(Wq, np.float64)
        return h @ w if kind == "not_transposed" else (h @ w.T) * (0.5 if kind == "half" else 1.0)
    return query_projection


@pytest.mark.parametrize("kind", ["query_of_token_0", "no_gain", "query_transposed_tokens"])
def test_dynamic_query_mutant_is_caught(kind, monkeypatch, oracle_mod):
    monkeypatch.setattr(oracle, "read_dynamic_query", _dynq_mutant(kind))
    assert _run_pins(oracle), f"dynamic-query mutant {kind} passed every pin"


@pytest.mark.parametrize("kind", ["not_transposed", "half"])
def test_projection_mutant_is_caught(kind, monkeypatch, oracle_mod):
    monkeypatch.setattr(oracle, "query_projection", _proj_mutant(kind))
    assert _run_pins(oracle), f"projection mutant {kind} passed every pin"
