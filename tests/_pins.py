"""Pins of the fp64 oracle: checks fixed by the pages and by mathematics.

Each check takes the oracle module and raises AssertionError when the oracle
disagrees with something that does not come from the oracle itself: a
hand-worked golden case, a closed form, an invariant of the definition, or the
independent pure-Python brute force. ``test_oracle_pins.py`` runs them against
the oracle; ``test_oracle_mutants.py`` runs them against oracles with planted
mistakes and requires each mistake to be caught.
"""
from __future__ import annotations

import itertools
import math

import numpy as np

from oracle import bruteforce
from tests._golden import load_cases


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"{what}: max abs error {err:.3e} > {tol:.1e}"


# ------------------------------------------------------------------ golden ----

def pin_golden(orc):
    """Hand-worked reads (tests/golden/worked_examples.txt)."""
    for c in load_cases():
        d = c["d"]
        if c["kind"] == "full":
            srcs = [np.asarray(s, dtype=np.float64).reshape(1, d) for s in c["src"]]
            out, _ = orc.read(srcs, c["w"][0], c["gamma"], c["eps"])
            _close(out[0], c["expect"][0], c["tol"], c["name"])
        else:
            N, S = c["N"], c["S"]
            emb = np.asarray(c["src"][0], dtype=np.float64).reshape(1, d)
            F = np.asarray(c["src"][1:], dtype=np.float64).reshape(N * S, 1, d)
            W = (np.tile(np.asarray(c["w_all"]), (N * S, 1)) if c["w_all"] is not None
                 else c["w"])
            G = np.tile(c["gamma"], (N * S, 1))
            out = orc.block_pass(emb, F, N, S, W, G, c["eps"])
            _close(out[:, 0, :], c["expect"], c["tol"], c["name"])


def pin_bf16_widening(orc):
    """bf16 storage is widened exactly: a single-source read returns it."""
    bits = np.array([0x3F80, 0xC000, 0x4049, 0x0001, 0x7F7F, 0x8000, 0x3EAB, 0xBF00],
                    dtype=np.uint16)
    expect = np.array([1.0, -2.0, 3.140625, 2.0 ** -133, 3.3895313892515355e38,
                       -0.0, 0.333984375, -0.5])
    src = orc.Bf16Bits(bits.reshape(1, 8))
    out, _ = orc.read([src], np.zeros(8), np.ones(8), 1e-6)
    assert np.array_equal(out[0], expect), f"bf16 widening: {out[0]} != {expect}"
    assert np.array_equal(orc.widen(src)[0], expect)


# ------------------------------------------------------------ closed forms ----

def pin_zero_query_is_mean(orc):
    """w = 0 gives the uniform mean of the sources (all pages: zero-init query)."""
    r = _rng(1)
    for n, T, d in [(1, 3, 5), (4, 6, 7), (9, 2, 16)]:
        V = r.standard_normal((n, T, d)) * np.sqrt(np.arange(1, n + 1))[:, None, None]
        out, lse = orc.full_read(V, n, np.zeros(d), r.standard_normal(d), 1e-6)
        _close(out, V.mean(axis=0), 1e-13, f"zero query mean n={n}")
        _close(lse, np.full(T, math.log(n)), 1e-13, "zero query lse = log n")


def pin_single_source_identity(orc):
    """One source (the first sublayer reads the embedding) returns it unchanged."""
    r = _rng(2)
    V = r.standard_normal((1, 5, 11)) * 3.0
    w = r.standard_normal(11)
    out, _ = orc.full_read(V, 1, w, np.ones(11), 1e-6)
    assert np.array_equal(out, V[0]), "single-source read must be the identity"


def pin_two_sources_logistic(orc):
    """d = 1, eps = 0: scores are +-w*gamma, so a_1 = 1/(1+exp(2 w gamma))."""
    r = _rng(3)
    for _ in range(8):
        x, y = abs(r.standard_normal()) + 0.1, -abs(r.standard_normal()) - 0.1
        w, g = r.standard_normal(), abs(r.standard_normal()) + 0.5
        a1 = 1.0 / (1.0 + math.exp(2.0 * w * g))
        srcs = [np.array([[x]]), np.array([[y]])]
        out, lse = orc.read(srcs, [w], [g], 0.0)
        _close(out[0, 0], (1 - a1) * x + a1 * y, 1e-14, "two-source logistic")
        _close(lse[0], math.log(math.exp(w * g) + math.exp(-w * g)), 1e-14, "two-source lse")


def pin_equal_sources(orc):
    """All sources equal: the read returns that source for any w."""
    r = _rng(4)
    v = r.standard_normal((3, 9))
    out, _ = orc.read([v] * 5, r.standard_normal(9) * 4, r.standard_normal(9), 1e-6)
    _close(out, v, 1e-14, "equal sources")


def pin_hardmax_limit(orc):
    """Large w: the read tends to the source with the largest score.

    d = 2, w = lambda * (1, 0), gamma = 1, eps = 0: the score of
    v = rho * (cos t, sin t) is lambda * sqrt(2) * cos t, whatever rho is; the
    source with the smallest |t| wins. Sources are built so that index 3 wins.
    """
    angles = [1.2, -0.9, 0.7, 0.05, -0.4, 2.5]
    radii = [5.0, 0.3, 2.0, 0.7, 9.0, 1.0]
    srcs = [np.array([[rho * math.cos(t), rho * math.sin(t)]]) for t, rho in zip(angles, radii)]
    out, _ = orc.read(srcs, [300.0, 0.0], [1.0, 1.0], 0.0)
    _close(out[0], srcs[3][0], 1e-12, "hardmax limit picks the largest score")


# --------------------------------------------------------------- invariants ----

def pin_permutation_invariance(orc):
    """The read is a sum over the source set: order does not matter."""
    r = _rng(5)
    n, T, d = 6, 4, 10
    V = r.standard_normal((n, T, d)) * np.arange(1, n + 1)[:, None, None]
    w, g = r.standard_normal(d) * 0.5, r.standard_normal(d)
    base, lb = orc.full_read(V, n, w, g, 1e-6)
    for p in [r.permutation(n) for _ in range(4)]:
        out, lse = orc.full_read(V[p], n, w, g, 1e-6)
        _close(out, base, 1e-13, "permutation invariance")
        _close(lse, lb, 1e-13, "permutation invariance (lse)")


def pin_key_scale_invariance(orc):
    """eps = 0: scaling a source changes its value but not its score.

    The read is then affine in the scale c of one source:
    z(c) = A + a_i * c * v_i with a_i independent of c.
    """
    r = _rng(6)
    n, T, d = 4, 3, 8
    V = r.standard_normal((n, T, d))
    w, g = r.standard_normal(d), r.standard_normal(d)
    outs = {}
    for c in (0.5, 2.0, 7.0):
        Vc = V.copy()
        Vc[2] *= c
        outs[c], _ = orc.full_read(Vc, n, w, g, 0.0)
    lhs = outs[7.0] - outs[0.5]
    rhs = (7.0 - 0.5) / (2.0 - 0.5) * (outs[2.0] - outs[0.5])
    _close(lhs, rhs, 1e-12, "score independent of the source scale")
    full_scaled, _ = orc.full_read(3.5 * V, n, w, g, 0.0)
    base, _ = orc.full_read(V, n, w, g, 0.0)
    _close(full_scaled, 3.5 * base, 1e-12, "scaling every source scales the read")


def pin_split_merge(orc):
    """Two parts merged by log-sum-exp equal the read over their union.

    This is the identity the two-stage Block AttnRes computation relies on
    (datacamp explainer, "two-stage computation": online-softmax merge).
    """
    r = _rng(7)
    n, T, d = 7, 5, 12
    V = r.standard_normal((n, T, d)) * 2
    w, g = r.standard_normal(d), r.standard_normal(d) + 1
    oa, la = orc.read([V[i] for i in range(3)], w, g, 1e-6)
    ob, lb = orc.read([V[i] for i in range(3, n)], w, g, 1e-6)
    ou, lu = orc.read([V[i] for i in range(n)], w, g, 1e-6)
    m = np.maximum(la, lb)
    ea, eb = np.exp(la - m), np.exp(lb - m)
    merged = (oa * ea[:, None] + ob * eb[:, None]) / (ea + eb)[:, None]
    _close(merged, ou, 1e-13, "split/merge = union")
    _close(np.logaddexp(la, lb), lu, 1e-13, "lse of the union")


def pin_block_s1_equals_full(orc):
    """Block AttnRes with one sublayer per block is Full AttnRes."""
    r = _rng(8)
    L, T, d = 6, 3, 5
    emb = r.standard_normal((T, d))
    F = r.standard_normal((L, T, d)) * 1.5
    W, G = r.standard_normal((L, d)), r.standard_normal((L, d))
    blk = orc.block_pass(emb, F, L, 1, W, G, 1e-6)
    hist = np.concatenate([emb[None], F[:-1]], axis=0)
    full = orc.full_pass(hist, L, W, G, 1e-6)
    _close(blk, full, 1e-13, "Block S=1 == Full")


def pin_block_zero_query_means(orc):
    """w = 0: each block read is the mean of its source set (written out here)."""
    r = _rng(9)
    N, S, T, d = 3, 4, 2, 3
    emb = r.standard_normal((T, d))
    F = r.standard_normal((N * S, T, d))
    out = orc.block_pass(emb, F, N, S, np.zeros((N * S, d)), np.ones((N * S, d)), 1e-6)
    for k in range(N * S):
        n, j = divmod(k, S)
        total = emb.copy()
        count = 1
        for m in range(n):                       # completed blocks 1..n
            total = total + sum(F[m * S + q] for q in range(S))
            count += 1
        if j > 0:                                # non-empty running sum
            total = total + sum(F[n * S + q] for q in range(j))
            count += 1
        _close(out[k], total / count, 1e-13, f"block mean at sublayer {k}")


def pin_stage1_and_merge_reference(orc):
    """Per-operation references agree with the block definition."""
    r = _rng(10)
    N, S, T, d = 3, 3, 4, 6
    emb = r.standard_normal((T, d))
    F = r.standard_normal((N * S, T, d))
    W, G = r.standard_normal((N * S, d)), r.standard_normal((N * S, d))
    full = orc.block_pass(emb, F, N, S, W, G, 1e-6)
    n = 2                                          # block index (0-based)
    Src = np.stack([emb, F[0:S].sum(0), F[S:2 * S].sum(0)])
    O, lse = orc.block_stage1(Src, n + 1, W[n * S:(n + 1) * S], G[n * S:(n + 1) * S], 1e-6)
    _close(O[0], full[n * S], 1e-13, "stage 1, first sublayer of a block")
    P = None
    for j in range(1, S):
        out, P = orc.block_merge(Src, n + 1, P, F[n * S + j - 1], P is None,
                                 W[n * S + j], G[n * S + j], 1e-6)
        _close(out, full[n * S + j], 1e-13, f"merge at in-block index {j}")


# --------------------------------------------------------------- brute force ----

def pin_bruteforce(orc):
    """Independent pure-Python fsum brute force on tiny shapes, all orders."""
    r = _rng(11)
    for n, T, d in [(1, 2, 1), (2, 3, 2), (3, 2, 3), (4, 1, 4), (5, 2, 3)]:
        V = r.standard_normal((n, T, d)) * np.arange(1, n + 1)[:, None, None]
        w, g = r.standard_normal(d), r.standard_normal(d)
        for perm in itertools.permutations(range(n)):
            out, lse = orc.full_read(V[list(perm)], n, w, g, 1e-3)
            for t in range(T):
                z, l = bruteforce.read([list(V[i, t]) for i in perm], list(w), list(g), 1e-3)
                _close(out[t], z, 1e-12, f"brute force read n={n}")
                _close(lse[t], l, 1e-12, f"brute force lse n={n}")
    # Full pass and every block size dividing the sublayer count.
    L, T, d = 6, 2, 3
    emb = r.standard_normal((T, d))
    F = r.standard_normal((L, T, d))
    W, G = r.standard_normal((L, d)) * 2, r.standard_normal((L, d))
    hist = np.concatenate([emb[None], F[:-1]])
    fp = orc.full_pass(hist, L, W, G, 1e-6)
    for S in [s for s in range(1, L + 1) if L % s == 0]:
        bp = orc.block_pass(emb, F, L // S, S, W, G, 1e-6)
        for t in range(T):
            ref = bruteforce.block_pass(list(emb[t]), [list(F[q, t]) for q in range(L)], S,
                                        [list(x) for x in W], [list(x) for x in G], 1e-6)
            _close(bp[:, t, :], ref, 1e-12, f"brute force block S={S}")
    for t in range(T):
        ref = bruteforce.full_pass([list(hist[i, t]) for i in range(L)],
                                   [list(x) for x in W], [list(x) for x in G], 1e-6)
        _close(fp[:, t, :], ref, 1e-12, "brute force full pass")


# ----------------------------------------------------------------- pre-norm ----

def pin_prenorm_constant_row(orc):
    """A constant row c * 1: out_k = gamma_k * c / sqrt(c^2 + eps) (closed form)."""
    d, c, eps = 5, -3.5, 0.25
    gamma = np.array([1.0, 0.5, -2.0, 3.0, 0.125])
    z = np.full((1, d), c)
    expect = gamma * c / math.sqrt(c * c + eps)
    _close(orc.prenorm(z, gamma, eps)[0], expect, 1e-14, "pre-norm of a constant row")


def pin_prenorm_unit_rms(orc):
    """gamma = 1, eps = 0: each output row is a positive multiple of its input
    with mean square exactly 1."""
    z = _rng(41).normal(size=(6, 9)) * np.arange(1, 7).reshape(6, 1)
    out = orc.prenorm(z, np.ones(9), 0.0)
    _close(np.mean(out * out, axis=1), np.ones(6), 1e-13, "mean square of the pre-norm")
    ratio = out / z
    _close(ratio, np.repeat(ratio[:, :1], 9, axis=1), 1e-12, "pre-norm is a per-row scaling")
    assert np.all(ratio > 0), "pre-norm flips signs"


def pin_prenorm_scale_invariance(orc):
    """eps = 0: RMSNorm_pre(c z) = RMSNorm_pre(z) for c > 0, and it is odd in z."""
    rng = _rng(42)
    z = rng.normal(size=(4, 7))
    gamma = rng.normal(size=7)
    base = orc.prenorm(z, gamma, 0.0)
    _close(orc.prenorm(13.0 * z, gamma, 0.0), base, 1e-12, "pre-norm scale invariance")
    _close(orc.prenorm(-z, gamma, 0.0), -base, 1e-14, "pre-norm is odd")


def pin_prenorm_of_zero_query_read(orc):
    """w = 0 read then pre-norm: the pre-norm of the plain mean of the sources,
    for a two-source hand case: sources (1, 3) and (3, 5), mean (2, 4), mean
    square 10, so with eps = 6 the row is (2, 4) / 4 scaled by gamma (0.5, 2)."""
    srcs = [np.array([[1.0, 3.0]]), np.array([[3.0, 5.0]])]
    z, _ = orc.read(srcs, np.zeros(2), np.ones(2), 1e-6)
    out = orc.prenorm(z, np.array([0.5, 2.0]), 6.0)
    _close(out[0], np.array([0.25, 2.0]), 1e-9, "pre-norm of the mean")


# ------------------------------------------------------ input-dependent query ----

def pin_dynamic_query_constant_rows(orc):
    """Every token's query equal to one w: the read equals the fixed-query read
    of the C oracle (a separate implementation), outputs and lse."""
    rng = _rng(61)
    n, T, d = 4, 5, 6
    V = rng.normal(size=(n, T, d)) * np.arange(1, n + 1).reshape(n, 1, 1)
    w = rng.normal(size=d)
    gamma = 1 + 0.3 * rng.normal(size=d)
    z, lse = orc.read_dynamic_query(list(V), np.tile(w, (T, 1)), gamma, 1e-3)
    rz, rl = orc.read(list(V), w, gamma, 1e-3)
    _close(z, rz, 1e-12, "constant-row query vs fixed query")
    _close(lse, rl, 1e-12, "constant-row query lse")


def pin_dynamic_query_per_token(orc):
    """Each token's result equals the fixed-query read with that token's query
    (token by token through the C oracle), and a zero query gives the mean."""
    rng = _rng(62)
    n, T, d = 3, 4, 5
    V = rng.normal(size=(n, T, d))
    Q = rng.normal(size=(T, d)) * 2.0
    gamma = 1 + 0.3 * rng.normal(size=d)
    z, _ = orc.read_dynamic_query(list(V), Q, gamma, 1e-6)
    for t in range(T):
        rz, _ = orc.read([V[i, t:t + 1] for i in range(n)], Q[t], gamma, 1e-6)
        _close(z[t], rz[0], 1e-12, f"token {t} with its own query")
    z0, _ = orc.read_dynamic_query(list(V), np.zeros((T, d)), gamma, 1e-6)
    _close(z0, V.mean(axis=0), 1e-14, "zero query is the mean")


def pin_query_projection(orc):
    """q = Wq h: the identity returns h, a permutation permutes its features,
    and a hand case: h = (1, 2), Wq = [[1, 1], [3, -1]] gives (3, 1)."""
    rng = _rng(63)
    H = rng.normal(size=(3, 4))
    _close(orc.query_projection(H, np.eye(4)), H, 0.0, "identity projection")
    P = np.eye(4)[[2, 0, 3, 1]]
    _close(orc.query_projection(H, P), H[:, [2, 0, 3, 1]], 0.0, "permutation projection")
    _close(orc.query_projection(np.array([[1.0, 2.0]]), np.array([[1.0, 1.0], [3.0, -1.0]])),
           np.array([[3.0, 1.0]]), 0.0, "hand-worked projection")


# ----------------------------------------------------------------- backward ----

def _fd_case(seed, n, T, d, eps):
    rng = _rng(seed)
    V = rng.normal(size=(n, T, d)) * np.arange(1, n + 1).reshape(n, 1, 1) ** 0.5
    w = rng.normal(size=d)
    gamma = 1 + 0.3 * rng.normal(size=d)
    dz = rng.normal(size=(T, d))
    return V, w, gamma, dz, eps


def pin_bwd_finite_differences(orc):
    """Gradients against central differences of the forward read (which is the
    C oracle, a separate implementation): L = sum(dz * z), step 1e-6, fp64."""
    V, w, gamma, dz, eps = _fd_case(51, 3, 2, 5, 0.1)
    dV, dw, dg = orc.read_bwd(list(V), w, gamma, eps, dz)
    h = 1e-6

    def loss(V_, w_, g_):
        z, _ = orc.read(list(V_), w_, g_, eps)
        return float(np.sum(z * dz))

    fd = np.zeros_like(V)
    for idx in np.ndindex(V.shape):
        vp, vm = V.copy(), V.copy()
        vp[idx] += h
        vm[idx] -= h
        fd[idx] = (loss(vp, w, gamma) - loss(vm, w, gamma)) / (2 * h)
    _close(dV, fd, 1e-7, "dV vs finite differences")
    eye = np.eye(V.shape[-1])
    fw = np.array([(loss(V, w + h * e, gamma) - loss(V, w - h * e, gamma)) / (2 * h) for e in eye])
    fg = np.array([(loss(V, w, gamma + h * e) - loss(V, w, gamma - h * e)) / (2 * h) for e in eye])
    _close(dw, fw, 1e-7, "dw vs finite differences")
    _close(dg, fg, 1e-7, "dgamma vs finite differences")


def pin_bwd_single_source(orc):
    """One source: z = v_0 whatever the score, so dv_0 = dz and dw = dgamma = 0."""
    V, w, gamma, dz, eps = _fd_case(52, 1, 3, 6, 1e-6)
    dV, dw, dg = orc.read_bwd(list(V), w, gamma, eps, dz)
    _close(dV[0], dz, 1e-14, "single-source dV")
    _close(dw, np.zeros(6), 1e-14, "single-source dw")
    _close(dg, np.zeros(6), 1e-14, "single-source dgamma")


def pin_bwd_equal_sources(orc):
    """n equal sources: the weights are 1/n and every dL/da_i is the same, so the
    score gradients vanish: dv_i = dz / n and dw = dgamma = 0."""
    V, w, gamma, dz, eps = _fd_case(53, 1, 2, 5, 1e-6)
    n = 4
    dV, dw, dg = orc.read_bwd([V[0]] * n, w, gamma, eps, dz)
    for i in range(n):
        _close(dV[i], dz / n, 1e-14, f"equal sources dV[{i}]")
    _close(dw, np.zeros(5), 1e-13, "equal sources dw")
    _close(dg, np.zeros(5), 1e-13, "equal sources dgamma")


def pin_bwd_permutation(orc):
    """Permuting the sources permutes dV and leaves dw and dgamma unchanged."""
    V, w, gamma, dz, eps = _fd_case(54, 4, 3, 5, 1e-3)
    dV, dw, dg = orc.read_bwd(list(V), w, gamma, eps, dz)
    perm = [2, 0, 3, 1]
    pV, pw, pg = orc.read_bwd([V[i] for i in perm], w, gamma, eps, dz)
    _close(pV, dV[perm], 1e-12, "permuted dV")
    _close(pw, dw, 1e-12, "permuted dw")
    _close(pg, dg, 1e-12, "permuted dgamma")


def _block_bwd_case(seed, N, S, T, d, eps):
    rng = _rng(seed)
    emb = rng.normal(size=(T, d))
    F = rng.normal(size=(N * S, T, d))
    W = 0.7 * rng.normal(size=(N * S, d))
    G = 1 + 0.3 * rng.normal(size=(N * S, d))
    dOut = rng.normal(size=(N * S, T, d))
    Src = np.stack([emb] + [F[(m - 1) * S:m * S].sum(axis=0) for m in range(1, N)])
    return emb, F, W, G, dOut, Src, eps


def pin_block_bwd_finite_differences(orc):
    """Block pass gradients against central differences of the C oracle's
    forward Block pass (summaries and running sums as exact sums of F):
    L = sum_k <dOut_k, out_k>, step 1e-6, fp64."""
    N, S = 2, 3
    emb, F, W, G, dOut, Src, eps = _block_bwd_case(55, N, S, 2, 3, 0.05)
    dEmb, dF, dW, dG = orc.block_pass_bwd(Src, F, N, S, W, G, eps, dOut)
    h = 1e-6

    def loss(e_, F_, W_, G_):
        return float(np.sum(orc.block_pass(e_, F_, N, S, W_, G_, eps) * dOut))

    def fd(x, f):
        out = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            out[idx] = (f(xp) - f(xm)) / (2 * h)
        return out

    _close(dEmb, fd(emb, lambda x: loss(x, F, W, G)), 1e-7, "block dEmb vs finite differences")
    _close(dF, fd(F, lambda x: loss(emb, x, W, G)), 1e-7, "block dF vs finite differences")
    _close(dW, fd(W, lambda x: loss(emb, F, x, G)), 1e-7, "block dW vs finite differences")
    _close(dG, fd(G, lambda x: loss(emb, F, W, x)), 1e-7, "block dGamma vs finite differences")


def pin_block_bwd_s1_is_full_pass_bwd(orc):
    """With S = 1 the Block pass is the Full pass over [emb, f_0, f_1, ...]
    (each summary is one output, no running sum), so its gradients are the
    sums of the Full reads' gradients."""
    L = 4
    emb, F, W, G, dOut, Src, eps = _block_bwd_case(56, L, 1, 3, 4, 1e-6)
    dEmb, dF, dW, dG = orc.block_pass_bwd(Src, F, L, 1, W, G, eps, dOut)
    V = np.concatenate([emb[None], F])
    ref = np.zeros_like(V)
    for k in range(L):
        dV, dw, dg = orc.read_bwd(list(V[:k + 1]), W[k], G[k], eps, dOut[k])
        ref[:k + 1] += dV
        _close(dW[k], dw, 1e-13, f"S=1 dW[{k}]")
        _close(dG[k], dg, 1e-13, f"S=1 dGamma[{k}]")
    _close(dEmb, ref[0], 1e-13, "S=1 dEmb")
    _close(dF[:L - 1], ref[1:L], 1e-13, "S=1 dF")
    _close(dF[L - 1], np.zeros_like(dF[L - 1]), 0.0, "S=1 dF of the last output (read by none)")


ALL_PINS = [
    pin_golden, pin_bf16_widening, pin_zero_query_is_mean, pin_single_source_identity,
    pin_two_sources_logistic, pin_equal_sources, pin_hardmax_limit,
    pin_permutation_invariance, pin_key_scale_invariance, pin_split_merge,
    pin_block_s1_equals_full, pin_block_zero_query_means, pin_stage1_and_merge_reference,
    pin_bruteforce, pin_prenorm_constant_row, pin_prenorm_unit_rms,
    pin_prenorm_scale_invariance, pin_prenorm_of_zero_query_read, pin_bwd_finite_differences,
    pin_bwd_single_source, pin_bwd_equal_sources, pin_bwd_permutation,
    pin_dynamic_query_constant_rows, pin_dynamic_query_per_token, pin_query_projection,
    pin_block_bwd_finite_differences, pin_block_bwd_s1_is_full_pass_bwd,
]
